"""The C ABI library builds, loads and exports every function include/*.h
declares; host-side argument validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

import sparse_mixture_experts_gemm_gb300 as moe
from sparse_mixture_experts_gemm_gb300 import buildlib as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("moe.h", "gdn.h")]


def header_functions():
    names = set()
    for path in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:moe|gdn)_\w+)\s*\(", src,
                                flags=re.M))
    return sorted(names)


def test_headers_are_all_listed():
    found = sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    assert found == sorted(os.path.basename(h) for h in HEADERS)


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def test_header_declares_the_boundary():
    fns = header_functions()
    for name in ["moe_create", "moe_route", "moe_forward", "moe_forward_host", "moe_host_join",
                 "moe_destroy", "moe_status", "moe_strerror", "gdn_scan"]:
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert name in moe.EXPORTED


def test_strerror(lib):
    assert moe.strerror(0) == "ok"
    assert "align" in moe.strerror(moe.MOE_ERR_ALIGNMENT)
    assert moe.strerror(-99) == "unknown error"


def _cfg(**kw):
    base = dict(d_model=512, n_experts=16, top_k=4, d_ff=128, n_shared=1, max_tokens=64,
                dtype=moe.MOE_BF16, w_router=0x1000, w_gate=0x2000, w_up=0x3000, w_down=0x4000,
                s_gate=0x5000, s_up=0x6000, s_down=0x7000, router_bias=None)
    base.update(kw)
    c = moe.moe_config()
    for k, v in base.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,code", [
    (dict(d_model=0), moe.MOE_ERR_INVALID_ARG),
    (dict(top_k=0), moe.MOE_ERR_INVALID_ARG),
    (dict(n_shared=2), moe.MOE_ERR_INVALID_ARG),
    (dict(w_gate=None), moe.MOE_ERR_INVALID_ARG),
    (dict(s_up=None), moe.MOE_ERR_INVALID_ARG),
    (dict(dtype=7), moe.MOE_ERR_INVALID_ARG),
    (dict(d_model=520), moe.MOE_ERR_UNSUPPORTED),
    (dict(d_ff=100), moe.MOE_ERR_UNSUPPORTED),
    (dict(n_experts=257), moe.MOE_ERR_UNSUPPORTED),
    (dict(top_k=9, n_experts=16), moe.MOE_ERR_UNSUPPORTED),
    (dict(top_k=5, n_experts=4), moe.MOE_ERR_UNSUPPORTED),
    (dict(max_tokens=70000), moe.MOE_ERR_UNSUPPORTED),
    (dict(w_down=0x4004), moe.MOE_ERR_ALIGNMENT),
    (dict(router_bias=0x8008), moe.MOE_ERR_ALIGNMENT),
])
def test_create_rejects_bad_config_on_host(lib, kw, code):
    h = ctypes.c_void_p()
    rc = lib.moe_create(ctypes.byref(_cfg(**kw)), ctypes.byref(h))
    assert rc == code and h.value is None


def test_null_handle_calls(lib):
    assert lib.moe_forward(None, None, 4, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_host(None, None, 4, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_host_join(None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, None, 4, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_destroy(None) == moe.MOE_OK
    assert lib.moe_create(None, None) == moe.MOE_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        moe.lib()


def _q4w(**kw):
    w = moe.moe_q4_weights()
    for i, name in enumerate(("gate", "up", "down", "s_gate", "s_up", "s_down")):
        base = 0x10000 * (i + 1)
        setattr(w, name, moe.moe_q4_matrix(base, base + 0x1000, base + 0x2000))
    for name, m in kw.items():
        setattr(w, name, m)
    return w


def _q4cfg(**kw):
    return _cfg(**{**dict(w_gate=None, w_up=None, w_down=None, s_gate=None, s_up=None,
                          s_down=None), **kw})


@pytest.mark.parametrize("cfg_kw,w_kw,code", [
    (dict(w_gate=0x2000), {}, moe.MOE_ERR_INVALID_ARG),       # bf16 expert weights given too
    (dict(s_down=0x7000), {}, moe.MOE_ERR_INVALID_ARG),
    (dict(dtype=moe.MOE_F32), {}, moe.MOE_ERR_UNSUPPORTED),    # 4-bit layers take bf16 tokens
    (dict(w_router=None), {}, moe.MOE_ERR_INVALID_ARG),
    ({}, dict(up=moe.moe_q4_matrix(0x20000, None, 0x22000)), moe.MOE_ERR_INVALID_ARG),
    ({}, dict(down=moe.moe_q4_matrix(0x30008, 0x31000, 0x32000)), moe.MOE_ERR_ALIGNMENT),
    ({}, dict(s_gate=moe.moe_q4_matrix(None, None, None)), moe.MOE_ERR_INVALID_ARG),
    # (top_k + n_shared) * d_ff / 64 = 9 * 32 > 160 pairs per down row
    (dict(top_k=8, d_ff=2048, n_experts=16), {}, moe.MOE_ERR_UNSUPPORTED),
    (dict(d_model=520), {}, moe.MOE_ERR_UNSUPPORTED),
])
def test_create_q4_rejects_bad_config_on_host(lib, cfg_kw, w_kw, code):
    h = ctypes.c_void_p()
    rc = lib.moe_create_q4(ctypes.byref(_q4cfg(**cfg_kw)), ctypes.byref(_q4w(**w_kw)),
                           ctypes.byref(h))
    assert rc == code and h.value is None


def test_create_q4_null_weights(lib):
    h = ctypes.c_void_p()
    assert lib.moe_create_q4(ctypes.byref(_q4cfg()), None, ctypes.byref(h)) == \
        moe.MOE_ERR_INVALID_ARG
    assert h.value is None


@pytest.mark.parametrize("args,code", [
    ((0x1000, moe.MOE_BF16, 4, 100, 0x2000, 0x3000, 0x4000), moe.MOE_ERR_INVALID_ARG),  # cols % 64
    ((0x1000, moe.MOE_BF16, -1, 64, 0x2000, 0x3000, 0x4000), moe.MOE_ERR_INVALID_ARG),
    ((0x1000, 5, 4, 64, 0x2000, 0x3000, 0x4000), moe.MOE_ERR_INVALID_ARG),              # dtype
    ((0x1000, moe.MOE_BF16, 4, 64, None, 0x3000, 0x4000), moe.MOE_ERR_INVALID_ARG),
    ((0x1000, moe.MOE_F32, 4, 64, 0x2008, 0x3000, 0x4000), moe.MOE_ERR_ALIGNMENT),
    ((0x1002, moe.MOE_BF16, 4, 64, 0x2000, 0x3000, 0x4000), moe.MOE_ERR_ALIGNMENT),
    ((None, moe.MOE_BF16, 0, 64, None, None, None), moe.MOE_OK),                      # no rows
])
def test_quantize_q4_validates_on_host(lib, args, code):
    assert lib.moe_quantize_q4(*args, None) == code


@pytest.mark.parametrize("args,code", [
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(Hk=0), moe.MOE_ERR_INVALID_ARG),
    (dict(Hk=3), moe.MOE_ERR_INVALID_ARG),          # 32 value heads over 3 key heads
    (dict(q=None), moe.MOE_ERR_INVALID_ARG),
    (dict(alpha=None), moe.MOE_ERR_INVALID_ARG),
    (dict(dk=64), moe.MOE_ERR_UNSUPPORTED),
    (dict(dv=24), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=0x2008), moe.MOE_ERR_ALIGNMENT),
    (dict(s_in=0x7004), moe.MOE_ERR_ALIGNMENT),
    (dict(beta=0x5002), moe.MOE_ERR_ALIGNMENT),
])
def test_gdn_scan_rejects_before_any_launch(lib, args, code):
    """Validation happens on the host, before anything touches a GPU."""
    a = dict(q=0x1000, k=0x2000, v=0x3000, alpha=0x4000, beta=0x5000, s_in=None, s_out=None,
             o=0x6000, T=16, Hk=16, Hv=32, dk=128, dv=128)
    a.update(args)
    rc = lib.gdn_scan(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["s_in"], a["s_out"],
                      a["o"], a["T"], a["Hk"], a["Hv"], a["dk"], a["dv"], None)
    assert rc == code



def test_set_option_rejects_null_handle_and_bad_values(lib):
    """moe_set_option validates on the host: a null handle is refused before
    any CUDA call."""
    assert lib.moe_set_option(None, moe.MOE_OPT_PAIR_MIN_TOKENS, 0) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_option(None, 99, 0) == moe.MOE_ERR_INVALID_ARG


def test_gemv_limit_option_is_declared():
    """The option numbers of the binding match the header's."""
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    for name in ("MOE_OPT_PAIR_MIN_TOKENS", "MOE_OPT_GEMV_MAX_TOKENS", "MOE_OPT_MMA2_MIN_TOKENS",
                 "MOE_OPT_MMA2_DOWN_MIN_TOKENS", "MOE_OPT_ROUTER_PAIR_MIN_TOKENS"):
        m = re.search(r"#define\s+" + name + r"\s+(\d+)", src)
        assert m and int(m.group(1)) == getattr(moe, name)
