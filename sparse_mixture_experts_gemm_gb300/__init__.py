"""Sparse Mixture-of-Experts feed-forward block on one GB300 (sm_103a).

Python binding of the C ABI in ``include/moe.h``: the functions below carry
the C names and only marshal arguments (torch tensors -> device pointers,
torch streams -> cudaStream_t).  Every step of the block runs in the CUDA
kernels of ``libmoe.so``; if that library is not built this module raises
instead of computing anything another way.

The block ("Optimizing on-device inference for Apple Silicon", sections "Qwen
creates three distinct workload shapes" and "Reduce intermediate traffic and
dispatch traffic"): a router picks top-k of E experts per token, each expert is
a SwiGLU MLP, the chosen experts' outputs are weighted by the renormalised
routing probabilities and a shared expert's output is added.
"""
from __future__ import annotations

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_ALIGNMENT = -2
MOE_ERR_UNSUPPORTED = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE_TIMEOUT = -5
MOE_ERR_DEVICE_BOUNDS = -6
MOE_ERR_OUT_OF_MEMORY = -7

MOE_BF16 = 0
MOE_F32 = 1

MOE_OPT_PAIR_MIN_TOKENS = 1
MOE_OPT_GEMV_MAX_TOKENS = 3
MOE_OPT_MMA2_MIN_TOKENS = 4
MOE_OPT_MMA2_DOWN_MIN_TOKENS = 5
MOE_OPT_ROUTER_PAIR_MIN_TOKENS = 6

KERNEL_KINDS = ["router", "permute", "gemm_gate_up", "gemm_down", "combine", "decode_router",
                "decode_gate_up", "decode_down", "gemv_gate_up", "gemv_down"]

EXPORTED = ["moe_create", "moe_route", "moe_forward", "moe_forward_routed", "moe_forward_host",
            "moe_host_join", "moe_status", "moe_set_option", "moe_destroy",
            "moe_strerror", "moe_profile", "moe_profile_read", "moe_debug_wait_timeout",
            "moe_decode_noalloc", "moe_noalloc_status", "moe_create_q4", "moe_quantize_q4",
            "gdn_scan"]

Q4_GROUP = 64  # columns per (scale, bias) pair of the 4-bit format


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


class moe_config(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("d_ff", ctypes.c_int), ("n_shared", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("dtype", ctypes.c_int),
                ("w_router", ctypes.c_void_p), ("w_gate", ctypes.c_void_p),
                ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p),
                ("s_down", ctypes.c_void_p), ("router_bias", ctypes.c_void_p)]


class moe_q4_matrix(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p)]


class moe_q4_weights(ctypes.Structure):
    _fields_ = [(n, moe_q4_matrix) for n in ("gate", "up", "down", "s_gate", "s_up", "s_down")]


_lib = None


def build(force: bool = False) -> str:
    """Compile libmoe.so in-tree (nvcc, sm_103a)."""
    from . import buildlib
    return buildlib.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m sparse_mixture_experts_gemm_gb300.buildlib`")
    L = ctypes.CDLL(LIB_PATH)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    L.moe_create.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(vp)]
    L.moe_route.argtypes = [vp, vp, ip, vp, vp, vp, vp]
    L.moe_forward.argtypes = [vp, vp, ip, vp, vp]
    L.moe_forward_routed.argtypes = [vp, vp, ip, vp, vp, vp, vp, vp]
    L.moe_forward_host.argtypes = [vp, vp, ip, vp, vp]
    L.moe_host_join.argtypes = [vp, vp]
    L.moe_status.argtypes = [vp, vp, ctypes.POINTER(ip)]
    L.moe_set_option.argtypes = [vp, ip, ctypes.c_longlong]
    L.moe_destroy.argtypes = [vp]
    L.moe_strerror.argtypes = [ip]
    L.moe_strerror.restype = ctypes.c_char_p
    L.moe_profile.argtypes = [vp, ip]
    L.moe_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float),
                                   ctypes.POINTER(ctypes.c_int64), ip]
    L.moe_debug_wait_timeout.argtypes = [vp, ip, vp]
    L.moe_decode_noalloc.argtypes = [ctypes.POINTER(moe_config), vp, vp, vp]
    L.moe_noalloc_status.argtypes = [vp, ctypes.POINTER(ip)]
    L.moe_create_q4.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(moe_q4_weights),
                                ctypes.POINTER(vp)]
    L.moe_quantize_q4.argtypes = [vp, ip, ctypes.c_longlong, ip, vp, vp, vp, vp]
    L.gdn_scan.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ip, ip, ip, ip, ip, vp]
    for name in EXPORTED:
        if name != "moe_strerror":
            getattr(L, name).restype = ip
    _lib = L
    return L


def strerror(code: int) -> str:
    try:
        return lib().moe_strerror(code).decode()
    except RuntimeError:
        return f"error {code}"


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc != MOE_OK:
        raise MoeError(rc, where)
    return rc


# ----------------------------------------------------------------- C names
def moe_create(cfg: moe_config) -> int:
    h = ctypes.c_void_p()
    _check(lib().moe_create(ctypes.byref(cfg), ctypes.byref(h)), "moe_create")
    return h.value


def moe_route(h: int, x, T: int, topk_idx, topk_w, counts, stream=None) -> int:
    return _check(lib().moe_route(h, _ptr(x), T, _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
                                  _stream(stream)), "moe_route")


def moe_forward(h: int, x, T: int, out, stream=None) -> int:
    return _check(lib().moe_forward(h, _ptr(x), T, _ptr(out), _stream(stream)), "moe_forward")


def moe_forward_routed(h: int, x, T: int, out, topk_idx=None, topk_w=None, counts=None,
                       stream=None) -> int:
    return _check(lib().moe_forward_routed(h, _ptr(x), T, _ptr(out), _ptr(topk_idx),
                                           _ptr(topk_w), _ptr(counts), _stream(stream)),
                  "moe_forward_routed")


def moe_forward_host(h: int, x_host, T: int, out_host, stream=None) -> int:
    return _check(lib().moe_forward_host(h, _ptr(x_host), T, _ptr(out_host), _stream(stream)),
                  "moe_forward_host")


def moe_host_join(h: int, stream=None) -> int:
    return _check(lib().moe_host_join(h, _stream(stream)), "moe_host_join")


def moe_status(h: int, stream=None) -> tuple[int, int]:
    """(code, detail) of the device status word; synchronises the stream."""
    detail = ctypes.c_int(0)
    rc = lib().moe_status(h, _stream(stream), ctypes.byref(detail))
    return rc, detail.value


def moe_destroy(h: int) -> int:
    return _check(lib().moe_destroy(h), "moe_destroy")


def moe_strerror(code: int) -> str:
    return strerror(code)


def moe_set_option(h: int, option: int, value: int) -> int:
    return _check(lib().moe_set_option(h, option, value), "moe_set_option")


def moe_profile(h: int, enable: bool) -> int:
    return _check(lib().moe_profile(h, 1 if enable else 0), "moe_profile")


def moe_profile_read(h: int) -> dict:
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(lib().moe_profile_read(h, ms, cnt, n), "moe_profile_read")
    return {name: (ms[i], cnt[i]) for i, name in enumerate(KERNEL_KINDS)}


def moe_debug_wait_timeout(h: int, wait_us: int, stream=None) -> int:
    return _check(lib().moe_debug_wait_timeout(h, wait_us, _stream(stream)),
                  "moe_debug_wait_timeout")


def moe_decode_noalloc(cfg: moe_config, x, out, stream=None) -> int:
    """Batch-1 forward without any device allocation (see include/moe.h): for
    callers that cannot allocate device memory and so cannot create a handle."""
    return _check(lib().moe_decode_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(out),
                                           _stream(stream)), "moe_decode_noalloc")


def moe_noalloc_status(stream=None) -> tuple[int, int]:
    """(code, detail) of moe_decode_noalloc's device status word on the current
    device; synchronises the stream and clears the word."""
    detail = ctypes.c_int(0)
    rc = lib().moe_noalloc_status(_stream(stream), ctypes.byref(detail))
    return rc, detail.value


def moe_create_q4(cfg: moe_config, w: moe_q4_weights) -> int:
    h = ctypes.c_void_p()
    _check(lib().moe_create_q4(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)),
           "moe_create_q4")
    return h.value


def moe_quantize_q4(w, dtype: int, rows: int, cols: int, codes, scales, biases,
                    stream=None) -> int:
    return _check(lib().moe_quantize_q4(_ptr(w), dtype, rows, cols, _ptr(codes), _ptr(scales),
                                        _ptr(biases), _stream(stream)), "moe_quantize_q4")


def quantize_q4(w, stream=None):
    """4-bit group-affine copy of a CUDA tensor w[..., cols] (bf16 or f32): returns
    (codes uint8 [..., cols/2], scales, biases: bf16 bits as int16 [..., cols/64])."""
    import torch
    cols = w.shape[-1]
    rows = w.numel() // cols
    lead = tuple(w.shape[:-1])
    codes = torch.empty(lead + (cols // 2,), dtype=torch.uint8, device=w.device)
    scales = torch.empty(lead + (cols // Q4_GROUP,), dtype=torch.int16, device=w.device)
    biases = torch.empty_like(scales)
    dt = {torch.bfloat16: MOE_BF16, torch.float32: MOE_F32}[w.dtype]
    moe_quantize_q4(w.contiguous(), dt, rows, cols, codes, scales, biases, stream)
    return codes, scales, biases


# ----------------------------------------------------------------- wrapper
class MoELayer:
    """One layer: owns the handle, keeps the caller's weight tensors alive.

    weights: dict with Wr [E][d], Wg/Wu [E][F][d], Wd [E][d][F], Sg/Su [F][d],
    Sd [d][F] (shared ones may be None), all on one CUDA device, bf16 or f32;
    bias: float32 [E] on the device, or None.
    """

    def __init__(self, weights: dict, top_k: int, max_tokens: int, bias=None):
        import torch
        Wr, Wg, Wd = weights["Wr"], weights["Wg"], weights["Wd"]
        E, d = Wr.shape
        F = Wg.shape[1]
        dt = {torch.bfloat16: MOE_BF16, torch.float32: MOE_F32}[Wr.dtype]
        shared = weights.get("Sg") is not None
        self.weights = weights
        self.bias = bias
        self.dtype = Wr.dtype
        self.d, self.E, self.F, self.k = d, E, F, top_k
        cfg = moe_config(d, E, top_k, F, 1 if shared else 0, max_tokens, dt,
                         _ptr(Wr), _ptr(Wg), _ptr(weights["Wu"]), _ptr(Wd),
                         _ptr(weights.get("Sg")), _ptr(weights.get("Su")),
                         _ptr(weights.get("Sd")), _ptr(bias))
        self.cfg = cfg
        self.handle = moe_create(cfg)

    def forward(self, x, out=None, stream=None):
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.d), dtype=self.dtype, device=x.device)
        moe_forward(self.handle, x, T, out, stream)
        return out

    def forward_routed(self, x, out=None, stream=None):
        """moe_forward_routed: (out, idx [T][k], w [T][k], counts [E]) -- the
        routing the forward's own kernels used."""
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.d), dtype=self.dtype, device=x.device)
        idx = torch.empty((T, self.k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, self.k), dtype=torch.float32, device=x.device)
        counts = torch.empty((self.E,), dtype=torch.int32, device=x.device)
        moe_forward_routed(self.handle, x, T, out, idx, w, counts, stream)
        return out, idx, w, counts

    def forward_host(self, x_host, out_host, stream=None):
        """moe_forward_host: x_host and out_host are CPU tensors (pinned for
        overlap); the result is there after host_join's stream work is done."""
        assert x_host.device.type == "cpu" and out_host.device.type == "cpu"
        assert x_host.is_contiguous() and out_host.is_contiguous()
        assert x_host.shape == out_host.shape and x_host.shape[1] == self.d
        assert x_host.dtype == self.dtype and out_host.dtype == self.dtype
        moe_forward_host(self.handle, x_host, x_host.shape[0], out_host, stream)
        return out_host

    def host_join(self, stream=None):
        moe_host_join(self.handle, stream)

    def route(self, x, stream=None):
        import torch
        T = x.shape[0]
        idx = torch.empty((T, self.k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, self.k), dtype=torch.float32, device=x.device)
        counts = torch.empty((self.E,), dtype=torch.int32, device=x.device)
        moe_route(self.handle, x, T, idx, w, counts, stream)
        return idx, w, counts

    def status(self, stream=None):
        return moe_status(self.handle, stream)

    def set_option(self, option: int, value: int) -> None:
        moe_set_option(self.handle, option, value)

    def close(self):
        if getattr(self, "handle", None):
            moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Q4Layer(MoELayer):
    """One layer whose expert weights are 4-bit group-affine (moe_create_q4).

    weights: dict with Wr [E][d] bf16 (the router stays bf16), and Wg, Wu, Wd,
    Sg, Su, Sd as (codes, scales, biases) triples of CUDA tensors in the layouts
    of the bf16 matrices ([E][F][d] -> codes [E][F][d/2], scales and biases
    [E][F][d/64]); shared triples None when there is no shared expert.  Runs the
    batch-1 path (one token), routing, and batches of up to max_tokens tokens
    when d and F are multiples of 512.
    """

    def __init__(self, weights: dict, top_k: int, max_tokens: int = 1, bias=None):
        import torch
        Wr = weights["Wr"]
        assert Wr.dtype == torch.bfloat16
        E, d = Wr.shape
        F = weights["Wg"][0].shape[1]
        shared = weights.get("Sg") is not None
        self.weights = weights
        self.bias = bias
        self.dtype = Wr.dtype
        self.d, self.E, self.F, self.k = d, E, F, top_k

        def mat(t):
            return moe_q4_matrix(*(None, None, None) if t is None else (_ptr(x) for x in t))

        qw = moe_q4_weights(mat(weights["Wg"]), mat(weights["Wu"]), mat(weights["Wd"]),
                            mat(weights.get("Sg")), mat(weights.get("Su")),
                            mat(weights.get("Sd")))
        cfg = moe_config(d, E, top_k, F, 1 if shared else 0, max_tokens, MOE_BF16, _ptr(Wr), None,
                         None, None, None, None, None, _ptr(bias))
        self.cfg, self.qw = cfg, qw
        self.handle = moe_create_q4(cfg, qw)


def gdn_scan(q, k, v, alpha, beta, state=None, out=None, state_out=None, stream=None):
    """Gated DeltaNet recurrent scan (include/gdn.h) over device tensors.

    q, k: bf16 [T][H_k][d_k]; v: bf16 [T][H_v][d_v]; alpha, beta: float32
    [T][H_v]; state: float32 [H_v][d_v][d_k] or None (zeros).  Returns
    (o bf16 [T][H_v][d_v], final state float32 [H_v][d_v][d_k]); `out` and
    `state_out` may be given (state_out may be `state`).  Asynchronous on
    `stream` (default: torch's current stream).
    """
    import torch
    T, Hk, dk = k.shape
    Hv, dv = v.shape[1], v.shape[2]
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("alpha", alpha, torch.float32),
                        ("beta", beta, torch.float32)):
        if t.dtype != dt or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    if q.shape != k.shape or v.shape[0] != T or alpha.shape != (T, Hv) or beta.shape != (T, Hv):
        raise ValueError("shapes of q, k, v, alpha, beta do not agree")
    if state is not None and (state.dtype != torch.float32 or tuple(state.shape) != (Hv, dv, dk)
                              or not state.is_contiguous()):
        raise ValueError("state must be a contiguous float32 [H_v][d_v][d_k] tensor")
    if out is None:
        out = torch.empty((T, Hv, dv), dtype=torch.bfloat16, device=v.device)
    if state_out is None:
        state_out = torch.empty((Hv, dv, dk), dtype=torch.float32, device=v.device)
    _check(lib().gdn_scan(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(state),
                          _ptr(state_out), _ptr(out), T, Hk, Hv, dk, dv, _stream(stream)),
           "gdn_scan")
    return out, state_out

