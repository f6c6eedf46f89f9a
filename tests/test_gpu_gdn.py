"""Gated DeltaNet scan (include/gdn.h) against the float64 oracle.

Bars: outputs o (bf16) row-normwise relative error <= 1e-2 per (token, head)
row, the same bar as the MoE block; the final fp32 state <= 1e-4 normwise per
head (fp32 arithmetic over up to a few thousand contracting steps stays near
1e-6; bf16 output rounding is 2^-9 relative).  Piecewise scans that pass the
state along are bit-identical to one scan when cut at multiples of 8 tokens.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_mixture_experts_gemm_gb300 as moe
from sparse_mixture_experts_gemm_gb300 import synth

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
S_TOL = 1e-4


@pytest.fixture(scope="module")
def dev():
    moe.build()
    return torch.device("cuda", 0)


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _oracle(inp):
    s = inp["state"]
    return oracle.gdn_scan(_bits(inp["q"]), _bits(inp["k"]), _bits(inp["v"]),
                           inp["alpha"].cpu().numpy(), inp["beta"].cpu().numpy(),
                           None if s is None else s.cpu().numpy())


def _errs(o, s, ro, rs):
    o = o.float().cpu().numpy().astype(np.float64)
    s = s.cpu().numpy().astype(np.float64)
    oe = np.abs(o - ro).max(axis=2) / np.maximum(np.abs(ro).max(axis=2), 1e-30)
    se = np.abs(s - rs).reshape(rs.shape[0], -1).max(axis=1) / np.abs(rs).reshape(rs.shape[0], -1).max(axis=1)
    return oe.max(), se.max()


def _to(inp, dev):
    return {k: (None if v is None else v.to(dev)) for k, v in inp.items()}


def run(dev, seed, T, Hk, Hv, dv, state=True):
    inp = synth.gdn_inputs(seed, T, Hk, Hv, 128, dv, "cpu", state=state)
    d = _to(inp, dev)
    o, s = moe.gdn_scan(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["state"])
    torch.cuda.synchronize()
    ro, rs = _oracle(inp)
    oe, se = _errs(o, s, ro, rs)
    assert oe <= O_TOL, oe
    assert se <= S_TOL, se
    return o, s, oe, se


@pytest.mark.parametrize("T,Hk,Hv,dv,state", [
    (37, 2, 4, 32, True),     # one full 32-token block and a ragged one
    (1, 1, 1, 16, False),     # a single token from a zero state
    (64, 1, 3, 48, True),     # three value heads on one key head, exactly two blocks
    (300, 4, 4, 16, True),    # one value head per key head
    (37, 4, 80, 32, True),    # 160 groups of 16 columns: two groups per CTA, ragged blocks
])
def test_scan_matches_oracle(dev, T, Hk, Hv, dv, state):
    run(dev, 100 + T, T, Hk, Hv, dv, state)


def test_scan_full_size_layer(dev):
    """2,048 tokens, 16 key heads, 32 value heads, d_k = d_v = 128: every
    output and the whole final state against the oracle."""
    _, _, oe, se = run(dev, 7, 2048, 16, 32, 128, state=True)
    print(f"full size: o {oe:.2e}, state {se:.2e}")


def test_long_scan_stays_accurate(dev):
    """8,192 tokens through two heads: the fp32 state keeps its accuracy."""
    run(dev, 8, 8192, 1, 2, 16, state=True)


def test_full_forget_and_tiny_gates(dev):
    """Gates of exactly 0 (the state is wiped), tiny gates and long runs of
    small gates against the oracle."""
    inp = synth.gdn_inputs(12, 96, 2, 4, 128, 16, "cpu", state=True)
    a = inp["alpha"]
    a[5] = 0.0
    a[17, 1] = 1e-7
    a[40:80] = 0.05  # long runs of strong forgetting
    d = _to(inp, dev)
    o, s = moe.gdn_scan(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["state"])
    torch.cuda.synchronize()
    ro, rs = _oracle(inp)
    oe, se = _errs(o, s, ro, rs)
    assert oe <= O_TOL and se <= S_TOL, (oe, se)


@pytest.mark.parametrize("cut", [64, 40, 45])
def test_pieces_match_one_scan(dev, cut):
    """A scan in two pieces (the first piece's state passed on) equals one
    scan: bit for bit when the cut is a multiple of 8 tokens, else within
    float rounding (1e-5 on the state, one bf16 step on the outputs)."""
    inp = _to(synth.gdn_inputs(9, 100, 2, 4, 128, 32, "cpu", state=True), dev)
    o, s = moe.gdn_scan(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], inp["state"])
    sl = {k: inp[k] for k in ("q", "k", "v", "alpha", "beta")}
    o1, s1 = moe.gdn_scan(*(sl[k][:cut].contiguous() for k in ("q", "k", "v", "alpha", "beta")),
                          inp["state"])
    o2, s2 = moe.gdn_scan(*(sl[k][cut:].contiguous() for k in ("q", "k", "v", "alpha", "beta")), s1)
    torch.cuda.synchronize()
    op = torch.cat([o1, o2])
    if cut % 8 == 0:
        assert torch.equal(op, o)
        assert torch.equal(s2, s)
    else:
        assert ((s2 - s).abs().max() / s.abs().max()).item() <= 1e-5
        assert ((op.float() - o.float()).abs() <= o.float().abs() * 2 ** -7 + 1e-6).all()


def test_state_in_place_and_empty_scan(dev):
    inp = _to(synth.gdn_inputs(10, 40, 1, 2, 128, 16, "cpu", state=True), dev)
    ref_o, ref_s = moe.gdn_scan(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"],
                                inp["state"])
    st = inp["state"].clone()
    o, s = moe.gdn_scan(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], st, state_out=st)
    torch.cuda.synchronize()
    assert s.data_ptr() == st.data_ptr()
    assert torch.equal(o, ref_o) and torch.equal(st, ref_s)
    # T = 0: the state passes through; no initial state means zeros
    e = {k: inp[k][:0].contiguous() for k in ("q", "k", "v", "alpha", "beta")}
    _, s0 = moe.gdn_scan(e["q"], e["k"], e["v"], e["alpha"], e["beta"], inp["state"])
    _, z = moe.gdn_scan(e["q"], e["k"], e["v"], e["alpha"], e["beta"], None)
    torch.cuda.synchronize()
    assert torch.equal(s0, inp["state"]) and not z.any()


@pytest.mark.parametrize("Hk,Hv,dv", [(2, 16, 32), (8, 8, 16)])
def test_scan_head_groupings(dev, Hk, Hv, dv):
    """Eight value heads per key head, and one per key head with eight heads."""
    run(dev, 200 + Hv, 77, Hk, Hv, dv, state=True)
