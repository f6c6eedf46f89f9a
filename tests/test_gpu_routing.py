"""The routing each path's own kernels compute and use, against the oracle.

moe_forward_routed hands back, next to the block's output, the expert indices
and weights its kernels chose for every token and the per-expert counts they
built ("Keep expert routing on the GPU": top-8, histogram, all on the GPU).
Every path is checked here through that call, not through a separate routing
launch: the batch-1 kernels (bf16, fp32 and 4-bit weights), the small-batch
cluster router, the tensor-core router of large chunks (counts summed over
chunks) and the fp32 router.  Bars: index sets and counts bit-exact, weights
within 1e-5 (inputs carry the routing margin, so no tie decides a choice).

The decode workload itself (fresh tokens through 40 distinct full-size
layers, 1,000 timed steps, replayed from one CUDA graph per step as the
benchmark runs it) is checked on all 1,000 x 40 (step, layer) routes, and on
the block outputs of 50 steps x 40 layers in full.
"""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
import sparse_mixture_experts_gemm_gb300 as moe
from sparse_mixture_experts_gemm_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.lib()
    return torch.device("cuda:0")


def _routed(layer, x, wr, k, bias=None, kinds=None):
    """forward_routed on x; routing checked against the oracle's router.
    kinds: the kernel kinds the call must launch (checked with the profile)."""
    if kinds is not None:
        moe.moe_profile(layer.handle, True)
    out, idx, w, counts = layer.forward_routed(x)
    if kinds is not None:
        moe.moe_profile(layer.handle, False)
    torch.cuda.synchronize()
    rc, detail = layer.status()
    assert rc == 0, f"device status {rc} detail {detail}"
    if kinds is not None:
        got = {n for n, (_, c) in moe.moe_profile_read(layer.handle).items() if c > 0}
        assert got == kinds, got
    b = None if bias is None else bias.detach().cpu().numpy().astype(np.float32)
    ridx, rw, _, rcounts = oracle.route(H.np_view(x), H.np_view(wr), k, bias=b)
    H.check_routing(idx, w, counts, ridx, rw, rcounts)
    return out, idx


DECODE = {"decode_router", "decode_gate_up", "decode_down"}
SMALL = {"router", "gemv_gate_up", "gemv_down", "combine"}
PREFILL = {"router", "gemm_gate_up", "gemm_down", "combine"}


@pytest.mark.parametrize("dtype,d,F,E,k,n_shared", [
    ("bf16", 2048, 512, 256, 8, 1),
    ("bf16", 1024, 256, 64, 8, 0),
    ("f32", 512, 128, 256, 8, 1),
])
def test_decode_kernels_routing(dev, dtype, d, F, E, k, n_shared):
    """T == 1: the top-k that the batch-1 gate/up kernel takes, per token."""
    w = synth.layer_weights(600 + d, d, F, E, n_shared, dtype, dev)
    x = H.margined_tokens(610 + d, 6, w["Wr"], k, dtype, device=dev)
    layer = moe.MoELayer(w, k, max_tokens=4)
    try:
        for i in range(x.shape[0]):
            _routed(layer, x[i:i + 1].clone(), w["Wr"], k, kinds=DECODE if i == 0 else None)
    finally:
        layer.close()


def test_decode_kernels_routing_with_bias(dev):
    d, F, E, k = 512, 128, 64, 8
    w = synth.layer_weights(620, d, F, E, 1, "bf16", dev)
    bias = synth.zipf_bias(621, E, 1.2).to(dev)
    x = H.margined_tokens(622, 5, w["Wr"], k, "bf16", bias=bias.cpu(), device=dev)
    layer = moe.MoELayer(w, k, max_tokens=1, bias=bias)
    try:
        for i in range(x.shape[0]):
            _routed(layer, x[i:i + 1].clone(), w["Wr"], k, bias=bias)
    finally:
        layer.close()


def test_q4_decode_kernels_routing(dev):
    """T == 1 on 4-bit expert weights: the top-k the router cluster publishes."""
    d, F, E, k = 2048, 512, 256, 8
    w = synth.q4_layer_weights(630, d, F, E, 1, dev)
    x = H.margined_tokens(631, 5, w["Wr"], k, "bf16", device=dev)
    layer = moe.Q4Layer(w, k)
    try:
        for i in range(x.shape[0]):
            _routed(layer, x[i:i + 1].clone(), w["Wr"], k, kinds=DECODE if i == 0 else None)
    finally:
        layer.close()


@pytest.mark.parametrize("T", [2, 5, 16, 17, 32, 33, 64])
def test_small_batch_router_routing(dev, T):
    """2..64 bf16 tokens: the cluster router's choice, weights and group sizes
    (tokens in passes of 16), before the grouped GEMV (at most 16 tokens of a
    bf16 layer) or the grouped GEMMs."""
    d, F, E, k = 2048, 512, 256, 8
    w = synth.layer_weights(640 + T, d, F, E, 1, "bf16", dev)
    x = H.margined_tokens(650 + T, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.MoELayer(w, k, max_tokens=64)
    try:
        _routed(layer, x, w["Wr"], k, kinds=SMALL if T <= 16 else PREFILL)
    finally:
        layer.close()


def test_q4_small_batch_routing(dev):
    d, F, E, k, T = 2048, 512, 256, 8, 7
    w = synth.q4_layer_weights(660, d, F, E, 1, dev)
    x = H.margined_tokens(661, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.Q4Layer(w, k, max_tokens=16)
    try:
        _routed(layer, x, w["Wr"], k, kinds=SMALL)
    finally:
        layer.close()


def test_chunked_prefill_routing_sums_counts_over_chunks(dev):
    """1,000 tokens on a 248-token handle: four chunks on the tensor-core router
    and an 8-token tail on the small-batch router, in one call; the counts are
    the whole call's."""
    d, F, E, k, T = 512, 128, 32, 4, 1000
    w = synth.layer_weights(670, d, F, E, 1, "bf16", dev)
    x = H.margined_tokens(671, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.MoELayer(w, k, max_tokens=248)
    try:
        _routed(layer, x, w["Wr"], k)
    finally:
        layer.close()


def test_fp32_router_routing(dev):
    """The fp32 configuration (tiny instance): the SIMT router's choice."""
    d, F, E, k, T = 512, 128, 256, 8, 32
    w = synth.layer_weights(0, d, F, E, 1, "f32", dev)
    x = H.margined_tokens(1000, T, w["Wr"], k, "f32", device=dev)
    layer = moe.MoELayer(w, k, max_tokens=20)  # two chunks
    try:
        _routed(layer, x, w["Wr"], k)
    finally:
        layer.close()


def test_q4_prefill_routing(dev):
    d, F, E, k, T = 2048, 512, 256, 8, 600
    w = synth.q4_layer_weights(680, d, F, E, 1, dev)
    x = H.margined_tokens(681, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.Q4Layer(w, k, max_tokens=T)
    try:
        _routed(layer, x, w["Wr"], k, kinds=PREFILL)
    finally:
        layer.close()


def test_routed_forward_equals_plain_forward(dev):
    """Handing back the routing changes no output bit, on every path."""
    d, F, E, k = 512, 256, 32, 4
    w = synth.layer_weights(690, d, F, E, 1, "bf16", dev)
    layer = moe.MoELayer(w, k, max_tokens=300)
    try:
        for T in (1, 3, 16, 17, 300, 777):
            x = synth.tokens(691 + T, T, d, "bf16", dev)
            a = layer.forward(x)
            b, *_ = layer.forward_routed(x)
            torch.cuda.synchronize()
            assert torch.equal(a, b), T
        assert layer.status()[0] == 0
    finally:
        layer.close()


# ------------------------------------------------------------ decode workload
DEC_LAYERS, DEC_STEPS, DEC_WARMUP, DEC_FULL = 40, 1000, 50, 50


def test_decode_workload_every_step_and_layer(dev):
    """The batch-1 decode workload as the benchmark runs it: 40 distinct
    full-size layers (seeds 1000 + l), one fresh token per step (the
    benchmark's seeded tokens, its 1,000 timed steps after 50 warm-up ones),
    each token the input of every layer, one CUDA graph replayed per step.
    Every (step, layer) route is compared with the oracle: exact where the
    oracle's k-th/(k+1)-th logit gap is at least the margin, and where it is
    not (these tokens are not re-drawn), the GPU's set must still be a top-k
    within the fp32 rounding of the logits.  The block outputs of the first 50
    steps whose routes all have the margin are compared with the oracle in
    full (all 40 layers)."""
    d, F, E, k, L = 2048, 512, 256, 8, DEC_LAYERS
    ws = [synth.layer_weights(1000 + l, d, F, E, 1, "bf16", dev) for l in range(L)]
    layers = [moe.MoELayer(w, k, max_tokens=1) for w in ws]
    xs = synth.tokens(1, DEC_STEPS + DEC_WARMUP, d, "bf16", dev)[DEC_WARMUP:].contiguous()
    try:
        x_in = torch.empty((1, d), dtype=torch.bfloat16, device=dev)
        outs = torch.empty((L, d), dtype=torch.bfloat16, device=dev)
        idx = torch.empty((L, k), dtype=torch.int32, device=dev)
        wts = torch.empty((L, k), dtype=torch.float32, device=dev)
        cnt = torch.empty((L, E), dtype=torch.int32, device=dev)
        st = torch.cuda.Stream(device=dev)

        def step():
            for l in range(L):
                moe.moe_forward_routed(layers[l].handle, x_in, 1, outs[l:l + 1], idx[l:l + 1],
                                       wts[l:l + 1], cnt[l], st)

        with torch.cuda.stream(st):
            x_in.copy_(xs[0:1])
            step()
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                step()
            h_idx = torch.empty((DEC_STEPS, L, k), dtype=torch.int32, device=dev)
            h_w = torch.empty((DEC_STEPS, L, k), dtype=torch.float32, device=dev)
            h_cnt = torch.empty((DEC_STEPS, L, E), dtype=torch.int32, device=dev)
            h_out = torch.empty((DEC_STEPS, L, d), dtype=torch.bfloat16, device=dev)
            for s in range(DEC_STEPS):
                x_in.copy_(xs[s:s + 1])
                g.replay()
                h_idx[s].copy_(idx)
                h_w[s].copy_(wts)
                h_cnt[s].copy_(cnt)
                h_out[s].copy_(outs)
            st.synchronize()
        for layer in layers:
            rc, detail = layer.status()
            assert rc == 0, f"device status {rc} detail {detail}"
        del g
    finally:
        for layer in layers:
            layer.close()

    gi = h_idx.cpu().numpy()
    gw = h_w.cpu().numpy().astype(np.float64)
    gc = h_cnt.cpu().numpy()
    x_np = H.np_view(xs)
    margined = np.ones((DEC_STEPS, L), dtype=bool)
    near = 0
    for l in range(L):
        ridx, rw, logits, _ = oracle.route(x_np, H.np_view(ws[l]["Wr"]), k)
        gap = H.kth_gap(logits, k)
        ok = gap >= H.MARGIN
        margined[:, l] = ok
        a = np.sort(gi[:, l], axis=1)
        b = np.sort(ridx, axis=1)
        bad = np.nonzero(ok & (a != b).any(1))[0]
        assert len(bad) == 0, f"layer {l}: steps {bad[:5]} routed differently"
        og = np.argsort(gi[:, l], axis=1, kind="stable")
        orf = np.argsort(ridx, axis=1, kind="stable")
        dw = np.abs(np.take_along_axis(gw[:, l], og, 1) - np.take_along_axis(rw, orf, 1))
        assert dw[ok].max() <= H.W_TOL, f"layer {l}: routing weight error {dw[ok].max():.3e}"
        # near ties: the GPU's set is still the k largest within fp32 rounding
        for s in np.nonzero(~ok)[0]:
            chosen = np.zeros(E, dtype=bool)
            chosen[gi[s, l]] = True
            lg = logits[s].astype(np.float64)
            assert lg[chosen].min() >= lg[~chosen].max() - 1e-4, (s, l)
            near += 1
        # counts: one per chosen expert, as the kernels used them
        onehot = np.zeros((DEC_STEPS, E), dtype=np.int64)
        np.add.at(onehot, (np.repeat(np.arange(DEC_STEPS), k), gi[:, l].reshape(-1)), 1)
        assert np.array_equal(gc[:, l], onehot), f"layer {l}: counts differ from the choice"
        assert np.allclose(gw[:, l].sum(1), 1.0, atol=1e-6)
    assert near < 0.05 * DEC_STEPS * L, near

    full = np.nonzero(margined.all(1))[0][:DEC_FULL]
    assert len(full) == DEC_FULL, len(full)
    rows = torch.as_tensor(full, device=dev)
    got = h_out[rows]
    for l in range(L):
        ref, *_ = H.oracle_forward(xs, ws[l], k, rows=full)
        err = H.row_rel_err(got[:, l], ref)
        assert err.max() <= H.OUT_TOL, f"layer {l}: max row rel err {err.max():.3e}"
