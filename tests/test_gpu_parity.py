"""GPU path against the CPU oracle, through the C ABI.

Bars: expert index sets and per-expert counts bit-exact; routing weights
within 1e-5; block output within 1e-2 row-normwise relative error (bf16 data,
fp32 accumulation, bf16 intermediates).  Routing is checked twice: the
standalone routing call (moe_route) and the routing the forward's own kernels
used (moe_forward_routed).  Every output row is compared, the full-size
4,096- and 16,384-token cases included, in the launch configuration the
benchmark uses; the 128K case compares two whole chunks.
"""
import numpy as np
import pytest
import torch

import helpers as H
import sparse_mixture_experts_gemm_gb300 as moe
from sparse_mixture_experts_gemm_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.lib()
    return torch.device("cuda:0")


def to_dev(w, dev):
    return {k: (None if v is None else v.to(dev)) for k, v in w.items()}


def run_case(dev, seed, T, d, F, E, k, dtype="bf16", n_shared=1, max_tokens=None, bias=None,
             rows=None, gen_device="cpu", gemv_max=None):
    w = synth.layer_weights(seed, d, F, E, n_shared, dtype, gen_device)
    x = H.margined_tokens(seed + 1000, T, w["Wr"], k, dtype, bias=bias, device=gen_device)
    wd = to_dev(w, dev)
    xd = x.to(dev)
    bd = None if bias is None else bias.to(dev)
    layer = moe.MoELayer(wd, k, max_tokens=max_tokens or max(T, 1), bias=bd)
    if gemv_max is not None:
        layer.set_option(moe.MOE_OPT_GEMV_MAX_TOKENS, gemv_max)
    try:
        if T <= layer.cfg.max_tokens:
            idx, wts, counts = layer.route(xd)
        out, f_idx, f_w, f_counts = layer.forward_routed(xd)
        torch.cuda.synchronize()
        rc, detail = layer.status()
        assert rc == 0, f"device status {rc} detail {detail}"
        ridx, rw, _, rcounts = H.oracle.route(H.np_view(x), H.np_view(w["Wr"]), k,
                                              bias=None if bias is None else bias.numpy())
        # the routing the forward's kernels used (counts summed over chunks)
        H.check_routing(f_idx, f_w, f_counts, ridx, rw, rcounts)
        if T <= layer.cfg.max_tokens:
            H.check_routing(idx, wts, counts, ridx, rw, rcounts)
        ref, oidx, ow, _ = H.oracle_forward(x, w, k, bias=bias, rows=rows)
        got = out if rows is None else out[torch.as_tensor(rows, device=dev)]
        err = H.row_rel_err(got, ref)
        assert err.max() <= H.OUT_TOL, f"max row rel err {err.max():.3e} at row {err.argmax()}"
        return out, err
    finally:
        layer.close()


def test_tiny_fp32_config(dev):
    """T=32, d=512, 256 experts top-8 + shared, F=128, fp32 throughout, seed 0."""
    _, err = run_case(dev, 0, 32, 512, 128, 256, 8, dtype="f32")
    assert err.max() < 5e-3


@pytest.mark.parametrize("T", [2, 3, 127, 128, 129, 300, 1000])
def test_bf16_multi_tile_ragged(dev, T):
    """Few experts, many rows each: several M tiles per expert with ragged tails,
    two N tiles in both GEMMs."""
    run_case(dev, 10 + T, T, 512, 256, 16, 4)


def test_bf16_mostly_empty_experts(dev):
    """256 experts, 40 tokens: most experts get no rows, some get one."""
    run_case(dev, 20, 40, 512, 128, 256, 8)


def test_bf16_no_shared_expert(dev):
    run_case(dev, 21, 200, 512, 128, 32, 4, n_shared=0)


def test_bf16_one_group_takes_every_token(dev):
    """A bias that makes experts 0..7 win for every token: 8 groups of T rows."""
    bias = torch.zeros(64)
    bias[:8] = 20.0
    run_case(dev, 22, 300, 512, 128, 64, 8, bias=bias)


def test_fp32_multi_tile(dev):
    run_case(dev, 23, 260, 256, 128, 8, 2, dtype="f32")


def test_chunking_does_not_change_output(dev):
    """Tokens are independent, so the chunk size must not change a single bit
    ("Bound temporary memory with request chunking") among chunks that take
    the same router: every chunk here holds more than 64 tokens (700 = 7 x
    100 = 2 x 350 = 1 x 700)."""
    d, F, E, k, T = 512, 128, 32, 4, 700
    w = to_dev(synth.layer_weights(30, d, F, E, 1, "bf16", "cpu"), dev)
    x = synth.tokens(31, T, d, "bf16", "cpu").to(dev)
    outs = []
    for mt in (100, 350, 1024):
        layer = moe.MoELayer(w, k, max_tokens=mt)
        outs.append(layer.forward(x))
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
        layer.close()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("dtype,q4", [("bf16", False), ("bf16", True), ("f32", False)])
def test_back_to_back_calls_equal_isolated_calls(dev, dtype, q4):
    """The kernels after the router start as programmatic dependents of their
    predecessor and wait for it inside: twelve forwards issued without a host
    synchronisation (alternating batches, chunked and unchunked, a small tail
    chunk, one-token calls between them) must equal the same forwards run
    one at a time with a synchronisation after each, bit for bit."""
    d, F, E, k = (512, 512, 32, 4) if q4 else (512, 256, 32, 4)
    if q4:
        w = synth.q4_layer_weights(50, d, F, E, 1, dev)
        layer = moe.Q4Layer(w, k, max_tokens=400)
    else:
        w = to_dev(synth.layer_weights(50, d, F, E, 1, dtype, "cpu"), dev)
        layer = moe.MoELayer(w, k, max_tokens=400)
    try:
        sizes = [1000, 1, 333, 1000, 5, 800, 1, 1000, 333, 2, 800, 1000]
        xs = [synth.tokens(51 + (i % 4), T, d, dtype, "cpu").to(dev)
              for i, T in enumerate(sizes)]
        outs = [torch.full_like(x, float("nan")) for x in xs]
        for x, o in zip(xs, outs):
            layer.forward(x, o)
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
        for i, x in enumerate(xs):
            want = layer.forward(x)
            torch.cuda.synchronize()
            assert torch.equal(outs[i], want), f"call {i} (T={sizes[i]}) differs"
        assert layer.status()[0] == 0
    finally:
        layer.close()


def test_token_permutation_equivariance(dev):
    d, F, E, k, T = 512, 128, 32, 4, 257
    w = to_dev(synth.layer_weights(32, d, F, E, 1, "bf16", "cpu"), dev)
    x = synth.tokens(33, T, d, "bf16", "cpu").to(dev)
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(3)).to(dev)
    layer = moe.MoELayer(w, k, max_tokens=T)
    a = layer.forward(x)
    b = layer.forward(x[perm].contiguous())
    torch.cuda.synchronize()
    layer.close()
    assert torch.equal(a[perm], b)


def test_decode_full_size_layer(dev):
    """Batch-1 path (d=2048, 256 experts top-8 + shared, F=512, bf16) for a few
    fresh tokens; also equal to the prefill path's result for the same token."""
    d, F, E, k = 2048, 512, 256, 8
    w = synth.layer_weights(1, d, F, E, 1, "bf16", dev)
    x = H.margined_tokens(1001, 6, w["Wr"], k, "bf16", device=dev)
    layer = moe.MoELayer(w, k, max_tokens=8)
    outs = [layer.forward(x[i:i + 1].clone()) for i in range(6)]
    pre = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.status()[0] == 0
    layer.close()
    out = torch.cat(outs)
    ref, *_ = H.oracle_forward(x, w, k)
    err = H.row_rel_err(out, ref)
    assert err.max() <= H.OUT_TOL, err
    err_pre = H.row_rel_err(pre, ref)
    assert err_pre.max() <= H.OUT_TOL, err_pre


def test_prefill_4k_full_size(dev):
    """T=4096, d=2048, 256 experts top-8 + shared, F=512, bf16: routing exact on
    every token, every output row against the oracle."""
    T = 4096
    run_case(dev, 2, T, 2048, 512, 256, 8, max_tokens=T, gen_device=dev)


def test_skewed_16k_full_size(dev):
    """T=16384 with a Zipf(1.2) router bias: a few experts take thousands of
    rows (the giant groups of the grouped GEMMs), many take none; routing
    exact on every token, every output row against the oracle."""
    T = 16384
    bias = synth.zipf_bias(3, 256, 1.2)
    _, err = run_case(dev, 3, T, 2048, 512, 256, 8, max_tokens=T, bias=bias, gen_device=dev)


def test_edge_calls(dev):
    d, F, E, k = 256, 128, 8, 2
    w = to_dev(synth.layer_weights(40, d, F, E, 1, "bf16", "cpu"), dev)
    layer = moe.MoELayer(w, k, max_tokens=16)
    x = torch.zeros((17, d), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(x)
    assert moe.lib().moe_forward(layer.handle, x.data_ptr(), 0, out.data_ptr(), None) == 0
    # misaligned pointer
    rc = moe.lib().moe_forward(layer.handle, x.data_ptr() + 2, 4, out.data_ptr(), None)
    assert rc == moe.MOE_ERR_ALIGNMENT
    # routing more tokens than one chunk
    idx = torch.empty((17, k), dtype=torch.int32, device=dev)
    wt = torch.empty((17, k), dtype=torch.float32, device=dev)
    cnt = torch.empty((E,), dtype=torch.int32, device=dev)
    rc = moe.lib().moe_route(layer.handle, x.data_ptr(), 17, idx.data_ptr(), wt.data_ptr(),
                             cnt.data_ptr(), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # overlapping in/out
    rc = moe.lib().moe_forward(layer.handle, x.data_ptr(), 4, x.data_ptr(), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    layer.close()


def test_device_timeout_is_reported_not_trapped(dev):
    """A bounded wait on a barrier nothing signals returns an error status and
    leaves the context usable."""
    d, F, E, k = 256, 128, 8, 2
    w = to_dev(synth.layer_weights(41, d, F, E, 1, "bf16", "cpu"), dev)
    layer = moe.MoELayer(w, k, max_tokens=64)
    moe.moe_debug_wait_timeout(layer.handle, 2000)
    rc, detail = layer.status()
    assert rc == moe.MOE_ERR_DEVICE_TIMEOUT and detail == 907
    assert layer.status()[0] == 0  # cleared by the read
    x = synth.tokens(42, 64, d, "bf16", "cpu").to(dev)
    layer.forward(x)
    torch.cuda.synchronize()
    assert layer.status()[0] == 0
    layer.close()


def test_long_prompt_128k_in_8k_chunks(dev):
    """T=131072 through one layer in 8192-token chunks (the long-prompt
    workload): routing and per-chunk expert counts exact on all 16 chunks,
    outputs of two whole chunks (the first and the last) against the oracle."""
    T, chunk, d, F, E, k = 131072, 8192, 2048, 512, 256, 8
    w = synth.layer_weights(4, d, F, E, 1, "bf16", dev)
    x = H.margined_tokens(1004, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.MoELayer(w, k, max_tokens=chunk)
    try:
        out, f_idx, f_w, f_counts = layer.forward_routed(x)
        routes = [layer.route(x[c0:c0 + chunk]) for c0 in range(0, T, chunk)]
        torch.cuda.synchronize()
        rc, detail = layer.status()
        assert rc == 0, f"device status {rc} detail {detail}"
    finally:
        layer.close()
    wr = H.np_view(w["Wr"])
    rcount_sum = np.zeros(E, dtype=np.int64)
    for ci, (idx, wts, counts) in enumerate(routes):
        xs = x[ci * chunk:(ci + 1) * chunk]
        ridx, rw, _, rcounts = H.oracle.route(H.np_view(xs), wr, k)
        H.check_routing(idx, wts, counts, ridx, rw, rcounts)
        # the forward's own routing of this chunk is the same
        sl = slice(ci * chunk, (ci + 1) * chunk)
        H.check_routing(f_idx[sl], f_w[sl], None, ridx, rw, None)
        rcount_sum += rcounts
    assert np.array_equal(f_counts.cpu().numpy(), rcount_sum), "call counts over 16 chunks"
    for ci in (0, T // chunk - 1):
        rows = np.arange(ci * chunk, (ci + 1) * chunk)
        ref, *_ = H.oracle_forward(x, w, k, rows=rows)
        err = H.row_rel_err(out[torch.as_tensor(rows, device=dev)], ref)
        assert err.max() <= H.OUT_TOL, f"chunk {ci}: max row rel err {err.max():.3e}"


@pytest.mark.parametrize("T,gemv_max", [(2, None), (5, None), (16, None), (17, None), (32, None),
                                        (33, None), (64, None), (17, 32), (32, 32), (8, 0)])
def test_small_batch_routing_path(dev, T, gemv_max):
    """Batches of at most 64 bf16 tokens route through one cluster launch (no
    placement kernel); up to the GEMV limit (16 by default, set here to 32
    or 0 as well) they then take the grouped GEMV (two column blocks up to
    16 tokens, four beyond), larger ones the grouped GEMMs: the full-size
    layer against the oracle, every output, and the kernel kinds."""
    d, F, E, k = 2048, 512, 256, 8
    w = synth.layer_weights(400 + T, d, F, E, 1, "bf16", dev)
    x = H.margined_tokens(410 + T, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.MoELayer(w, k, max_tokens=64)
    if gemv_max is not None:
        layer.set_option(moe.MOE_OPT_GEMV_MAX_TOKENS, gemv_max)
    limit = 16 if gemv_max is None else gemv_max
    try:
        moe.moe_profile(layer.handle, True)
        out = layer.forward(x)
        moe.moe_profile(layer.handle, False)
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
        kinds = {name for name, (_, n) in moe.moe_profile_read(layer.handle).items() if n > 0}
        want = ({"router", "gemv_gate_up", "gemv_down", "combine"} if T <= limit
                else {"router", "gemm_gate_up", "gemm_down", "combine"})
        assert kinds == want, kinds
    finally:
        layer.close()
    ref, *_ = H.oracle_forward(x, w, k)
    err = H.row_rel_err(out, ref)
    assert err.max() <= H.OUT_TOL, err.max()


def test_small_batch_with_router_bias(dev):
    """The small-batch router adds the per-expert bias before the selection."""
    E, k = 64, 8
    bias = synth.zipf_bias(7, E, 1.2)
    run_case(dev, 44, 9, 512, 128, E, k, bias=bias)


@pytest.mark.parametrize("T,E,k,n_shared", [(16, 4, 2, 1), (13, 8, 3, 0), (9, 2, 1, 1), (3, 8, 2, 0),
                                            (32, 4, 2, 1), (29, 2, 1, 0), (24, 3, 2, 1)])
def test_small_batch_crowded_experts(dev, T, E, k, n_shared):
    """Small batches whose routed experts get more than 8 (up to 32) tokens:
    the second to fourth column blocks of the grouped GEMV (its limit set to
    32 tokens), with and without the shared expert."""
    run_case(dev, 50 + T, T, 256, 128, E, k, n_shared=n_shared, max_tokens=32, gemv_max=32)


def test_chunks_of_up_to_64_tokens_mix_paths(dev):
    """130 tokens on a 48-token handle: chunks of 48 (cluster routing, grouped
    GEMMs), 48 and 34 (the same), every output against the oracle; and 60
    tokens on a 40-token handle: 40 (cluster routing, grouped GEMMs) then 20
    (cluster routing, four-block grouped GEMV with its limit at 32)."""
    run_case(dev, 95, 130, 512, 128, 32, 4, max_tokens=48)
    run_case(dev, 96, 60, 512, 128, 32, 4, max_tokens=40, gemv_max=32)


def test_chunked_prefill_with_a_small_tail(dev):
    """A 1,000-token batch on a 248-token handle: four full chunks on the
    grouped GEMMs, then an 8-token tail on the small-batch kernels; every
    output against the oracle."""
    run_case(dev, 91, 1000, 512, 128, 32, 4, max_tokens=248)


def test_small_batch_beyond_the_router_limit(dev):
    """16 tokens of d = 8192 (256 KB of tokens) do not fit the small router's
    shared memory: the batch takes the tensor-core router and grouped GEMMs."""
    d, F, E, k, T = 8192, 128, 16, 2, 16
    w = synth.layer_weights(92, d, F, E, 1, "bf16", dev)
    x = H.margined_tokens(93, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.MoELayer(w, k, max_tokens=T)
    try:
        moe.moe_profile(layer.handle, True)
        out = layer.forward(x)
        moe.moe_profile(layer.handle, False)
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
        kinds = {name for name, (_, n) in moe.moe_profile_read(layer.handle).items() if n > 0}
        assert kinds == {"router", "gemm_gate_up", "gemm_down", "combine"}, kinds
    finally:
        layer.close()
    ref, *_ = H.oracle_forward(x, w, k)
    assert H.row_rel_err(out, ref).max() <= H.OUT_TOL


def test_small_batch_partial_router_cluster(dev):
    """40 experts: a cluster of three router CTAs, the last one holding only
    8 experts (its other warps clamp to a valid row and write nothing)."""
    run_case(dev, 94, 11, 512, 128, 40, 6, n_shared=1, max_tokens=16)
