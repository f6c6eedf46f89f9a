"""Batch-1 path (moe_forward with T == 1) against the oracle, through the C ABI.

The path is three kernels chained with programmatic dependent launch (router
+ shared gate/up, routed gate/up, down + combine); the handle's per-kernel
profile confirms that exactly those ran.  Bars as in the prefill tests: block
output within 1e-2 row-normwise relative error.
"""
import numpy as np
import pytest
import torch

import helpers as H
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


def _kinds_run(layer, x):
    moe.moe_profile(layer.handle, True)
    layer.forward(x)
    moe.moe_profile(layer.handle, False)
    prof = moe.moe_profile_read(layer.handle)
    return {name for name, (_, n) in prof.items() if n > 0}


# (dtype, d, F, E, k, n_shared)
CASES = [
    ("bf16", 2048, 512, 256, 8, 1),     # the full-size decode layer
    ("bf16", 2048, 512, 256, 8, 0),     # no shared expert
    ("f32", 512, 128, 256, 8, 1),       # the tiny config, fp32 throughout
    ("bf16", 256, 128, 8, 2, 1),        # few experts, short rows
    ("bf16", 1024, 256, 64, 8, 1),
    ("bf16", 4096, 1024, 16, 4, 1),     # long rows: the kernels' streamed tails
]


@pytest.mark.parametrize("dtype,d,F,E,k,n_shared", CASES)
def test_decode_matches_oracle(dev, dtype, d, F, E, k, n_shared):
    w = synth.layer_weights(50 + d + E, d, F, E, n_shared, dtype, dev)
    n_tok = 5
    x = H.margined_tokens(60 + d, n_tok, w["Wr"], k, dtype, device=dev)
    layer = moe.MoELayer(w, k, max_tokens=8)
    try:
        kinds = _kinds_run(layer, x[0:1].clone())
        assert kinds == {"decode_router", "decode_gate_up", "decode_down"}, kinds
        outs = [layer.forward(x[i:i + 1].clone()) for i in range(n_tok)]
        torch.cuda.synchronize()
        rc, detail = layer.status()
        assert rc == 0, f"device status {rc} detail {detail}"
    finally:
        layer.close()
    out = torch.cat(outs)
    ref, *_ = H.oracle_forward(x, w, k)
    err = H.row_rel_err(out, ref)
    assert err.max() <= H.OUT_TOL, err


def test_decode_layer_stack_in_a_cuda_graph(dev):
    """Four chained layers captured once and replayed with new tokens: the
    programmatic launch chain keeps each layer behind the one whose output it
    reads, and replays equal eager runs bit for bit."""
    d, F, E, k, L = 2048, 512, 256, 8, 4
    ws = [synth.layer_weights(70 + l, d, F, E, 1, "bf16", dev) for l in range(L)]
    layers = [moe.MoELayer(w, k, max_tokens=1) for w in ws]
    try:
        xin = torch.empty((1, d), dtype=torch.bfloat16, device=dev)
        outs = [torch.empty((1, d), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        stream = torch.cuda.Stream(device=dev)
        # every layer reads the previous layer's output: a real dependency
        with torch.cuda.stream(stream):
            for l in range(L):
                layers[l].forward(xin if l == 0 else outs[l - 1], out=outs[l], stream=stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                layers[l].forward(xin if l == 0 else outs[l - 1], out=outs[l], stream=stream)
        toks = synth.tokens(80, 3, d, "bf16", dev)
        for step in range(3):
            xin.copy_(toks[step:step + 1])
            g.replay()
            torch.cuda.synchronize()
            got = [o.clone() for o in outs]
            # eager reference for the same chain
            h = toks[step:step + 1].clone()
            for l in range(L):
                h = layers[l].forward(h)
                torch.cuda.synchronize()
                assert torch.equal(got[l], h), f"step {step} layer {l}"
        for layer in layers:
            assert layer.status()[0] == 0
    finally:
        for layer in layers:
            layer.close()


def test_decode_layer_stack_sample_against_oracle(dev):
    """A sample of the decode workload: fresh tokens fed through a stack of
    distinct full-size layers (each token is every layer's input), each
    (step, layer) output against the oracle, with all steps captured in one
    CUDA graph per step as the benchmark runs them."""
    d, F, E, k, L, steps = 2048, 512, 256, 8, 4, 12
    ws = [synth.layer_weights(1000 + l, d, F, E, 1, "bf16", dev) for l in range(L)]
    layers = [moe.MoELayer(w, k, max_tokens=1) for w in ws]
    try:
        xin = torch.empty((1, d), dtype=torch.bfloat16, device=dev)
        outs = torch.empty((L, d), dtype=torch.bfloat16, device=dev)
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            for l in range(L):
                layers[l].forward(xin, out=outs[l:l + 1], stream=stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                layers[l].forward(xin, out=outs[l:l + 1], stream=stream)
        # tokens with the routing margin in every layer of the stack
        cand = synth.tokens(1100, 4 * steps, d, "bf16", dev)
        keep = np.ones(4 * steps, dtype=bool)
        for l in range(L):
            _, _, logits, _ = H.oracle.route(H.np_view(cand), H.np_view(ws[l]["Wr"]), k)
            keep &= H.kth_gap(logits, k) >= H.MARGIN
        assert keep.sum() >= steps
        toks = cand[torch.as_tensor(np.nonzero(keep)[0][:steps], device=dev)].contiguous()
        got = []
        for s in range(steps):
            xin.copy_(toks[s:s + 1])
            g.replay()
            torch.cuda.synchronize()
            got.append(outs.clone())
        for layer in layers:
            assert layer.status()[0] == 0
    finally:
        for layer in layers:
            layer.close()
    for l in range(L):
        ref, *_ = H.oracle_forward(toks, ws[l], k)
        out_l = torch.stack([got[s][l] for s in range(steps)])
        err = H.row_rel_err(out_l, ref)
        assert err.max() <= H.OUT_TOL, f"layer {l}: max row rel err {err.max():.3e}"
