"""Prefill chunks captured in a CUDA graph, through the C ABI.

Every forward launch is asynchronous and allocation-free, and the kernels of a
chunk are chained by programmatic dependent launch (the router too, after the
previous kernel on the stream).  A stack of chained layers captured once must
give, at every replay with new tokens, the same bits as the same calls made
eagerly: at 1,024 tokens (cluster router, grouped GEMMs; the second layer on
the cluster-pair GEMMs, the third on the two-CTA-MMA GEMMs), at 20 tokens
(cluster router and grouped GEMMs in the same three modes) and at 12
tokens (small-batch router and grouped GEMVs).
"""
import pytest
import torch

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


@pytest.mark.parametrize("T", [1024, 20, 12])
def test_prefill_stack_in_a_cuda_graph(dev, T):
    d, F, E, k, L = 1024, 256, 64, 4, 3
    layers = [moe.MoELayer(synth.layer_weights(700 + l, d, F, E, 1, "bf16", dev), k, max_tokens=T)
              for l in range(L)]
    layers[1].set_option(moe.MOE_OPT_PAIR_MIN_TOKENS, 0)
    layers[2].set_option(moe.MOE_OPT_MMA2_MIN_TOKENS, 0)
    layers[2].set_option(moe.MOE_OPT_MMA2_DOWN_MIN_TOKENS, 0)
    try:
        x_in = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        outs = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        st = torch.cuda.Stream(device=dev)

        def stack():
            for l in range(L):
                layers[l].forward(x_in if l == 0 else outs[l - 1], out=outs[l], stream=st)

        toks = synth.tokens(710 + T, 4 * T, d, "bf16", dev)
        with torch.cuda.stream(st):
            x_in.copy_(toks[:T])
            stack()
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                stack()
        for step in range(1, 4):
            x_in.copy_(toks[step * T:(step + 1) * T])
            g.replay()
            torch.cuda.synchronize()
            got = [o.clone() for o in outs]
            h = toks[step * T:(step + 1) * T].clone()
            for l in range(L):
                h = layers[l].forward(h)
                torch.cuda.synchronize()
                assert torch.equal(got[l], h), f"step {step} layer {l}"
        for layer in layers:
            rc, detail = layer.status()
            assert rc == 0, f"device status {rc} detail {detail}"
        del g
    finally:
        for layer in layers:
            layer.close()
