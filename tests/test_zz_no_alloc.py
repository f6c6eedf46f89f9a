"""The allocation-free batch-1 entry point, moe_decode_noalloc.

It serves callers that cannot allocate device memory (and therefore cannot
create a handle, since moe_create allocates the workspace): its scratch is a
static array inside the library.  Its output must match the handle-based
moe_forward with T == 1 on consecutive calls: the array keeps the previous
call's contents, and no value of one call may leak into the next.
This file is collected last so that a failure here does not hide the others.
"""
import ctypes

import pytest
import torch

import helpers as H
import sparse_mixture_experts_gemm_gb300 as moe
from sparse_mixture_experts_gemm_gb300 import synth


def test_rejects_layers_beyond_the_static_scratch():
    moe.build()
    c = moe.moe_config(2048, 256, 8, 4096, 1, 1, moe.MOE_BF16, 0x1000, 0x2000, 0x3000, 0x4000,
                       0x5000, 0x6000, 0x7000, None)
    rc = moe.lib().moe_decode_noalloc(ctypes.byref(c), 0x8000, 0x9000, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,d,F,E,k", [("bf16", 2048, 512, 256, 8), ("f32", 512, 128, 256, 8)])
def test_noalloc_matches_handle_path_on_consecutive_calls(dtype, d, F, E, k):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    dev = torch.device("cuda:0")
    w = synth.layer_weights(77, d, F, E, 1, dtype, dev)
    xs = synth.tokens(78, 2, d, dtype, dev)
    layer = moe.MoELayer(w, k, max_tokens=4)
    cfg = layer.cfg
    lib = moe.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for i in range(2):  # two calls in a row, different tokens
        x = xs[i:i + 1].contiguous()
        ref = layer.forward(x)
        out = torch.full_like(x, float("nan"))
        rc = lib.moe_decode_noalloc(ctypes.byref(cfg), x.data_ptr(), out.data_ptr(), stream)
        assert rc == moe.MOE_OK
        torch.cuda.synchronize()
        err = H.row_rel_err(out, ref.double().cpu().numpy())
        assert err.max() <= H.OUT_TOL, f"call {i}: rel err {err.max():.3e}"
    assert layer.status()[0] == 0
    layer.close()
