"""The allocation-free batch-1 entry point, moe_decode_noalloc.

It serves callers that cannot allocate device memory and therefore cannot
create a handle (moe_create allocates the handle's workspace): an
application whose allocator owns the whole device pool, a serving loop that
must not allocate once it runs, a plugin that is only handed device pointers.
Its scratch, and its device status word, live in a static array inside the
library.

Checked here, through the C ABI: on two calls in a row with different tokens
its output equals the handle-based moe_forward with T == 1 bit for bit (the
same kernels on the same inputs; the array keeps the previous call's
contents, and nothing of one call may leak into the next) and is within the
block's 1e-2 bar of the oracle; its status word reads clean after those
calls, and a device wait that runs out is reported through it
(moe_noalloc_status) instead of being lost.
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
    xs = H.margined_tokens(78, 2, w["Wr"], k, dtype, device=dev)
    layer = moe.MoELayer(w, k, max_tokens=4)
    cfg = layer.cfg
    lib = moe.lib()
    stream = torch.cuda.current_stream().cuda_stream
    try:
        # a clean status word to start from (an earlier test may have used it)
        moe.moe_noalloc_status()
        outs = []
        for i in range(2):  # two calls in a row, different tokens
            x = xs[i:i + 1].contiguous()
            ref = layer.forward(x)
            out = torch.full_like(x, float("nan"))
            rc = lib.moe_decode_noalloc(ctypes.byref(cfg), x.data_ptr(), out.data_ptr(), stream)
            assert rc == moe.MOE_OK
            torch.cuda.synchronize()
            assert torch.equal(out, ref), f"call {i}: differs from the handle path"
            outs.append(out)
        assert moe.moe_noalloc_status() == (moe.MOE_OK, 0)
        assert layer.status()[0] == 0
    finally:
        layer.close()
    want, *_ = H.oracle_forward(xs, w, k)
    err = H.row_rel_err(torch.cat(outs), want)
    assert err.max() <= H.OUT_TOL, f"rel err against the oracle {err.max():.3e}"


@pytest.mark.gpu
def test_noalloc_reports_a_device_timeout():
    """A bounded wait that runs out is recorded in the entry point's own status
    word (the test hook's wait on a barrier nothing signals, with no handle)
    and read back, then cleared, by moe_noalloc_status; a call after it still
    runs clean."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    dev = torch.device("cuda:0")
    moe.moe_noalloc_status()
    moe.moe_debug_wait_timeout(None, 2000)
    rc, detail = moe.moe_noalloc_status()
    assert rc == moe.MOE_ERR_DEVICE_TIMEOUT and detail == 907, (rc, detail)
    assert moe.moe_noalloc_status() == (moe.MOE_OK, 0)  # cleared by the read
    d, F, E, k = 512, 128, 16, 4
    w = synth.layer_weights(79, d, F, E, 1, "bf16", dev)
    layer = moe.MoELayer(w, k, max_tokens=1)
    try:
        x = synth.tokens(80, 1, d, "bf16", dev)
        out = torch.empty_like(x)
        moe.moe_decode_noalloc(layer.cfg, x, out)
        ref = layer.forward(x)
        torch.cuda.synchronize()
        assert moe.moe_noalloc_status() == (moe.MOE_OK, 0)
        assert torch.equal(out, ref)
    finally:
        layer.close()
