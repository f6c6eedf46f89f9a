"""moe_forward_host: the block on host buffers, staged through two device slots.

Every result must equal moe_forward on device copies of the same tokens bit
for bit (the same kernels run on the same values), whatever the overlap of
neighbouring calls: a call's copy-in waits only for the forward two calls back,
its copy-out runs beside the next forward.  The device forward itself is
checked against the oracle elsewhere; one case here also checks the oracle.
"""
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


def _pinned(t):
    return t.contiguous().pin_memory()


def _issue_and_compare(layer, xs, pinned=True):
    """Issue every batch back to back, join once, compare with device calls."""
    hx = [(_pinned(x) if pinned else x.clone()) for x in xs]
    hy = [torch.full_like(x, float("nan")) for x in hx]
    if pinned:
        hy = [y.pin_memory() for y in hy]
    for x, y in zip(hx, hy):
        layer.forward_host(x, y)
    layer.host_join()
    torch.cuda.synchronize()
    rc, detail = layer.status()
    assert rc == 0, f"device status {rc} detail {detail}"
    for i, (x, y) in enumerate(zip(xs, hy)):
        want = layer.forward(x.cuda()).cpu()
        assert torch.equal(y, want), f"batch {i} (T={x.shape[0]}) differs"
    return hy


def test_pipelined_batches_equal_device_calls(dev):
    """Ragged sizes, the slots grown twice (to 300, then 700 tokens: chunks of
    a 512-token handle), a one-token call (decode kernels) and a two-token one
    (small-batch kernels) between the prefill batches."""
    d, F, E, k = 512, 256, 16, 4
    w = {kk: (None if v is None else v.to(dev))
         for kk, v in synth.layer_weights(40, d, F, E, 1, "bf16", "cpu").items()}
    layer = moe.MoELayer(w, k, max_tokens=512)
    try:
        sizes = [300, 300, 120, 700, 1, 2, 300, 45]
        xs = [synth.tokens(41 + i, T, d, "bf16", "cpu") for i, T in enumerate(sizes)]
        _issue_and_compare(layer, xs)
    finally:
        layer.close()


def test_host_batches_against_oracle(dev):
    d, F, E, k, T = 512, 128, 32, 4, 200
    wc = synth.layer_weights(42, d, F, E, 1, "bf16", "cpu")
    w = {kk: (None if v is None else v.to(dev)) for kk, v in wc.items()}
    xs = [H.margined_tokens(43 + i, T, wc["Wr"], k, "bf16") for i in range(3)]
    layer = moe.MoELayer(w, k, max_tokens=T)
    try:
        ys = _issue_and_compare(layer, xs)
    finally:
        layer.close()
    for x, y in zip(xs, ys):
        ref, *_ = H.oracle_forward(x, wc, k)
        assert H.row_rel_err(y, ref).max() <= H.OUT_TOL


def test_pageable_host_buffers(dev):
    """Ordinary (pageable) host memory: the copies hold up the host, results
    are the same."""
    d, F, E, k = 512, 128, 16, 4
    w = {kk: (None if v is None else v.to(dev))
         for kk, v in synth.layer_weights(44, d, F, E, 0, "bf16", "cpu").items()}
    layer = moe.MoELayer(w, k, max_tokens=256)
    try:
        xs = [synth.tokens(45 + i, T, d, "bf16", "cpu") for i, T in enumerate([256, 77, 256])]
        _issue_and_compare(layer, xs, pinned=False)
    finally:
        layer.close()


def test_unsupported_batch_is_refused_before_any_copy(dev):
    """A 4-bit layer with F = 256 runs at most 32 tokens per batch: a 40-token
    host call returns MOE_ERR_UNSUPPORTED and leaves the output untouched."""
    w = synth.q4_layer_weights(9, 1024, 256, 16, 1, dev)
    layer = moe.Q4Layer(w, 4, max_tokens=64)
    try:
        x = _pinned(synth.tokens(46, 40, 1024, "bf16", "cpu"))
        y = torch.zeros_like(x).pin_memory()
        with pytest.raises(moe.MoeError) as e:
            layer.forward_host(x, y)
        assert e.value.code == moe.MOE_ERR_UNSUPPORTED
        layer.host_join()
        torch.cuda.synchronize()
        assert not y.any()
        _issue_and_compare(layer, [x[:2].clone(), x[2:34].clone()])
    finally:
        layer.close()


def test_full_size_batches_equal_device_calls(dev):
    """T=4096, d=2048, 256 experts top-8 + shared, F=512, bf16: three batches
    back to back, as the end-to-end benchmark issues them."""
    d, F, E, k, T = 2048, 512, 256, 8, 4096
    w = synth.layer_weights(2, d, F, E, 1, "bf16", dev)
    layer = moe.MoELayer(w, k, max_tokens=T)
    try:
        xs = [synth.tokens(1002 + i, T, d, "bf16", "cpu") for i in range(3)]
        _issue_and_compare(layer, xs)
    finally:
        layer.close()
