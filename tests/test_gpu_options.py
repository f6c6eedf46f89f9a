"""Launch options that must not change a result bit, through the C ABI.

* MOE_OPT_PAIR_MIN_TOKENS: grouped GEMMs on clusters of two CTAs.  Two CTAs
  of a thread-block cluster multiply consecutive 128-row tiles of one expert
  group with the same weight tile, each loading half of it into both; a
  group's last tile (odd tile counts) runs beside the next N tile of the same
  rows, and with an odd number of N tiles one CTA of the last item runs
  without rows.  Every tile is the same MMA sequence as in the one-CTA mode.
* MOE_OPT_MMA2_MIN_TOKENS / MOE_OPT_MMA2_DOWN_MIN_TOKENS: the gate/up and
  the down GEMM on the two-CTA MMA.  A cluster of two CTAs computes 256 x 256
  tiles (M tiles 2q and 2q + 1 of a group; with an odd tile count the second
  CTA of a group's last items has no rows), each CTA staging half of the
  weight tile; the MMA runs over K in the same order.

Outputs must be equal bit for bit across the settings; each case is also
checked against the oracle on every row (1e-2 row-normwise).
"""
import pytest
import torch

import helpers as H
import oracle
import sparse_mixture_experts_gemm_gb300 as moe
from sparse_mixture_experts_gemm_gb300 import synth

pytestmark = pytest.mark.gpu

OFF = 1 << 40  # no chunk is that large


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.lib()
    return torch.device("cuda:0")


def run_mode(layer, x, pair, mma2, mma2_down):
    layer.set_option(moe.MOE_OPT_PAIR_MIN_TOKENS, pair)
    layer.set_option(moe.MOE_OPT_MMA2_MIN_TOKENS, mma2)
    layer.set_option(moe.MOE_OPT_MMA2_DOWN_MIN_TOKENS, mma2_down)
    out = layer.forward(x)
    torch.cuda.synchronize()
    rc, detail = layer.status()
    assert rc == 0, f"device status {rc} detail {detail} (options {pair}, {mma2}, {mma2_down})"
    return out


def both_modes(layer, x):
    """Outputs of the one-CTA, cluster-pair and two-CTA-MMA grouped GEMMs
    (the last also checked with a one-CTA down GEMM after it)."""
    one = run_mode(layer, x, OFF, OFF, OFF)
    pair = run_mode(layer, x, 0, OFF, OFF)
    mma2 = run_mode(layer, x, OFF, 0, 0)
    mixed = run_mode(layer, x, OFF, 0, OFF)
    assert_bit_equal(mma2, mixed, "two-CTA gate/up + one-CTA down")
    return one, pair, mma2


def assert_bit_equal(one, other, what):
    if not torch.equal(one, other):
        diff = (one.float() - other.float()).abs()
        rows = torch.nonzero(diff.amax(dim=1) > 0).flatten()
        raise AssertionError(f"{what}: {rows.numel()} rows differ (first {rows[:8].tolist()}), "
                             f"max abs diff {diff.max().item():.3e}")


# (seed, T, d, F, E, k, n_shared, max_tokens, skew)
CASES = [
    (50, 700, 768, 384, 16, 4, 1, 700, False),   # 3 N tiles in both GEMMs: idle CTAs
    (51, 1000, 512, 256, 8, 2, 0, 1000, False),  # no shared expert, several M tiles per group
    (52, 129, 512, 256, 16, 4, 1, 129, False),   # single-tile groups only
    (53, 300, 512, 128, 64, 8, 1, 300, True),    # 8 groups of 300 rows (3 M tiles each)
    (54, 3000, 512, 256, 32, 4, 1, 1024, False),  # chunks of 1024, 1024, 952
    (55, 128, 512, 256, 16, 4, 1, 128, True),    # 4 groups of exactly 128 rows, 12 empty
    (56, 256, 512, 256, 16, 4, 1, 256, True),    # 4 groups of exactly 256 rows: full pairs
    (57, 384, 768, 128, 16, 4, 0, 384, True),    # 3 M tiles per group, no shared expert
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[1]}_d{c[2]}_F{c[3]}_E{c[4]}")
def test_cluster_modes_equal_one_cta_mode_and_oracle(dev, case):
    seed, T, d, F, E, k, n_shared, max_tokens, skew = case
    bias = None
    if skew:
        bias = torch.zeros(E)
        bias[:k] = 20.0
    w = synth.layer_weights(seed, d, F, E, n_shared, "bf16", "cpu")
    x = H.margined_tokens(seed + 1000, T, w["Wr"], k, "bf16", bias=bias, device="cpu")
    wd = {kk: (None if v is None else v.to(dev)) for kk, v in w.items()}
    layer = moe.MoELayer(wd, k, max_tokens=max_tokens, bias=None if bias is None else bias.to(dev))
    try:
        one, pair, mma2 = both_modes(layer, x.to(dev))
    finally:
        layer.close()
    assert_bit_equal(one, pair, "cluster pair")
    ref, *_ = H.oracle_forward(x, w, k, bias=bias)
    for name, out in (("cluster pair", pair), ("two-CTA MMA", mma2)):
        err = H.row_rel_err(out, ref)
        assert err.max() <= H.OUT_TOL, f"{name}: max row rel err {err.max():.3e} at row {err.argmax()}"
    assert_bit_equal(one, mma2, "two-CTA MMA")


def test_cluster_modes_full_size_4k_bit_equal(dev):
    """T=4096, d=2048, 256 experts top-8 + shared, F=512 (the one-CTA result is
    checked against the oracle on every row in test_gpu_parity)."""
    d, F, E, k, T = 2048, 512, 256, 8, 4096
    w = synth.layer_weights(2, d, F, E, 1, "bf16", dev)
    x = H.margined_tokens(1002, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.MoELayer(w, k, max_tokens=T)
    try:
        one, pair, mma2 = both_modes(layer, x)
    finally:
        layer.close()
    assert_bit_equal(one, pair, "cluster pair")
    assert_bit_equal(one, mma2, "two-CTA MMA")


def test_cluster_modes_full_size_16k_skewed_bit_equal(dev):
    """T=16384 with the Zipf(1.2) router bias: giant groups of many M tiles."""
    d, F, E, k, T = 2048, 512, 256, 8, 16384
    bias = synth.zipf_bias(3, E, 1.2)
    w = synth.layer_weights(3, d, F, E, 1, "bf16", dev)
    x = H.margined_tokens(1003, T, w["Wr"], k, "bf16", bias=bias, device=dev)
    layer = moe.MoELayer(w, k, max_tokens=T, bias=bias.to(dev))
    try:
        one, pair, mma2 = both_modes(layer, x)
    finally:
        layer.close()
    assert_bit_equal(one, pair, "cluster pair")
    assert_bit_equal(one, mma2, "two-CTA MMA")


@pytest.mark.parametrize("T,d,E,k", [(300, 2048, 256, 8), (4096, 2048, 256, 8), (1000, 768, 64, 4)],
                         ids=lambda v: str(v))
def test_router_clusters_of_two_equal_clusters_of_four(dev, T, d, E, k):
    """MOE_OPT_ROUTER_PAIR_MIN_TOKENS: the cluster router on clusters of two
    CTAs (each half of d, its two quarter partials added before the
    exchange) against clusters of four (one quarter each): the logits are
    (q0 + q1) + (q2 + q3) either way, so indices, weights, counts and the
    layer's output must be equal bit for bit; routing also against the oracle."""
    F = 256
    w = synth.layer_weights(60 + T, d, F, E, 1, "bf16", dev)
    x = H.margined_tokens(1060 + T, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.MoELayer(w, k, max_tokens=T)
    res = {}
    try:
        for name, v in (("four", OFF), ("two", 0)):
            layer.set_option(moe.MOE_OPT_ROUTER_PAIR_MIN_TOKENS, v)
            idx, wt, counts = layer.route(x)
            out = layer.forward(x)
            torch.cuda.synchronize()
            rc, detail = layer.status()
            assert rc == 0, f"device status {rc} detail {detail} ({name})"
            res[name] = (idx, wt, counts, out)
    finally:
        layer.close()
    for a, b, what in zip(res["four"], res["two"], ("indices", "weights", "counts", "output")):
        assert_bit_equal(a.reshape(a.shape[0], -1), b.reshape(b.shape[0], -1), f"router clusters: {what}")
    idx_ref, w_ref, _, counts_ref = oracle.route(H.np_view(x), H.np_view(w["Wr"]), k)
    H.check_routing(*res["two"][:3], idx_ref, w_ref, counts_ref)
