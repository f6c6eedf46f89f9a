"""Pins of the CPU oracle to things other than itself.

Each ``pin_*`` takes ``mutation`` (0 = the oracle as committed; n > 0 = a build of
moe_oracle.c with planted mistake n) and raises AssertionError when the oracle
disagrees with what the mathematics fixes:

* brute force: every expert on every token, masked by a top-k taken with
  numpy's argsort (a different selection routine than the oracle's);
* library routines: scipy's softmax, torch's silu and matmul in float64;
* closed forms: two-expert routing weights are a logistic function of the
  logit gap; hand-derived tiny blocks (tests/golden/hand_cases.json);
* invariants: routing weights sum to 1, counts sum to T*k, token-permutation
  equivariance.

The block these pins fix is the one of "Optimizing on-device inference for
Apple Silicon", section "Qwen creates three distinct workload shapes" (router
over 256 experts picks 8, plus one shared expert) and section "Reduce
intermediate traffic and dispatch traffic" (gated input projections, output
projection scaled by the routing score, shared result added).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special
import torch
import torch.nn.functional as Fnn

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng_case(seed, T, d, F, E, n_shared=1, dtype=np.float32):
    r = np.random.default_rng(seed)
    x = r.standard_normal((T, d)).astype(np.float32)
    wr = (r.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    wg = (r.standard_normal((E, F, d)) / math.sqrt(d)).astype(np.float32)
    wu = (r.standard_normal((E, F, d)) / math.sqrt(d)).astype(np.float32)
    wd = (r.standard_normal((E, d, F)) / math.sqrt(F)).astype(np.float32)
    if n_shared:
        sg = (r.standard_normal((F, d)) / math.sqrt(d)).astype(np.float32)
        su = (r.standard_normal((F, d)) / math.sqrt(d)).astype(np.float32)
        sd = (r.standard_normal((d, F)) / math.sqrt(F)).astype(np.float32)
    else:
        sg = su = sd = None
    return dict(x=x, wr=wr, wg=wg, wu=wu, wd=wd, sg=sg, su=su, sd=sd)


def _topk_numpy(logits32: np.ndarray, k: int) -> np.ndarray:
    """Per-row indices of the k largest values, ties to the lower index (stable sort of -l)."""
    order = np.argsort(-logits32.astype(np.float64), axis=1, kind="stable")
    return order[:, :k]


def pin_route_vs_numpy(mutation=0):
    """Selection, weights and counts against numpy/scipy on random inputs."""
    c = _rng_case(11, 48, 40, 8, 24, n_shared=0)
    k = 5
    idx, w, logits, counts = oracle.route(c["x"], c["wr"], k, nthreads=2, mutation=mutation)
    ref_logits = (c["x"].astype(np.float64) @ c["wr"].astype(np.float64).T)
    assert np.allclose(logits, ref_logits, rtol=1e-6, atol=1e-6)
    ref_idx = _topk_numpy(ref_logits.astype(np.float32), k)
    assert np.array_equal(np.sort(idx, 1), np.sort(ref_idx, 1)), "top-k sets"
    assert np.array_equal(idx, ref_idx), "top-k order (descending logit)"
    p = scipy.special.softmax(ref_logits.astype(np.float32).astype(np.float64), axis=1)
    psel = np.take_along_axis(p, ref_idx, 1)
    assert np.allclose(w, psel / psel.sum(1, keepdims=True), rtol=1e-9, atol=1e-12)
    assert np.array_equal(counts, np.bincount(ref_idx.ravel(), minlength=24))


def pin_full_softmax_when_k_equals_E(mutation=0):
    """k = E: the weights are the plain softmax over all logits (scipy)."""
    c = _rng_case(12, 16, 24, 4, 12, n_shared=0)
    idx, w, logits, _ = oracle.route(c["x"], c["wr"], 12, nthreads=1, mutation=mutation)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(p, idx, 1), rtol=1e-12, atol=1e-15)
    assert np.array_equal(np.sort(idx, 1), np.tile(np.arange(12), (16, 1)))


def pin_weights_sum_and_ratio(mutation=0):
    """Invariants: sum_j w = 1; w_i / w_j = exp(l_i - l_j) (softmax ratio)."""
    c = _rng_case(13, 64, 32, 4, 32, n_shared=0)
    idx, w, logits, counts = oracle.route(c["x"], c["wr"], 8, nthreads=2, mutation=mutation)
    assert np.allclose(w.sum(1), 1.0, atol=1e-12)
    l = np.take_along_axis(logits.astype(np.float64), idx, 1)
    assert np.allclose(w[:, 1:] / w[:, :1], np.exp(l[:, 1:] - l[:, :1]), rtol=1e-10)
    assert counts.sum() == 64 * 8
    # every chosen logit beats every unchosen one
    mask = np.zeros_like(logits, dtype=bool)
    np.put_along_axis(mask, idx, True, 1)
    assert (np.where(mask, logits, np.inf).min(1) >= np.where(mask, -np.inf, logits).max(1)).all()


def pin_two_expert_logistic(mutation=0):
    """Closed form: E = 2, k = 2, d = 1 -> w = logistic(+-(a - b)), ordered by logit."""
    a, b = 0.75, -0.5
    x = np.array([[1.0]], np.float32)
    wr = np.array([[a], [b]], np.float32)
    idx, w, _, counts = oracle.route(x, wr, 2, nthreads=1, mutation=mutation)
    assert idx.tolist() == [[0, 1]]
    s = 1.0 / (1.0 + math.exp(-(a - b)))
    assert abs(w[0, 0] - s) < 1e-12 and abs(w[0, 1] - (1 - s)) < 1e-12
    assert counts.tolist() == [1, 1]


def pin_bf16_widening(mutation=0):
    """bf16 bit patterns are widened exactly: 0x3F80 = 1, 0x4000 = 2, 0xC040 = -3."""
    x = np.array([[0x3F80]], np.uint16)
    wr = np.array([[0x4000], [0xC040]], np.uint16)
    idx, w, logits, _ = oracle.route(x, wr, 1, nthreads=1, mutation=mutation)
    assert logits.tolist() == [[2.0, -3.0]] and idx.tolist() == [[0]] and w.tolist() == [[1.0]]


def pin_bias_enters_logits(mutation=0):
    """A router bias is added to the logits before selection."""
    c = _rng_case(14, 8, 16, 4, 8, n_shared=0)
    bias = np.linspace(-3, 3, 8).astype(np.float32)
    _, _, logits, _ = oracle.route(c["x"], c["wr"], 2, bias=bias, nthreads=1, mutation=mutation)
    ref = c["x"].astype(np.float64) @ c["wr"].astype(np.float64).T + bias
    assert np.allclose(logits, ref, rtol=1e-6, atol=1e-6)


def _torch_swiglu(x, wg, wu, wd):
    x, wg, wu, wd = (torch.from_numpy(np.asarray(a, np.float64)) for a in (x, wg, wu, wd))
    return (Fnn.silu(x @ wg.T) * (x @ wu.T)) @ wd.T


def pin_dense_swiglu(mutation=0):
    """E = 1, k = 1, no shared expert: the block is a dense SwiGLU MLP (torch float64)."""
    c = _rng_case(15, 12, 24, 20, 1, n_shared=0)
    out, idx, w, counts = oracle.forward(c["x"], c["wr"], c["wg"], c["wu"], c["wd"], 1,
                                         nthreads=2, mutation=mutation)
    ref = _torch_swiglu(c["x"], c["wg"][0], c["wu"][0], c["wd"][0]).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert (idx == 0).all() and (w == 1.0).all() and counts.tolist() == [12]


def pin_dense_plus_shared(mutation=0):
    """E = 1, k = 1 with the shared expert: out = E_0(x) + S(x) (torch float64)."""
    c = _rng_case(16, 10, 16, 12, 1, n_shared=1)
    out, *_ = oracle.forward(c["x"], c["wr"], c["wg"], c["wu"], c["wd"], 1, sg=c["sg"],
                             su=c["su"], sd=c["sd"], nthreads=2, mutation=mutation)
    ref = (_torch_swiglu(c["x"], c["wg"][0], c["wu"][0], c["wd"][0])
           + _torch_swiglu(c["x"], c["sg"], c["su"], c["sd"])).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def pin_all_experts_masked(mutation=0):
    """Brute force: evaluate every expert on every token, mask by numpy's top-k, weight by
    scipy's softmax renormalised over the chosen, add the shared expert."""
    E, k, T, d, F = 16, 4, 20, 32, 12
    c = _rng_case(17, T, d, F, E, n_shared=1)
    out, idx, w, counts = oracle.forward(c["x"], c["wr"], c["wg"], c["wu"], c["wd"], k,
                                         sg=c["sg"], su=c["su"], sd=c["sd"], nthreads=2,
                                         mutation=mutation)
    x64 = c["x"].astype(np.float64)
    logits = (x64 @ c["wr"].astype(np.float64).T).astype(np.float32)
    top = _topk_numpy(logits, k)
    mask = np.zeros((T, E))
    np.put_along_axis(mask, top, 1.0, 1)
    p = scipy.special.softmax(logits.astype(np.float64), axis=1) * mask
    p /= p.sum(1, keepdims=True)
    g = np.einsum("td,efd->tef", x64, c["wg"].astype(np.float64))
    u = np.einsum("td,efd->tef", x64, c["wu"].astype(np.float64))
    h = g * scipy.special.expit(g) * u
    y = np.einsum("tef,edf->ted", h, c["wd"].astype(np.float64))
    ref = np.einsum("te,ted->td", p, y) + _torch_swiglu(c["x"], c["sg"], c["su"], c["sd"]).numpy()
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)
    assert np.array_equal(counts, np.bincount(top.ravel(), minlength=E))


def pin_permutation_equivariance(mutation=0):
    """Tokens are independent: out(P x) == P out(x) bit for bit."""
    c = _rng_case(18, 24, 32, 8, 16, n_shared=1)
    perm = np.random.default_rng(5).permutation(24)
    args = (c["wr"], c["wg"], c["wu"], c["wd"], 4)
    kw = dict(sg=c["sg"], su=c["su"], sd=c["sd"], nthreads=3, mutation=mutation)
    out, idx, w, counts = oracle.forward(c["x"], *args, **kw)
    out_p, idx_p, w_p, counts_p = oracle.forward(c["x"][perm], *args, **kw)
    assert np.array_equal(out_p, out[perm]) and np.array_equal(idx_p, idx[perm])
    assert np.array_equal(w_p, w[perm]) and np.array_equal(counts_p, counts)


def pin_hand_cases(mutation=0):
    """Hand-derived tiny blocks with closed-form outputs (tests/golden/hand_cases.json)."""
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        a = {k: (None if v is None else np.array(v, np.float32)) for k, v in case["inputs"].items()}
        out, idx, w, counts = oracle.forward(a["x"], a["wr"], a["wg"], a["wu"], a["wd"],
                                             case["k"], sg=a.get("sg"), su=a.get("su"),
                                             sd=a.get("sd"), nthreads=1, mutation=mutation)
        exp = case["expected"]
        assert idx.tolist() == exp["idx"], case["name"]
        assert np.allclose(w, np.array(exp["w"]), rtol=0, atol=1e-12), case["name"]
        assert np.allclose(out, np.array(exp["out"]), rtol=0, atol=1e-12), case["name"]
        assert counts.tolist() == exp["counts"], case["name"]


# ---------------------------------------------------------------- 4-bit weights
# The 4-bit group-affine format of "Optimizing on-device inference for Apple
# Silicon", section "Dequantise weights within matrix multiplication": 4-bit
# codes, one bfloat16 scale and one bfloat16 bias per 64 weights along a row,
# w = scale * q + bias.  Reading of the pages (silent on the packing): two codes
# per byte along the row, the even column in the low nibble.

def _bf16(v: float) -> int:
    """bfloat16 bit pattern of a value exactly representable in bfloat16."""
    b = np.array([v], np.float32).view(np.uint32)[0]
    assert b & 0xFFFF == 0, v
    return int(b >> 16)


def _q4(rows, cols, code=0, scale=1.0, bias=0.0):
    """A rows x cols matrix with every code, scale and bias set to the given values."""
    codes = np.full((rows, cols // 2), (code & 15) | ((code & 15) << 4), np.uint8)
    sc = np.full((rows, cols // 64), _bf16(scale), np.uint16)
    bi = np.full((rows, cols // 64), _bf16(bias), np.uint16)
    return codes, sc, bi


def _q4_probe(wg, x, mutation):
    """E = 1, k = 1, no shared expert, up = all ones (code 0, bias 1), down =
    all ones: out[i] = sum_f silu(g_f) with g = Wg x, and silu(0) = 0, so a
    gate matrix with one non-zero row f0 gives out[i] = silu((Wg x)[f0])."""
    d, F = x.shape[1], wg[0].shape[0]
    wr = np.zeros((1, d), np.float32)
    wu = _q4(F, d, 0, 1.0, 1.0)
    wd = _q4(d, F, 0, 1.0, 1.0)
    out, *_ = oracle.forward(x, wr, [wg], [wu], [wd], 1, nthreads=1, mutation=mutation, q4=True,
                             F=F)
    return out


def _silu(z):
    return z / (1.0 + math.exp(-z))


def pin_q4_nibble_order(mutation=0):
    """One code byte 0x1F at column pair (2j, 2j + 1) of row 0, scale 1, bias 0:
    the even column holds 15 (low nibble), the odd column 1 (high nibble)."""
    d, F, j = 128, 64, 5
    codes, sc, bi = _q4(F, d, 0, 1.0, 0.0)
    codes[0, j] = 0x1F
    x = np.zeros((2, d), np.float32)
    x[0, 2 * j] = 1.0
    x[1, 2 * j + 1] = 1.0
    out = _q4_probe((codes, sc, bi), x, mutation)
    assert np.allclose(out[0], _silu(15.0), rtol=0, atol=1e-12)
    assert np.allclose(out[1], _silu(1.0), rtol=0, atol=1e-12)


def pin_q4_groups_scale_bias(mutation=0):
    """Row 0 with code 3 everywhere, scale 1 and bias 0.5 for columns 0..63,
    scale 2 and bias -1 for columns 64..127: w = 3 s + b = 3.5 then 5 (a swap of
    scale and bias, or a group of another size, gives other values)."""
    d, F = 128, 64
    codes, sc, bi = _q4(F, d, 0, 1.0, 0.0)
    codes[0, :] = 0x33
    sc[0, 0], bi[0, 0] = _bf16(1.0), _bf16(0.5)
    sc[0, 1], bi[0, 1] = _bf16(2.0), _bf16(-1.0)
    x = np.zeros((4, d), np.float32)
    for t, c in enumerate((0, 63, 64, 127)):
        x[t, c] = 1.0
    out = _q4_probe((codes, sc, bi), x, mutation)
    for t, w in enumerate((3.5, 3.5, 5.0, 5.0)):
        assert np.allclose(out[t], _silu(w), rtol=0, atol=1e-12), (t, out[t, 0])


def pin_q4_zero_codes_are_bias(mutation=0):
    """Every code 0: each weight is its group's bias.  A gate row of bias b and
    x = all ones gives g = d b for that row and 0 (bias 0) for the others; the
    all-ones up matrix gives u = d for every row, so out[i] = silu(d b) d."""
    d, F = 128, 64
    codes, sc, bi = _q4(F, d, 0, 4.0, 0.0)
    bi[0, :] = _bf16(0.25)
    x = np.ones((1, d), np.float32)
    out = _q4_probe((codes, sc, bi), x, mutation)
    assert np.allclose(out[0], _silu(d * 0.25) * d, rtol=1e-14, atol=0)


def pin_q4_matches_dense(mutation=0):
    """Q4 expert weights whose values are exact in bfloat16 (power-of-two scales,
    small biases) give the same block output as the same values stored dense."""
    r = np.random.default_rng(31)
    T, d, F, E, k = 6, 128, 64, 4, 2

    def rand_q4(rows, cols):
        codes = r.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
        sc = r.choice([_bf16(v) for v in (0.125, 0.25, 0.5)], (rows, cols // 64)).astype(np.uint16)
        bi = r.choice([_bf16(v) for v in (-1.0, -0.5, 0.0, 0.5)], (rows, cols // 64)).astype(
            np.uint16)
        lo = (codes & 15).astype(np.float64)
        hi = (codes >> 4).astype(np.float64)
        q = np.stack([lo, hi], axis=-1).reshape(rows, cols)

        def val(b):
            return np.array(b, np.uint32).__lshift__(16).view(np.float32).astype(np.float64)

        dense = q * np.repeat(val(sc), 64, axis=1) + np.repeat(val(bi), 64, axis=1)
        return (codes, sc, bi), dense.astype(np.float32)

    x = r.standard_normal((T, d)).astype(np.float32)
    wr = (r.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    q_g, q_u, q_d, d_g, d_u, d_d = [], [], [], [], [], []
    for _ in range(E):
        a, b = rand_q4(F, d)
        q_g.append(a), d_g.append(b)
        a, b = rand_q4(F, d)
        q_u.append(a), d_u.append(b)
        a, b = rand_q4(d, F)
        q_d.append(a), d_d.append(b)
    sq = [rand_q4(F, d), rand_q4(F, d), rand_q4(d, F)]
    out_q, idx_q, *_ = oracle.forward(x, wr, q_g, q_u, q_d, k, sg=sq[0][0], su=sq[1][0],
                                      sd=sq[2][0], nthreads=2, mutation=mutation, q4=True, F=F)
    out_d, idx_d, *_ = oracle.forward(x, wr, np.stack(d_g), np.stack(d_u), np.stack(d_d), k,
                                      sg=sq[0][1], su=sq[1][1], sd=sq[2][1], nthreads=2)
    assert np.array_equal(idx_q, idx_d)
    assert np.allclose(out_q, out_d, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- the quantiser
# oracle.quantize_q4 (the reading of the pages stated in its docstring) against
# what the format fixes: values already on a group's grid come back exactly,
# every value lands within half a step of its code, a constant group has
# scale 0.

def _grid_matrix(r, rows, cols):
    """Codes, scales and biases with power-of-two scales and small biases, each
    group using both code 0 and code 15, and the float32 values they encode."""
    q = r.integers(0, 16, (rows, cols)).astype(np.uint8)
    q[:, 0::64] = 0
    q[:, 1::64] = 15
    sc = r.choice([0.0078125, 0.015625, 0.03125, 0.0625], (rows, cols // 64)).astype(np.float32)
    bi = r.choice([-0.25, -0.125, -0.0625, 0.03125], (rows, cols // 64)).astype(np.float32)
    vals = q * np.repeat(sc, 64, axis=1) + np.repeat(bi, 64, axis=1)
    # explicit byte layout: column 2j in the low nibble of byte j
    codes = np.zeros((rows, cols // 2), np.uint8)
    for j in range(cols // 2):
        codes[:, j] = q[:, 2 * j] + 16 * q[:, 2 * j + 1]
    bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)  # exact: few mantissa bits
    return codes, bits(sc), bits(bi), vals.astype(np.float32)


def pin_quantize_recovers_grid(mutation=0):
    r = np.random.default_rng(41)
    codes, sc, bi, vals = _grid_matrix(r, 6, 256)
    c2, s2, b2 = oracle.quantize_q4(vals, mutation=mutation)
    assert np.array_equal(s2, sc) and np.array_equal(b2, bi)
    assert np.array_equal(c2, codes)
    # the same from bfloat16 input (the values are exact in bfloat16)
    c3, s3, b3 = oracle.quantize_q4(oracle._bf16_bits(vals), mutation=mutation)
    assert np.array_equal(c3, codes) and np.array_equal(s3, sc) and np.array_equal(b3, bi)


def pin_quantize_half_step_bound(mutation=0):
    """Random N(0, 1/2048) weights: |scale * q + bias - w| <= scale / 2 up to
    the bfloat16 rounding of scale and bias (2^-8 relative)."""
    r = np.random.default_rng(43)
    w = (r.standard_normal((64, 512)) / math.sqrt(2048)).astype(np.float32)
    c, sc, bi = oracle.quantize_q4(w, mutation=mutation)
    err = np.abs(oracle.dequantize_q4(c, sc, bi) - w).reshape(64, 8, 64).max(axis=2)
    s = oracle._bf16_value(sc).astype(np.float64)
    b = np.abs(oracle._bf16_value(bi).astype(np.float64))
    assert (err <= s / 2 + 2.0 ** -8 * (b + 15 * s)).all(), (err / s).max()


def pin_quantize_constant_group(mutation=0):
    w = np.full((2, 128), 0.3, np.float32)
    w[1, 64:] = -2.5
    c, sc, bi = oracle.quantize_q4(w, mutation=mutation)
    assert (sc == 0).all() and (c == 0).all()
    assert np.allclose(oracle._bf16_value(bi), [[0.30078125, 0.30078125], [0.30078125, -2.5]])


QUANT_PINS = [pin_quantize_recovers_grid, pin_quantize_half_step_bound,
              pin_quantize_constant_group]

ALL_PINS = [pin_route_vs_numpy, pin_full_softmax_when_k_equals_E, pin_weights_sum_and_ratio,
            pin_two_expert_logistic, pin_bf16_widening, pin_bias_enters_logits, pin_dense_swiglu,
            pin_dense_plus_shared, pin_all_experts_masked, pin_permutation_equivariance,
            pin_hand_cases, pin_q4_nibble_order, pin_q4_groups_scale_bias,
            pin_q4_zero_codes_are_bias, pin_q4_matches_dense]


# ---------------------------------------------------------------- Gated DeltaNet scan
def _gdn_case(seed, T, Hk, Hv, dk, dv, unit_keys=True, state=True):
    """Random float32 inputs of the scan (exact float64 values on both sides)."""
    r = np.random.default_rng(seed)
    k = r.standard_normal((T, Hk, dk)).astype(np.float32)
    if unit_keys:
        k /= np.linalg.norm(k, axis=2, keepdims=True)
    q = (r.standard_normal((T, Hk, dk)) / np.sqrt(dk)).astype(np.float32)
    v = r.standard_normal((T, Hv, dv)).astype(np.float32)
    alpha = r.uniform(0.6, 1.0, (T, Hv)).astype(np.float32)
    beta = r.uniform(0.05, 1.0, (T, Hv)).astype(np.float32)
    s0 = r.standard_normal((Hv, dv, dk)).astype(np.float32) if state else None
    return q, k, v, alpha, beta, s0


def pin_gdn_hand_case(mutation=0):
    """Two tokens worked by hand (tests/golden/gdn_hand.json)."""
    with open(os.path.join(GOLDEN, "gdn_hand.json")) as f:
        c = json.load(f)
    a = {kk: np.asarray(c[kk], np.float32) for kk in ("q", "k", "v", "alpha", "beta", "state_in")}
    o, s = oracle.gdn_scan(a["q"], a["k"], a["v"], a["alpha"], a["beta"], a["state_in"],
                           mutation=mutation)
    assert np.array_equal(o, np.asarray(c["o"])), o
    assert np.array_equal(s, np.asarray(c["state_out"])), s


def pin_gdn_delta_invariant(mutation=0):
    """The delta rule's defining property: after a token, the state recalls
    alpha r + beta (v - alpha r) |k|^2 at that token's key k, r being the recall
    before the token (for a unit key: (1 - beta) alpha r + beta v, the value
    written in); checked step by step through a scan (the state of each prefix
    continues into the next token)."""
    q, k, v, alpha, beta, s0 = _gdn_case(11, 6, 2, 4, 8, 8)
    s = s0.astype(np.float64)
    for t in range(6):
        heads = np.arange(4) // 2
        kt = k[t][heads].astype(np.float64)
        before = np.einsum("hji,hi->hj", s, kt)
        _, s = oracle.gdn_scan(q[t:t + 1], k[t:t + 1], v[t:t + 1], alpha[t:t + 1],
                               beta[t:t + 1], s, mutation=mutation)
        after = np.einsum("hji,hi->hj", s, kt)
        a, b = alpha[t][:, None].astype(np.float64), beta[t][:, None].astype(np.float64)
        kk = np.sum(kt * kt, axis=1)[:, None]
        want = a * before + b * (v[t].astype(np.float64) - a * before) * kk
        assert np.allclose(after, want, rtol=1e-12, atol=1e-12)


def pin_gdn_pure_decay(mutation=0):
    """beta = 0 leaves only the gate: S_T = (prod alpha) S_0 and
    o_t = (prod_{s<=t} alpha_s) S_0 q_t (closed form)."""
    q, k, v, alpha, beta, s0 = _gdn_case(12, 5, 1, 2, 4, 4)
    beta[:] = 0
    o, s = oracle.gdn_scan(q, k, v, alpha, beta, s0, mutation=mutation)
    g = np.cumprod(alpha.astype(np.float64), axis=0)  # [T][Hv]
    s64 = s0.astype(np.float64)
    want_o = g[:, :, None] * np.einsum("hji,ti->thj", s64, q[:, 0].astype(np.float64))
    assert np.allclose(o, want_o, rtol=1e-12, atol=1e-12)
    assert np.allclose(s, g[-1][:, None, None] * s64, rtol=1e-12, atol=1e-12)


def _gdn_parallel_form(q, k, v, alpha, beta, s0):
    """The same outputs from the scan's closed form, one value head at a time:
    S_t = G_t S_0 + sum_{i<=t} g_{t,i} u_i k_i^T with G_t = prod_{s<=t} alpha_s,
    g_{t,i} = prod_{i<s<=t} alpha_s, and the deltas u the solution of the unit
    lower-triangular system u_t + beta_t sum_{i<t} g_{t,i} (k_t . k_i) u_i =
    beta_t (v_t - G_t S_0 k_t) (scipy's triangular solve); o_t = S_t q_t."""
    import scipy.linalg
    T, Hk, dk = k.shape
    _, Hv, dv = v.shape
    o = np.zeros((T, Hv, dv))
    s_out = np.zeros((Hv, dv, dk))
    for h in range(Hv):
        kk = k[:, h // (Hv // Hk)].astype(np.float64)
        qq = q[:, h // (Hv // Hk)].astype(np.float64)
        la = np.cumsum(np.log(alpha[:, h].astype(np.float64)))
        G = np.exp(la)
        g = np.tril(np.exp(la[:, None] - la[None, :]))  # g[t, i], i <= t
        b = beta[:, h].astype(np.float64)
        S0 = s0[h].astype(np.float64)  # [dv][dk]
        L = b[:, None] * np.tril(g * (kk @ kk.T), -1)
        rhs = b[:, None] * (v[:, h].astype(np.float64) - G[:, None] * (kk @ S0.T))
        U = scipy.linalg.solve_triangular(np.eye(T) + L, rhs, lower=True, unit_diagonal=True)
        o[:, h] = G[:, None] * (qq @ S0.T) + (g * (qq @ kk.T)) @ U
        s_out[h] = G[-1] * S0 + (U * g[-1][:, None]).T @ kk
    return o, s_out


def pin_gdn_parallel_form(mutation=0):
    """Sequential scan == closed form through a triangular solve (another
    algorithm for the same recurrence), with grouped key heads."""
    for seed, (T, Hk, Hv, dk, dv) in ((13, (9, 2, 4, 8, 8)), (14, (7, 1, 3, 4, 6))):
        q, k, v, alpha, beta, s0 = _gdn_case(seed, T, Hk, Hv, dk, dv, unit_keys=seed == 13)
        o, s = oracle.gdn_scan(q, k, v, alpha, beta, s0, mutation=mutation)
        wo, ws = _gdn_parallel_form(q, k, v, alpha, beta, s0)
        assert np.allclose(o, wo, rtol=1e-9, atol=1e-9)
        assert np.allclose(s, ws, rtol=1e-9, atol=1e-9)


def pin_gdn_zero_state_default(mutation=0):
    """No initial state means a zero state: the first output is
    beta_1 (k_1 . q_1) v_1."""
    q, k, v, alpha, beta, _ = _gdn_case(15, 1, 1, 2, 4, 4, state=False)
    o, _ = oracle.gdn_scan(q, k, v, alpha, beta, None, mutation=mutation)
    want = beta[0][:, None] * float(k[0, 0] @ q[0, 0]) * v[0]
    assert np.allclose(o[0], want, rtol=1e-6, atol=1e-7)


GDN_PINS = [pin_gdn_hand_case, pin_gdn_delta_invariant, pin_gdn_pure_decay, pin_gdn_parallel_form,
            pin_gdn_zero_state_default]
