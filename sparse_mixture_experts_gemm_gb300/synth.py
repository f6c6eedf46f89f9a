"""Seeded synthetic inputs for the MoE block.

This module only draws random numbers.  It holds none of the block's arithmetic
(no routing, no projections), so both the CUDA path and the CPU oracle may take
their inputs from it.  Every tensor comes from one ``torch.Generator`` on the
device the tensor is made on, seeded once per call, in a fixed order:

    Wr, Sg, Su, Sd, Wg, Wu, Wd        (layer_weights, q4_layer_weights; a 4-bit
                                       matrix draws codes, scales, biases)
    x                                 (tokens)
    q, k, v, alpha, beta, state       (gdn_inputs, the Gated DeltaNet scan)

Distributions follow the workloads the block is measured on: activations
x ~ N(0, 1); every projection ~ N(0, 1/fan_in), fan_in = d for the router and
the gate/up projections, F for the down projections.  Values are drawn in the
storage type directly (bfloat16 or float32).

A torch generator on CUDA and one on the CPU give different streams for the same
seed; a caller that needs the same values on both sides draws once and copies.
"""
from __future__ import annotations

import math

import torch

_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


def _dt(dtype):
    return _DTYPES[dtype] if isinstance(dtype, str) else dtype


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, dtype, device):
    t = torch.empty(shape, dtype=dtype, device=device)
    t.normal_(0.0, std, generator=g)
    return t


def layer_weights(seed: int, d: int, F: int, E: int, n_shared: int = 1, dtype="bf16",
                  device="cpu") -> dict:
    """One layer's weights in the library's layouts.

    Wr [E][d]; Wg, Wu [E][F][d]; Wd [E][d][F]; Sg, Su [F][d]; Sd [d][F]
    (shared tensors are None when n_shared == 0).
    """
    dtype = _dt(dtype)
    g = _gen(seed, device)
    sd_in, sd_ff = 1.0 / math.sqrt(d), 1.0 / math.sqrt(F)
    w = {"Wr": _normal((E, d), sd_in, g, dtype, device)}
    if n_shared:
        w["Sg"] = _normal((F, d), sd_in, g, dtype, device)
        w["Su"] = _normal((F, d), sd_in, g, dtype, device)
        w["Sd"] = _normal((d, F), sd_ff, g, dtype, device)
    else:
        w["Sg"] = w["Su"] = w["Sd"] = None
    w["Wg"] = _normal((E, F, d), sd_in, g, dtype, device)
    w["Wu"] = _normal((E, F, d), sd_in, g, dtype, device)
    w["Wd"] = _normal((E, d, F), sd_ff, g, dtype, device)
    return w


def _q4_matrix(shape, std, g, device):
    """Random 4-bit group-affine matrix of logical shape [..., rows, cols]:
    codes uniform over 0..15 (two per byte), per 64-column group a bfloat16
    scale ~ std * U(0.27, 0.37) and bias ~ -std * U(2.0, 2.8), about the
    steps and minima that groups of 64 N(0, std^2) weights give."""
    *lead, rows, cols = shape
    codes = torch.randint(0, 256, (*lead, rows, cols // 2), dtype=torch.uint8, device=device,
                          generator=g)
    gs = (*lead, rows, cols // 64)
    sc = torch.empty(gs, dtype=torch.float32, device=device).uniform_(0.27 * std, 0.37 * std,
                                                                      generator=g)
    bi = torch.empty(gs, dtype=torch.float32, device=device).uniform_(-2.8 * std, -2.0 * std,
                                                                      generator=g)
    return (codes, sc.to(torch.bfloat16).view(torch.int16),
            bi.to(torch.bfloat16).view(torch.int16))


def q4_layer_weights(seed: int, d: int, F: int, E: int, n_shared: int = 1,
                     device="cpu") -> dict:
    """One layer with 4-bit expert weights: Wr [E][d] bfloat16 as in
    layer_weights, and Wg, Wu, Wd, Sg, Su, Sd as (codes uint8, scales int16,
    biases int16) triples, bfloat16 bits in the int16 tensors, in the layouts
    of the bf16 matrices (codes [.., rows][cols / 2], scales and biases
    [.., rows][cols / 64])."""
    g = _gen(seed, device)
    sd_in, sd_ff = 1.0 / math.sqrt(d), 1.0 / math.sqrt(F)
    w = {"Wr": _normal((E, d), sd_in, g, torch.bfloat16, device)}
    if n_shared:
        w["Sg"] = _q4_matrix((F, d), sd_in, g, device)
        w["Su"] = _q4_matrix((F, d), sd_in, g, device)
        w["Sd"] = _q4_matrix((d, F), sd_ff, g, device)
    else:
        w["Sg"] = w["Su"] = w["Sd"] = None
    w["Wg"] = _q4_matrix((E, F, d), sd_in, g, device)
    w["Wu"] = _q4_matrix((E, F, d), sd_in, g, device)
    w["Wd"] = _q4_matrix((E, d, F), sd_ff, g, device)
    return w


def tokens(seed: int, T: int, d: int, dtype="bf16", device="cpu") -> torch.Tensor:
    """x ~ N(0, 1), [T][d]."""
    return _normal((T, d), 1.0, _gen(seed, device), _dt(dtype), device)


def fresh_rows(seed: int, attempt: int, n: int, d: int, dtype="bf16", device="cpu") -> torch.Tensor:
    """n fresh N(0, 1) rows for re-drawing tokens; a distinct stream per (seed, attempt)."""
    return _normal((n, d), 1.0, _gen(seed * 1000003 + 7919 * (attempt + 1), device), _dt(dtype),
                   device)


def zipf_bias(seed: int, E: int, s: float = 1.2) -> torch.Tensor:
    """Skewed-routing router bias, float32 [E] (CPU).

    A seeded random permutation pi of the experts ranks them; the expert of rank
    r (1-based) gets the bias -s * ln(r), the logarithm of a Zipf(s) weight up to
    a constant, so a few experts draw thousands of tokens and many draw none.
    """
    g = _gen(seed, "cpu")
    perm = torch.randperm(E, generator=g)
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    b = torch.empty(E, dtype=torch.float64)
    b[perm] = -s * torch.log(ranks)
    return b.to(torch.float32)


def gdn_inputs(seed: int, T: int, Hk: int, Hv: int, dk: int, dv: int, device="cpu",
               state: bool = False) -> dict:
    """Inputs of a Gated DeltaNet scan, drawn in the order q, k, v, alpha, beta,
    state: q and k per head ~ N(0, 1) rescaled to unit length (the model
    normalises them before the scan), q further by 1/sqrt(d_k) (its query
    scale), stored bf16; v ~ N(0, 1) bf16; the gate alpha = exp(-softplus(z)),
    z ~ N(-2.5, 1) (mostly 0.8..1, a long tail toward forgetting) and the write
    strength beta = sigmoid(N(0, 1)), both float32 [T][H_v]; the initial state
    (if asked for) ~ N(0, 0.1^2) float32 [H_v][d_v][d_k], else None."""
    g = _gen(seed, device)
    f32 = torch.float32

    def unit(shape):
        t = torch.randn(shape, generator=g, device=device, dtype=f32)
        return t / t.norm(dim=-1, keepdim=True)

    q = (unit((T, Hk, dk)) / math.sqrt(dk)).to(torch.bfloat16)
    k = unit((T, Hk, dk)).to(torch.bfloat16)
    v = torch.randn((T, Hv, dv), generator=g, device=device, dtype=f32).to(torch.bfloat16)
    z = torch.randn((T, Hv), generator=g, device=device, dtype=f32) - 2.5
    alpha = torch.exp(-torch.nn.functional.softplus(z))
    beta = torch.sigmoid(torch.randn((T, Hv), generator=g, device=device, dtype=f32))
    s0 = (torch.randn((Hv, dv, dk), generator=g, device=device, dtype=f32) * 0.1) if state else None
    return {"q": q, "k": k, "v": v, "alpha": alpha, "beta": beta, "state": s0}

