"""Shared test helpers: seeded inputs with a routing margin, oracle calls on
torch tensors, and the comparison metrics used by the parity tests.

Routing margin: the parity bar is exact expert indices, so inputs are drawn
such that, for every token, the k-th largest router logit exceeds the
(k+1)-th by at least MARGIN (computed by the oracle's router on the stored
inputs).  Tokens below the margin are re-drawn from a fresh seeded stream.
MARGIN = 1e-3 is far above the fp32 summation-order error of a 2048-term dot
product of bf16 values (about 1e-6), so both sides must pick the same set.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_mixture_experts_gemm_gb300 import synth

MARGIN = 1e-3
OUT_TOL = 1e-2      # row-normwise relative error of the block output
W_TOL = 1e-5        # absolute error of the routing weights


def np_view(t: torch.Tensor) -> np.ndarray:
    """Host numpy view for the oracle: bf16 -> uint16 bit patterns, f32 as is."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


def kth_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Per-token gap between the k-th and (k+1)-th largest logit."""
    if logits.shape[1] <= k:
        return np.full(logits.shape[0], np.inf)
    part = -np.sort(-logits.astype(np.float64), axis=1)
    return part[:, k - 1] - part[:, k]


def margined_tokens(seed: int, T: int, wr: torch.Tensor, k: int, dtype, bias=None,
                    device="cpu", max_rounds: int = 50) -> torch.Tensor:
    """x [T][d] ~ N(0, 1) with every token's top-k/top-(k+1) logit gap >= MARGIN."""
    d = wr.shape[1]
    x = synth.tokens(seed, T, d, dtype, device)
    wr_np = np_view(wr)
    b_np = None if bias is None else bias.detach().cpu().numpy().astype(np.float32)
    bad = np.arange(T)
    for attempt in range(max_rounds):
        xs = x[torch.as_tensor(bad, device=x.device)] if len(bad) < T else x
        _, _, logits, _ = oracle.route(np_view(xs), wr_np, k, bias=b_np)
        sel = kth_gap(logits, k) < MARGIN
        bad = bad[sel]
        if len(bad) == 0:
            return x
        fresh = synth.fresh_rows(seed, attempt, len(bad), d, dtype, device)
        x[torch.as_tensor(bad, device=x.device)] = fresh
    raise RuntimeError("could not draw tokens with the routing margin")


def oracle_forward(x: torch.Tensor, w: dict, k: int, bias=None, rows=None):
    """Oracle on (a subset of) tokens; weights passed as bf16 bits / f32 arrays."""
    xs = x if rows is None else x[torch.as_tensor(rows, device=x.device)]
    E = w["Wr"].shape[0]

    def per_expert(name):
        t = np_view(w[name])
        return [t[e] for e in range(E)]

    sh = w.get("Sg") is not None
    return oracle.forward(np_view(xs), np_view(w["Wr"]), per_expert("Wg"), per_expert("Wu"),
                          per_expert("Wd"), k,
                          sg=np_view(w["Sg"]) if sh else None, su=np_view(w["Su"]) if sh else None,
                          sd=np_view(w["Sd"]) if sh else None,
                          bias=None if bias is None else bias.detach().cpu().numpy())


def row_rel_err(got: torch.Tensor, ref: np.ndarray) -> np.ndarray:
    """max_i |got - ref| / max_i |ref| per row."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    den = np.abs(ref).max(1)
    den = np.where(den == 0, 1.0, den)
    return np.abs(g - ref).max(1) / den


def check_routing(idx_gpu, w_gpu, counts_gpu, idx_ref, w_ref, counts_ref, rows=None):
    """Exact index sets and counts; weights within W_TOL matched by expert id."""
    ig = idx_gpu.detach().cpu().numpy()
    wg = w_gpu.detach().cpu().numpy().astype(np.float64)
    if rows is not None:
        ig, wg = ig[rows], wg[rows]
    og = np.argsort(ig, axis=1, kind="stable")
    orf = np.argsort(idx_ref, axis=1, kind="stable")
    ig_s = np.take_along_axis(ig, og, 1)
    ir_s = np.take_along_axis(idx_ref, orf, 1)
    bad = np.nonzero((ig_s != ir_s).any(1))[0]
    assert len(bad) == 0, f"{len(bad)} tokens routed differently, first {bad[:5]}"
    dw = np.abs(np.take_along_axis(wg, og, 1) - np.take_along_axis(w_ref, orf, 1)).max()
    assert dw <= W_TOL, f"routing weight error {dw:.3e}"
    if counts_gpu is not None:
        cg = counts_gpu.detach().cpu().numpy()
        assert np.array_equal(cg, counts_ref), "per-expert counts differ"
    # the order contract: descending weight
    assert (np.diff(wg, axis=1) <= 1e-7).all(), "weights not in descending order"
