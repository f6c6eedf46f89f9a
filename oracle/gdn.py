"""CPU oracle of the Gated DeltaNet recurrent scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this module; the product library never loads it.

"Optimizing on-device inference for Apple Silicon", section "Qwen creates
three distinct workload shapes": a Gated DeltaNet layer compresses the past
into a recurrent state of fixed size; a learned gate decides how much of the
existing state is kept, and a delta update writes in what the current token
carries; each token depends on the state the previous one left.  Section "Keep
the recurrent state on chip": the state is a matrix, kept in 32-bit float with
its gate, while the query and key (and value) activations stay bfloat16.

The pages name the update but do not print it; the reading taken is the
published gated delta rule (Yang, Kautz and Hatamizadeh, "Gated Delta Networks:
Improving Mamba2 with Delta Rule").  With the state S of a value head stored
as columns -- S[j] is the d_k-vector of value coordinate j -- one token t does

    r_j   = S[j] . k_t                      (what the state recalls at key k_t)
    u_j   = beta_t * (v_t[j] - alpha_t * r_j)   (the delta: new value minus the decayed recall)
    S[j] <- alpha_t * S[j] + u_j * k_t      (decay, then write u at key k_t)
    o_t[j] = S[j] . q_t                     (read with the query, after the write)

i.e. S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T in matrix
form.  alpha_t (the gate, in (0, 1]) and beta_t (the write strength) are per
token and value head; value head h reads key head h // (H_v / H_k).  Every
step is evaluated in float64 from the exact input values, token after token,
in the order above.  Layouts: q, k [T][H_k][d_k]; v, o [T][H_v][d_v]; alpha,
beta [T][H_v]; state [H_v][d_v][d_k] (column j of head h contiguous).

mutation plants a mistake for the pin tests: 1 drops alpha from the recall in
the delta, 2 skips the decay of the state, 3 reads the output before the
write, 4 maps value head h to key head h % H_k, 5 recalls with the state
transposed, 6 scales only v by beta (u = beta v - alpha r).
"""
from __future__ import annotations

import numpy as np


def _values(a) -> np.ndarray:
    """float64 values of bf16 bit patterns (uint16) or of a float array."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def gdn_scan(q, k, v, alpha, beta, state=None, mutation: int = 0):
    """Returns (o [T][H_v][d_v], final state [H_v][d_v][d_k]), both float64."""
    q, k, v = _values(q), _values(k), _values(v)
    alpha = np.asarray(alpha, np.float64)
    beta = np.asarray(beta, np.float64)
    T, Hk, dk = k.shape
    _, Hv, dv = v.shape
    assert q.shape == k.shape and alpha.shape == (T, Hv) and beta.shape == (T, Hv)
    assert Hv % Hk == 0
    heads = np.arange(Hv) % Hk if mutation == 4 else np.arange(Hv) // (Hv // Hk)
    S = np.zeros((Hv, dv, dk)) if state is None else _values(state).copy()
    assert S.shape == (Hv, dv, dk)
    o = np.zeros((T, Hv, dv))
    for t in range(T):
        kt, qt = k[t][heads], q[t][heads]  # [Hv][dk]
        a, b = alpha[t][:, None], beta[t][:, None]
        if mutation == 5:
            r = np.einsum("hij,hi->hj", S, kt)  # (meaningful only when dk == dv)
        else:
            r = np.einsum("hji,hi->hj", S, kt)
        if mutation == 1:
            u = b * (v[t] - r)
        elif mutation == 6:
            u = b * v[t] - a * r
        else:
            u = b * (v[t] - a * r)
        if mutation == 3:
            o[t] = np.einsum("hji,hi->hj", S, qt)
        S = (S if mutation == 2 else a[:, :, None] * S) + u[:, :, None] * kt[:, None, :]
        if mutation != 3:
            o[t] = np.einsum("hji,hi->hj", S, qt)
    return o, S
