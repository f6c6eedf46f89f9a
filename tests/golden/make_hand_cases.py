"""Writes hand_cases.json: tiny MoE blocks whose outputs have closed forms.

The expected values are evaluated here from the closed forms stated in each
case's "derivation" (logistic sigma(z) = 1 / (1 + e^-z), silu(z) = z sigma(z));
nothing here calls the oracle or the CUDA library.  The block is the one of
"Optimizing on-device inference for Apple Silicon", section "Qwen creates three
distinct workload shapes" (router picks k experts, plus a shared expert) and
section "Reduce intermediate traffic and dispatch traffic" (gated input
projections; output projection scaled by the routing score; shared result
added).  Run: python tests/golden/make_hand_cases.py
"""
import json
import math
import os


def sig(z):
    return 1.0 / (1.0 + math.exp(-z))


cases = []

# 1: one-hot router, top-1, no shared expert.
h = 2.0 * sig(2.0)  # silu(2) * u, u = 1
cases.append({
    "name": "one_hot_top1",
    "k": 1,
    "derivation": "logits = x Wr^T = [1, 2] -> expert 1, w = 1; g = 2, u = 1, h = silu(2) = 2 sigma(2);"
                  " y = Wd_1 h = [h, -2h]",
    "inputs": {"x": [[1, 2]], "wr": [[1, 0], [0, 1]],
               "wg": [[[1, 0]], [[0, 1]]], "wu": [[[1, 1]], [[1, 0]]],
               "wd": [[[1], [1]], [[1], [-2]]], "sg": None, "su": None, "sd": None},
    "expected": {"idx": [[1]], "w": [[1.0]], "out": [[h, -2.0 * h]], "counts": [0, 1]},
})

# 2: two experts, both chosen, plus the shared expert.
w0, w1 = sig(1.0), 1.0 - sig(1.0)
out2 = w0 * sig(1.0) + w1 * 2.0 * sig(2.0) + 6.0 * sig(1.0)
cases.append({
    "name": "two_experts_with_shared",
    "k": 2,
    "derivation": "logits [0.5, -0.5] -> w = [sigma(1), 1 - sigma(1)]; expert 0: g = 1, u = 1 ->"
                  " h = sigma(1); expert 1: g = 2, u = 1 -> h = 2 sigma(2); Wd = 1; shared: g = 1,"
                  " u = 3, Sd = 2 -> 6 sigma(1); out = w0 sigma(1) + w1 2 sigma(2) + 6 sigma(1)",
    "inputs": {"x": [[1]], "wr": [[0.5], [-0.5]], "wg": [[[1]], [[2]]], "wu": [[[1]], [[1]]],
               "wd": [[[1]], [[1]]], "sg": [[1]], "su": [[3]], "sd": [[2]]},
    "expected": {"idx": [[0, 1]], "w": [[w0, w1]], "out": [[out2]], "counts": [1, 1]},
})

# 3: tied top logits; the lower expert index comes first.
cases.append({
    "name": "tie_goes_to_lower_index",
    "k": 2,
    "derivation": "logits [1, 1, 0] -> experts [0, 1] (tie to lower index), w = [1/2, 1/2];"
                  " h0 = 2 silu(1) = 2 sigma(1), h1 = 2 silu(-1) = -2 sigma(-1);"
                  " out = sigma(1) - sigma(-1) = tanh(1/2)",
    "inputs": {"x": [[1]], "wr": [[1], [1], [0]], "wg": [[[1]], [[-1]], [[5]]],
               "wu": [[[2]], [[2]], [[2]]], "wd": [[[1]], [[1]], [[1]]],
               "sg": None, "su": None, "sd": None},
    "expected": {"idx": [[0, 1]], "w": [[0.5, 0.5]], "out": [[math.tanh(0.5)]],
                 "counts": [1, 1, 0]},
})

here = os.path.dirname(os.path.abspath(__file__))
with open(os.path.join(here, "hand_cases.json"), "w") as f:
    f.write('{"source": "closed forms, see tests/golden/make_hand_cases.py",\n "cases": [\n')
    f.write(",\n".join("  " + json.dumps(c) for c in cases))
    f.write("\n ]}\n")
