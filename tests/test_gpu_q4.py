"""4-bit group-affine expert weights on the GPU, through the C ABI.

* moe_quantize_q4 against oracle.quantize_q4 on the same values: codes, scales
  and biases bit for bit (both sides take every decision in float32).
* The batch-1 path of a 4-bit handle (moe_create_q4, moe_forward with T == 1)
  against the oracle's 4-bit forward on the same codes, scales and biases,
  drawn by the seeded generator: block output within 1e-2 row-normwise
  relative error, as for the bf16 path.
"""
import numpy as np
import pytest
import torch

import helpers as H
import oracle
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


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("dtype,shape", [
    ("bf16", (8, 64)),
    ("bf16", (256, 2048)),
    ("bf16", (3, 512, 2048)),      # a stack of expert matrices
    ("f32", (100, 4096)),
    ("f32", (17, 192)),
])
def test_quantizer_matches_oracle(dev, dtype, shape):
    g = torch.Generator(device=dev)
    g.manual_seed(hash(shape) % 1000)
    w = torch.empty(shape, dtype=synth._dt(dtype), device=dev).normal_(0, 0.02, generator=g)
    # a few constant groups and one group with a single outlier
    flat = w.view(-1, shape[-1])
    flat[0, :64] = 0.375
    if flat.shape[0] > 2:
        flat[2, :64] = 0.0
        flat[2, 7] = 1.0
    codes, scales, biases = moe.quantize_q4(w)
    torch.cuda.synchronize()
    host = H.np_view(flat)
    rc, rs, rb = oracle.quantize_q4(host)
    assert np.array_equal(codes.view(-1, shape[-1] // 2).cpu().numpy(), rc)
    assert np.array_equal(_bits(scales.view(-1, shape[-1] // 64)), rs)
    assert np.array_equal(_bits(biases.view(-1, shape[-1] // 64)), rb)


def _oracle_q4(x, w, k, F, rows=None):
    """The oracle's 4-bit forward on the same codes, scales and biases (on the
    given token rows only, when rows is set)."""
    E = w["Wr"].shape[0]
    if rows is not None:
        x = x[torch.as_tensor(rows, device=x.device)]

    def triple(t):
        return None if t is None else (t[0].cpu().numpy(), _bits(t[1]), _bits(t[2]))

    per = {n: triple(w[n]) for n in ("Wg", "Wu", "Wd")}
    experts = {n: [(c[e], s[e], b[e]) for e in range(E)] for n, (c, s, b) in per.items()}
    return oracle.forward(H.np_view(x), H.np_view(w["Wr"]), experts["Wg"], experts["Wu"],
                          experts["Wd"], k, sg=triple(w.get("Sg")), su=triple(w.get("Su")),
                          sd=triple(w.get("Sd")), q4=True, F=F)


# (d, F, E, k, n_shared)
CASES = [
    (2048, 512, 256, 8, 1),     # the full-size decode layer
    (2048, 512, 256, 8, 0),     # no shared expert
    (256, 128, 8, 2, 1),        # few experts, short rows
    (1024, 256, 64, 8, 1),
    (8192, 256, 16, 4, 1),      # four 64-column groups per lane
    (16384, 128, 8, 2, 1),      # the longest rows: eight groups per lane
    (2048, 4096, 8, 1, 1),      # the widest down rows: 128 (slot, group) pairs
]


@pytest.mark.parametrize("d,F,E,k,n_shared", CASES)
def test_q4_decode_matches_oracle(dev, d, F, E, k, n_shared):
    w = synth.q4_layer_weights(150 + d + E, d, F, E, n_shared, dev)
    n_tok = 4
    x = H.margined_tokens(160 + d, n_tok, w["Wr"], k, "bf16", device=dev)
    layer = moe.Q4Layer(w, k)
    try:
        moe.moe_profile(layer.handle, True)
        layer.forward(x[0:1].clone())
        moe.moe_profile(layer.handle, False)
        prof = moe.moe_profile_read(layer.handle)
        kinds = {name for name, (_, n) in prof.items() if n > 0}
        assert kinds == {"decode_router", "decode_gate_up", "decode_down"}, kinds
        outs = [layer.forward(x[i:i + 1].clone()) for i in range(n_tok)]
        torch.cuda.synchronize()
        rc, detail = layer.status()
        assert rc == 0, f"device status {rc} detail {detail}"
    finally:
        layer.close()
    out = torch.cat(outs)
    ref, *_ = _oracle_q4(x, w, k, F)
    err = H.row_rel_err(out, ref)
    assert err.max() <= H.OUT_TOL, err


def test_q4_handle_routes_and_checks_batches(dev):
    d, F, E, k = 2048, 512, 256, 8
    w = synth.q4_layer_weights(7, d, F, E, 1, dev)
    x = H.margined_tokens(8, 2, w["Wr"], k, "bf16", device=dev)
    layer = moe.Q4Layer(w, k)
    try:
        idx, wt, counts = layer.route(x[0:1].clone())
        torch.cuda.synchronize()
        ri, rw, _, rc = oracle.route(H.np_view(x[0:1]), H.np_view(w["Wr"]), k)
        H.check_routing(idx, wt, counts, ri, rw, rc)
        # a batch on a handle made for one token at a time runs as chunks of
        # one token through the grouped GEMMs
        out = torch.empty((2, d), dtype=torch.bfloat16, device=dev)
        moe.moe_forward(layer.handle, x, 2, out)
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
        ref, *_ = _oracle_q4(x, w, k, F)
        assert H.row_rel_err(out, ref).max() <= H.OUT_TOL
    finally:
        layer.close()


def _diff_report(a, b):
    """Where two bf16 tensors differ bit-wise: count, first indices, NaNs,
    largest difference."""
    ne = a.view(torch.int16) != b.view(torch.int16)
    idx = ne.nonzero()[:8].tolist()
    diff = (a.float() - b.float()).abs().nan_to_num(0.0)
    return (f"{int(ne.sum())} differing of {a.numel()} at {idx}, NaN {int(a.isnan().sum())}"
            f"/{int(b.isnan().sum())}, max |diff| {diff.max().item():.4g}, "
            f"max |a| {a.float().abs().nan_to_num(0.0).max().item():.4g}")


def test_q4_layer_stack_in_a_cuda_graph(dev):
    """Four chained 4-bit layers captured once; replays equal eager runs bit for
    bit."""
    d, F, E, k, L = 2048, 512, 256, 8, 4
    ws = [synth.q4_layer_weights(170 + l, d, F, E, 1, dev) for l in range(L)]
    layers = [moe.Q4Layer(w, k) for w in ws]
    try:
        xin = torch.empty((1, d), dtype=torch.bfloat16, device=dev)
        outs = [torch.empty((1, d), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            for l in range(L):
                layers[l].forward(xin if l == 0 else outs[l - 1], out=outs[l], stream=stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                layers[l].forward(xin if l == 0 else outs[l - 1], out=outs[l], stream=stream)
        toks = synth.tokens(180, 3, d, "bf16", dev)
        for step in range(3):
            xin.copy_(toks[step:step + 1])
            g.replay()
            torch.cuda.synchronize()
            got = [o.clone() for o in outs]
            h = toks[step:step + 1].clone()
            for l in range(L):
                h = layers[l].forward(h)
                torch.cuda.synchronize()
                assert torch.equal(got[l].view(torch.int16), h.view(torch.int16)), (
                    f"step {step} layer {l}: {_diff_report(got[l], h)}; "
                    f"status {[lay.status() for lay in layers]}")
        for layer in layers:
            assert layer.status()[0] == 0
    finally:
        for layer in layers:
            layer.close()


def test_q4_batches_need_d_and_f_multiples_of_512(dev):
    """The grouped GEMMs read scale/bias rows of 16-byte pitch: a layer with
    F = 256 runs batches only where every chunk takes the small-batch kernels
    (at most 32 tokens) and refuses larger ones; 2 and 20 tokens run (two and
    four column blocks of the grouped GEMV) and match the oracle, and so do 40
    tokens through a handle with 16-token chunks (16 + 16 + 8)."""
    w = synth.q4_layer_weights(9, 1024, 256, 16, 1, dev)
    x = H.margined_tokens(10, 40, w["Wr"], 4, "bf16", device=dev)
    layer = moe.Q4Layer(w, 4, max_tokens=64)
    try:
        out = torch.empty((40, 1024), dtype=torch.bfloat16, device=dev)
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward(layer.handle, x, 40, out)
        assert e.value.code == moe.MOE_ERR_UNSUPPORTED
        got2 = layer.forward(x[:2].clone())
        got20 = layer.forward(x[:20].clone())
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
    finally:
        layer.close()
    chunked = moe.Q4Layer(w, 4, max_tokens=16)
    try:
        got40 = chunked.forward(x)
        torch.cuda.synchronize()
        assert chunked.status()[0] == 0
    finally:
        chunked.close()
    ref, *_ = _oracle_q4(x, w, 4, 256)
    assert H.row_rel_err(got2, ref[:2]).max() <= H.OUT_TOL
    assert H.row_rel_err(got20, ref[:20]).max() <= H.OUT_TOL
    assert H.row_rel_err(got40, ref).max() <= H.OUT_TOL


# (d, F, E, k, n_shared, T, max_tokens)
PREFILL_CASES = [
    (512, 512, 8, 2, 1, 300, 512),       # ragged tiles, few experts
    (1024, 512, 16, 4, 0, 130, 256),     # no shared expert
    (2048, 1024, 32, 8, 1, 520, 1024),   # wider F: 8 gate/up N tiles
    (2048, 512, 256, 8, 1, 384, 192),    # the full-size layer, in two chunks
]


@pytest.mark.parametrize("d,F,E,k,n_shared,T,max_tokens", PREFILL_CASES)
def test_q4_prefill_matches_oracle(dev, d, F, E, k, n_shared, T, max_tokens):
    """Batches through the 4-bit grouped GEMMs (dequantisation in the GEMM,
    the weights rounded once to bf16) against the oracle's exact 4-bit
    forward; row-normwise 1e-2 as for the bf16 path."""
    w = synth.q4_layer_weights(200 + d + E + T, d, F, E, n_shared, dev)
    x = H.margined_tokens(210 + T, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.Q4Layer(w, k, max_tokens=max_tokens)
    try:
        moe.moe_profile(layer.handle, True)
        out = layer.forward(x)
        moe.moe_profile(layer.handle, False)
        torch.cuda.synchronize()
        rc, detail = layer.status()
        assert rc == 0, f"device status {rc} detail {detail}"
        kinds = {name for name, (_, n) in moe.moe_profile_read(layer.handle).items() if n > 0}
        assert {"gemm_gate_up", "gemm_down"} <= kinds, kinds
    finally:
        layer.close()
    ref, *_ = _oracle_q4(x, w, k, F)
    err = H.row_rel_err(out, ref)
    assert err.max() <= H.OUT_TOL, err.max()


def test_q4_prefill_4k_sample_against_oracle(dev):
    """The 4096-token prefill of the full-size layer through the 4-bit GEMMs;
    64 sampled tokens against the oracle (token rows are independent)."""
    d, F, E, k, T = 2048, 512, 256, 8, 4096
    w = synth.q4_layer_weights(300, d, F, E, 1, dev)
    x = synth.tokens(301, T, d, "bf16", dev)
    layer = moe.Q4Layer(w, k, max_tokens=T)
    try:
        out = layer.forward(x)
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
    finally:
        layer.close()
    rows = np.random.default_rng(5).choice(T, 64, replace=False)
    _, _, logits, _ = oracle.route(H.np_view(x[torch.as_tensor(rows, device=dev)]),
                                   H.np_view(w["Wr"]), k)
    keep = rows[H.kth_gap(logits, k) >= H.MARGIN]
    assert len(keep) >= 48
    ref, *_ = _oracle_q4(x, w, k, F, rows=keep)
    err = H.row_rel_err(out[torch.as_tensor(keep, device=dev)], ref)
    assert err.max() <= H.OUT_TOL, err.max()


@pytest.mark.parametrize("T", [2, 7, 16, 17, 32, 33, 64])
def test_q4_small_batch_path(dev, T):
    """Batches of at most 32 tokens on 4-bit weights take the small-batch
    kernels (one routing launch, the 4-bit grouped GEMV, the combine), and up
    to 64 the same routing launch before the grouped GEMMs: the full-size
    layer against the oracle, every output, and the kernel kinds."""
    d, F, E, k = 2048, 512, 256, 8
    w = synth.q4_layer_weights(60 + T, d, F, E, 1, dev)
    x = H.margined_tokens(70 + T, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.Q4Layer(w, k, max_tokens=64)
    try:
        moe.moe_profile(layer.handle, True)
        got = layer.forward(x)
        moe.moe_profile(layer.handle, False)
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
        kinds = {name for name, (_, n) in moe.moe_profile_read(layer.handle).items() if n > 0}
        want = ({"router", "gemv_gate_up", "gemv_down", "combine"} if T <= 32
                else {"router", "gemm_gate_up", "gemm_down", "combine"})
        assert kinds == want, kinds
    finally:
        layer.close()
    ref, *_ = _oracle_q4(x, w, k, F)
    assert H.row_rel_err(got, ref).max() <= H.OUT_TOL


def test_q4_small_batch_crowded_experts(dev):
    """4-bit small batch with routed groups of more than 8 tokens and F = 128
    (one 128-column super-step in the down projection)."""
    d, F, E, k, T = 256, 128, 4, 2, 16
    w = synth.q4_layer_weights(80, d, F, E, 1, dev)
    x = H.margined_tokens(81, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.Q4Layer(w, k, max_tokens=16)
    try:
        got = layer.forward(x)
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
    finally:
        layer.close()
    ref, *_ = _oracle_q4(x, w, k, F)
    assert H.row_rel_err(got, ref).max() <= H.OUT_TOL



def test_q4_small_batch_without_shared_expert(dev):
    """4-bit small batch with no shared expert and 40 experts (a partial router CTA)."""
    d, F, E, k, T = 512, 256, 40, 4, 9
    w = synth.q4_layer_weights(82, d, F, E, 0, dev)
    x = H.margined_tokens(83, T, w["Wr"], k, "bf16", device=dev)
    layer = moe.Q4Layer(w, k, max_tokens=16)
    try:
        got = layer.forward(x)
        torch.cuda.synchronize()
        assert layer.status()[0] == 0
    finally:
        layer.close()
    ref, *_ = _oracle_q4(x, w, k, F)
    assert H.row_rel_err(got, ref).max() <= H.OUT_TOL
