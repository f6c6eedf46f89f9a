"""CPU oracle of the sparse MoE feed-forward block -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it (see ``moe_oracle.c`` for the definition it evaluates and
the passages of "Optimizing on-device inference for Apple Silicon" it follows).

Arrays are numpy: bfloat16 data is passed as its uint16 bit patterns
(``dtype=0``), float32 as float32 (``dtype=1``).  All results come back in
float64 except the router logits (float32, the precision in which the top-k
decision is taken).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}


class Dims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("F", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("n_shared", ctypes.c_int), ("dtype", ctypes.c_int),
                ("wdtype", ctypes.c_int)]


class Q4(ctypes.Structure):
    """One expert matrix in the 4-bit group-affine format (codes, scales, biases)."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p)]


def lib_path(mutation: int = 0) -> str:
    if mutation == 0:
        return os.path.join(_HERE, "liboracle.so")
    return os.path.join(_HERE, "_mut", f"liboracle_m{mutation}.so")


def build(mutation: int = 0, force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (OpenMP, -O2, IEEE arithmetic)."""
    out = lib_path(mutation)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           f"-DORACLE_MUTATION={mutation}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(mutation: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutation in _LIBS:
            return _LIBS[mutation]
        lib = ctypes.CDLL(build(mutation))
        vp, ip = ctypes.c_void_p, ctypes.c_int
        lib.oracle_route.argtypes = [ctypes.POINTER(Dims), vp, ip, vp, vp, vp, vp, vp, vp, ip]
        lib.oracle_route.restype = ip
        lib.oracle_forward.argtypes = [ctypes.POINTER(Dims), vp, ip, vp, vp,
                                       vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ip]
        lib.oracle_forward.restype = ip
        _LIBS[mutation] = lib
        return lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return 0
    if a.dtype == np.float32:
        return 1
    raise TypeError(f"oracle takes uint16 (bf16 bits) or float32, got {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dt=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if dt is not None and a.dtype != dt:
        raise TypeError(f"expected {dt}, got {a.dtype}")
    return a


def _default_threads() -> int:
    return int(os.environ.get("ORACLE_THREADS", os.cpu_count() or 1))


def route(x, wr, k, bias=None, nthreads=None, mutation=0):
    """Router of the block: returns (idx[T][k] int32, w[T][k] f64, logits[T][E] f32, counts[E] int32).

    x: [T][d], wr: [E][d], same element type; bias: float32 [E] or None.
    """
    x, wr = _c(x), _c(wr)
    dt = _dtype_code(x)
    assert _dtype_code(wr) == dt
    T, d = x.shape
    E = wr.shape[0]
    bias = _c(bias, np.float32)
    dims = Dims(d, 1, E, k, 0, dt, dt)
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    logits = np.zeros((T, E), np.float32)
    counts = np.zeros((E,), np.int32)
    rc = load(mutation).oracle_route(ctypes.byref(dims), _ptr(x), T, _ptr(wr), _ptr(bias),
                                     _ptr(idx), _ptr(w), _ptr(logits), _ptr(counts),
                                     nthreads or _default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_route failed: {rc}")
    return idx, w, logits, counts


def forward(x, wr, wg, wu, wd, k, sg=None, su=None, sd=None, bias=None, nthreads=None,
            mutation=0, q4=False, F=None):
    """The whole block: returns (out[T][d] f64, idx, w, counts).

    wg, wu: [E][F][d] arrays or length-E sequences of [F][d] arrays (None where an
    expert is never selected); wd likewise with [d][F].  sg/su/sd: shared expert
    ([F][d], [F][d], [d][F]) or all None for no shared expert.  With q4=True
    every expert matrix is instead a (codes uint8 [rows][cols/2], scales uint16
    [rows][cols/64], biases uint16 [rows][cols/64]) triple of the 4-bit
    group-affine format, and F must be given.
    """
    x, wr = _c(x), _c(wr)
    dt = _dtype_code(x)
    T, d = x.shape
    E = wr.shape[0]
    keep = []  # arrays and records that must outlive the call

    def one(a):
        """Pointer to one expert matrix (dense array or Q4 record)."""
        if a is None:
            return None
        if q4:
            c, sc, bi = (_c(a[0], np.uint8), _c(a[1], np.uint16), _c(a[2], np.uint16))
            rec = Q4(c.ctypes.data, sc.ctypes.data, bi.ctypes.data)
            keep.extend([c, sc, bi, rec])
            return ctypes.addressof(rec)
        arr = _c(a)
        assert _dtype_code(arr) == dt
        keep.append(arr)
        return arr.ctypes.data

    def plist(ws):
        return (ctypes.c_void_p * E)(*[one(a) for a in ws])

    wg_p, wu_p, wd_p = plist(wg), plist(wu), plist(wd)
    if F is None:
        F = next(a.shape[0] for a in wg if a is not None) if any(a is not None for a in wg) else (
            sg.shape[0])
    n_shared = 0 if sg is None else 1
    if q4:
        sgp, sup, sdp = one(sg), one(su), one(sd)
    else:
        sg, su, sd = _c(sg), _c(su), _c(sd)
        sgp, sup, sdp = _ptr(sg), _ptr(su), _ptr(sd)
    bias = _c(bias, np.float32)
    dims = Dims(d, F, E, k, n_shared, dt, 2 if q4 else dt)
    out = np.zeros((T, d), np.float64)
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    counts = np.zeros((E,), np.int32)
    rc = load(mutation).oracle_forward(
        ctypes.byref(dims), _ptr(x), T, _ptr(wr), _ptr(bias),
        ctypes.cast(wg_p, ctypes.c_void_p), ctypes.cast(wu_p, ctypes.c_void_p),
        ctypes.cast(wd_p, ctypes.c_void_p), sgp, sup, sdp,
        _ptr(out), _ptr(idx), _ptr(w), _ptr(counts), nthreads or _default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_forward failed: {rc}")
    del keep  # the pointed-to arrays lived until here
    return out, idx, w, counts


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(v, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _bf16_value(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def quantize_q4(w, mutation: int = 0):
    """4-bit group-affine quantisation of w[rows][cols] (float32, or bf16 bits as
    uint16), cols a multiple of 64.  Returns (codes uint8 [rows][cols/2], scales
    uint16 [rows][cols/64], biases uint16 [rows][cols/64]), bf16 bit patterns.

    "Optimizing on-device inference for Apple Silicon", section "Dequantise
    weights within matrix multiplication": every weight is a 4-bit code and
    every group of 64 weights shares one bfloat16 scale and one bias, from which
    its values are rebuilt as scale * code + bias.  The page does not say how
    the codes are chosen; the reading taken here is the plain min/max one:
    bias = the group minimum and scale = (max - min) / 15, each rounded to
    bfloat16, code = the nearest integer (ties to even) to (w - bias) / scale,
    clamped to 0..15 (0 where the scale is 0).  Every decision is taken in
    float32.  Packing: two codes per byte along the row, the even column in the
    low nibble.

    mutation plants a mistake for the pin tests: 1 packs the odd column in the
    low nibble, 2 rounds the code down, 3 divides the range by 16.
    """
    w = np.asarray(w)
    v = _bf16_value(w) if w.dtype == np.uint16 else np.asarray(w, np.float32)
    rows, cols = v.shape
    assert cols % 64 == 0
    g = v.reshape(rows, cols // 64, 64)
    lo = g.min(axis=2)
    hi = g.max(axis=2)
    steps = np.float32(16.0 if mutation == 3 else 15.0)
    scales = _bf16_bits((hi - lo) / steps)
    biases = _bf16_bits(lo)
    s = _bf16_value(scales)[:, :, None]
    b = _bf16_value(biases)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (g - b) / np.where(s > 0, s, np.float32(1.0))
    q = np.floor(r) if mutation == 2 else np.rint(r)
    q = np.where(s > 0, np.clip(q, 0, 15), 0).astype(np.uint8).reshape(rows, cols)
    even, odd = q[:, 0::2], q[:, 1::2]
    codes = (odd | (even << 4)) if mutation == 1 else (even | (odd << 4))
    return codes.astype(np.uint8), scales, biases


def dequantize_q4(codes, scales, biases) -> np.ndarray:
    """float64 values scale * code + bias of a 4-bit matrix (layout as quantize_q4)."""
    codes = np.asarray(codes, np.uint8)
    rows = codes.shape[0]
    q = np.stack([codes & 15, codes >> 4], axis=-1).reshape(rows, -1).astype(np.float64)
    s = np.repeat(_bf16_value(scales).astype(np.float64), 64, axis=1)
    b = np.repeat(_bf16_value(biases).astype(np.float64), 64, axis=1)
    return q * s + b


from .gdn import gdn_scan  # noqa: E402  (the Gated DeltaNet scan, float64)
