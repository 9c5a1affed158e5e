"""CPU oracle for the fused MoE layer forward (test infrastructure).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It wraps `moe_oracle.c` (plain fp64 C with OpenMP over
tokens/pairs) through ctypes.  It shares no code with the GPU library.

Parity pins live in tests/test_oracle_*.py; every function here says which
part of the pages it follows in moe_oracle.c's comments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i = ctypes.c_int
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_decode.restype = ctypes.c_double
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_encode_n.argtypes = [P, ctypes.c_long, P]
            L.oracle_e4m3_encode_n.restype = None
            L.oracle_quantize_act.argtypes = [P, ctypes.c_long, P, P]
            L.oracle_quantize_act.restype = None
            L.oracle_quantize.argtypes = [ctypes.c_double, ctypes.c_float]
            L.oracle_quantize.restype = ctypes.c_uint8
            L.oracle_route_topk.argtypes = [P, i, i, i, i, P, P]
            L.oracle_route_topk.restype = None
            L.oracle_align.argtypes = [P, i, i, i, i, P, P, P, P, P]
            L.oracle_align.restype = None
            L.oracle_moe_forward.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, i, P, i, P, P, P,
                                             P, P, P, ctypes.c_float, P, i]
            L.oracle_moe_forward.restype = ctypes.c_int
            L.oracle_inv_rope_quant.argtypes = [P, P, P, P, i, i, i, i, P, P, P]
            L.oracle_inv_rope_quant.restype = i
            L.oracle_max_threads.argtypes = []
            L.oracle_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(t, dtype):
    """torch tensor / array-like -> C-contiguous numpy array of `dtype` (host copy).

    Same-width integer types (bf16 bits, E4M3 codes) are reinterpreted, not
    converted."""
    if hasattr(t, "detach"):
        import torch
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        elif t.dtype == torch.float8_e4m3fn:
            t = t.view(torch.uint8)
        t = t.numpy()
    a = np.asarray(t)
    want = np.dtype(dtype)
    if a.dtype.kind in "iu" and want.kind in "iu" and a.dtype.itemsize == want.itemsize:
        a = a.view(want)
    else:
        a = a.astype(want)
    return np.ascontiguousarray(a)


def e4m3_decode(code: int) -> float:
    return lib().oracle_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return int(lib().oracle_e4m3_encode(float(v)))


def e4m3_encode_array(v) -> np.ndarray:
    flat = np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel())
    out = np.zeros(flat.size, np.uint8)
    lib().oracle_e4m3_encode_n(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(np.shape(v))


def quantize(v: float, s: float) -> int:
    return int(lib().oracle_quantize(float(v), float(s)))


def quantize_act(x):
    """bf16 tensor -> (E4M3 codes uint8 (same shape), s fp32)."""
    xb = _np(x, np.uint16)
    codes = np.zeros(xb.shape, np.uint8)
    s = np.zeros(1, np.float32)
    lib().oracle_quantize_act(_ptr(xb), xb.size, _ptr(codes), _ptr(s))
    return codes, float(s[0])


def route_topk(logits, top_k: int, renormalize: bool):
    """-> (ids int32 [T,k], weights fp64 [T,k])."""
    lg = _np(logits, np.float32)
    T, E = lg.shape
    ids = np.zeros((T, top_k), np.int32)
    w = np.zeros((T, top_k), np.float64)
    lib().oracle_route_topk(_ptr(lg), T, E, top_k, int(bool(renormalize)), _ptr(ids), _ptr(w))
    return ids, w


def align(ids, E: int, block_m: int):
    """-> dict(counts [E], offsets [E+1], sorted_ids [num_padded], tile_expert, num_padded)."""
    ids = _np(ids, np.int32)
    T, k = ids.shape
    P = T * k
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    cap = P + E * (block_m - 1)
    sorted_ids = np.zeros(max(cap, 1), np.int32)
    tile_expert = np.zeros(max(cap // block_m, 1), np.int32)
    num_padded = np.zeros(1, np.int32)
    lib().oracle_align(_ptr(ids), T, k, E, block_m, _ptr(counts), _ptr(offsets),
                       _ptr(sorted_ids), _ptr(tile_expert), _ptr(num_padded))
    n = int(num_padded[0])
    return dict(counts=counts, offsets=offsets, sorted_ids=sorted_ids[:n],
                tile_expert=tile_expert[: n // block_m], num_padded=n)


def moe_forward(x, logits, w13, w2, w13_scale, w2_scale, top_k: int, renormalize: bool,
                rows=None, nthreads: int = 0, h_amax: float | None = None):
    """Whole-layer oracle.

    x: bf16 [T,H] (torch) or int16/uint16 bits; logits fp32 [T,E];
    w13 [E,2I,H], w2 [E,H,I]: uint8 E4M3 codes (scales given) or bf16 (scales None).
    rows: optional token indices whose output rows are wanted (all when None).
    h_amax: FP8 only: the max |h| the scale of h is taken from instead of this
    call's own (a tensor-parallel shard passes the max over all shards).
    Returns dict(out fp64 [n_rows,H], ids, weights, counts, s_x, s_h, h_amax)
    where h_amax is this call's own max |h| over its routed pairs.
    """
    xb = _np(x, np.uint16)
    lg = _np(logits, np.float32)
    T, H = xb.shape
    E = lg.shape[1]
    is_fp8 = w13_scale is not None
    if is_fp8:
        w13n = _np(w13, np.uint8)
        w2n = _np(w2, np.uint8)
        s13 = _np(w13_scale, np.float32)
        s2 = _np(w2_scale, np.float32)
    else:
        w13n = _np(w13, np.uint16)
        w2n = _np(w2, np.uint16)
        s13 = s2 = None
    I = w13n.shape[1] // 2
    assert w13n.shape == (E, 2 * I, H) and w2n.shape == (E, H, I)
    rows_np = None if rows is None else np.ascontiguousarray(np.asarray(rows, np.int32))
    n_rows = T if rows_np is None else rows_np.size
    out = np.zeros((max(n_rows, 1), H), np.float64)
    P = T * top_k
    ids = np.zeros(max(P, 1), np.int32)
    w = np.zeros(max(P, 1), np.float64)
    counts = np.zeros(E, np.int32)
    sx = np.zeros(1, np.float32)
    sh = np.zeros(1, np.float32)
    ha = np.zeros(1, np.float32)
    rc = lib().oracle_moe_forward(_ptr(xb), _ptr(lg), _ptr(w13n), _ptr(w2n), _ptr(s13), _ptr(s2),
                                  int(is_fp8), T, H, I, E, top_k, int(bool(renormalize)),
                                  _ptr(rows_np), n_rows, _ptr(out), _ptr(ids), _ptr(w),
                                  _ptr(counts), _ptr(sx), _ptr(sh),
                                  float(h_amax) if h_amax is not None else 0.0, _ptr(ha),
                                  int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_moe_forward failed ({rc})")
    return dict(out=out[:n_rows], ids=ids[:P].reshape(T, top_k), weights=w[:P].reshape(T, top_k),
                counts=counts, s_x=float(sx[0]), s_h=float(sh[0]), h_amax=float(ha[0]))


def inv_rope_quant(x, positions, cos_tab, sin_tab):
    """Inverse rotary embedding + per-head E4M3 quantisation (the oracle's
    reading of the pages' fused inverse-RoPE / per-head FP8 kernel).
    x: bf16 [T, NH, D]; positions: int [T]; cos_tab, sin_tab: fp32 [max_pos, D/2].
    -> dict(codes uint8 [T, NH, D], scales fp32 [NH], y fp32 [T, NH, D])."""
    xb = _np(x, np.uint16)
    T, NH, D = xb.shape
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int32))
    c = np.ascontiguousarray(np.asarray(cos_tab, dtype=np.float32))
    sn = np.ascontiguousarray(np.asarray(sin_tab, dtype=np.float32))
    codes = np.zeros((T, NH, D), np.uint8)
    scales = np.zeros(NH, np.float32)
    y = np.zeros((T, NH, D), np.float32)
    rc = lib().oracle_inv_rope_quant(_ptr(xb), _ptr(pos), _ptr(c), _ptr(sn), T, NH, D, c.shape[0],
                                     _ptr(codes), _ptr(scales), _ptr(y))
    if rc != 0:
        raise ValueError("odd head size or position outside the tables")
    return dict(codes=codes, scales=scales, y=y)


def max_threads() -> int:
    return int(lib().oracle_max_threads())


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
