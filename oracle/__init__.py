"""CPU oracle for causal FP8 (E4M3) attention with the pages' numerics options.

TEST INFRASTRUCTURE: only tests/, the smoke check and the benchmark's CPU
baseline leg use this package.  It shares no code with the CUDA library and
never imports it.  The arithmetic lives in attnq_oracle.cpp (plain C++17,
strict IEEE); this module marshals numpy arrays into it.  Closed forms from the
P-cast page are in oracle.closed_forms.

Every function here has a pin in tests/test_oracle_*.py; nothing is "parity
unpinned" except the two items listed in closed_forms' header.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

ROTATE = 1
CENTER_K = 2
TILE_SCALES = 8
I8QK = 16
SCALE_TILE = 128
F32 = 0
BF16 = 1
NO_PCAST = 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        i32, i64, u32, f32 = C.c_int, C.c_int64, C.c_uint, C.c_float
        L.orc_e4m3_decode.restype = C.c_double
        L.orc_e4m3_decode.argtypes = [C.c_uint8]
        L.orc_e4m3_encode.restype = C.c_uint8
        L.orc_e4m3_encode.argtypes = [f32]
        L.orc_e4m3_encode_array.argtypes = [P, P, i64]
        L.orc_int8_encode_array.argtypes = [P, P, i64]
        L.orc_e4m3_encode_bits_range.argtypes = [C.c_uint64, i64, P]
        L.orc_double_to_bf16_array.argtypes = [P, P, i64]
        L.orc_fwht.argtypes = [P, i32]
        L.orc_mean_key.argtypes = [i32, i32, i32, P, P]
        L.orc_prepare.restype = i32
        L.orc_prepare.argtypes = [i32, i32, i32, i32, i32, i32, u32, i32, P, P, P, P, P, P, P, P, P, P, P]
        L.orc_attn_exact.restype = i32
        L.orc_attn_exact.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, i32, P, i32, P, i32, P]
        L.orc_attn_quant.restype = i32
        L.orc_attn_quant.argtypes = [i32, i32, i32, i32, i32, u32, P, P, P, P, P, P, f32, i32, i32, i32, i32, i32,
                                     P, i32, P, i32, P, P]
        L.orc_attn_ponly.restype = i32
        L.orc_attn_ponly.argtypes = [i32, i32, i32, i32, i32, P, P, P, f32, i32, i32, i32, i32, i32, P, i32, P, i32,
                                     P, P]
        L.orc_err.restype = i32
        L.orc_err.argtypes = [i64, i64, P, P, P]
        L.orc_set_threads.argtypes = [i32]
        L.orc_get_threads.restype = i32
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def threads() -> int:
    return int(lib().orc_get_threads())


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle status {code}")
        self.code = code


def _check(rc):
    if rc != 0:
        raise OracleError(rc)


# ---- E4M3 ------------------------------------------------------------------

def e4m3_decode_table() -> np.ndarray:
    L = lib()
    return np.array([L.orc_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_p(x), _p(out), x.size)
    return out


def int8_encode(x) -> np.ndarray:
    """Symmetric INT8 codes: nearest integer, ties to even, saturated to +-127."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.int8)
    lib().orc_int8_encode_array(_p(x), _p(out), x.size)
    return out


def e4m3_encode_bits(start: int, count: int) -> np.ndarray:
    """Codes for every float32 bit pattern start .. start+count-1."""
    out = np.empty(count, dtype=np.uint8)
    lib().orc_e4m3_encode_bits_range(start, count, _p(out))
    return out


def round_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_double_to_bf16_array(_p(x), _p(out), x.size)
    return out


# ---- rotation, mean --------------------------------------------------------

def fwht(x) -> np.ndarray:
    """Unnormalised FWHT along the last axis (float32, stages h = 1, 2, ...)."""
    x = np.array(x, dtype=np.float32, copy=True)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        lib().orc_fwht(_p(row), d)
        flat[r] = row
    return flat.reshape(x.shape)


def mean_key(k_head, dtype: int) -> np.ndarray:
    k_head = np.ascontiguousarray(k_head)
    N, d = k_head.shape
    mu = np.empty(d, dtype=np.float32)
    lib().orc_mean_key(N, d, dtype, _p(k_head), _p(mu))
    return mu


def _dtype_of(a) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError("inputs are float32 arrays or bf16 bit patterns (uint16)")


def prepare(q, k, v, flags: int = 0, signs=None, stat_len: int = 0):
    """Operand preparation. Returns dict with q8, k8, v8 (natural layout),
    q_descale [B*Hq], k_descale, v_descale [B*Hkv], k_mean [B*Hkv*d].  With
    TILE_SCALES, q_descale and k_descale hold one descale per 128-row tile:
    [B*Hq*ntiles] and [B*Hkv*ntiles], ntiles = ceil(N / 128).  stat_len = P
    (1..N; 0 means N) takes the mean key and the per-(batch, head) scales
    over the first P tokens of each slice (causal-prefix statistics).  With
    I8QK, q8 and k8 are int8 arrays of symmetric INT8 codes (descale =
    amax / 127); v8 stays E4M3."""
    q, k, v = (np.ascontiguousarray(a) for a in (q, k, v))
    dt = _dtype_of(q)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if signs is not None:
        signs = np.ascontiguousarray(signs, dtype=np.int8)
    nst = (N + SCALE_TILE - 1) // SCALE_TILE if flags & TILE_SCALES else 1
    out = dict(q8=np.empty(q.shape, np.uint8), k8=np.empty(k.shape, np.uint8), v8=np.empty(v.shape, np.uint8),
               q_descale=np.empty(B * Hq * nst, np.float32), k_descale=np.empty(B * Hkv * nst, np.float32),
               v_descale=np.empty(B * Hkv, np.float32), k_mean=np.empty(B * Hkv * d, np.float32))
    rc = lib().orc_prepare(B, Hq, Hkv, N, d, dt, flags, int(stat_len), _p(signs), _p(q), _p(k), _p(v), _p(out["q8"]),
                           _p(out["k8"]), _p(out["v8"]), _p(out["q_descale"]), _p(out["k_descale"]),
                           _p(out["v_descale"]), _p(out["k_mean"]))
    _check(rc)
    if flags & I8QK:
        out["q8"], out["k8"] = out["q8"].view(np.int8), out["k8"].view(np.int8)
    return out


def _lists(bh_list, rows):
    bl = None if bh_list is None else np.ascontiguousarray(bh_list, dtype=np.int32)
    rl = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    return bl, rl


def attn_exact(q, k, v, causal: bool = True, bh_list=None, rows=None) -> np.ndarray:
    """Exact attention in double; output [n_bh, n_rows, d] (all heads/rows by default)."""
    q, k, v = (np.ascontiguousarray(a) for a in (q, k, v))
    dt = _dtype_of(q)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    bl, rl = _lists(bh_list, rows)
    nbh = B * Hq if bl is None else len(bl)
    nr = N if rl is None else len(rl)
    O = np.empty((nbh, nr, d), np.float64)
    _check(lib().orc_attn_exact(B, Hq, Hkv, N, d, dt, _p(q), _p(k), _p(v), int(causal), _p(bl), nbh, _p(rl), nr,
                                _p(O)))
    return O


def attn_quant(prep, shape, flags: int, S: float, kv_order: int, causal: bool, kv_tile: int, k_sink: int = 4,
               mode: int = 0, bh_list=None, rows=None):
    """Quantised forward emulation on prepared E4M3 operands (natural layout;
    with I8QK in flags, INT8 Q and K codes and an exact integer q.k).

    shape = (B, Hq, Hkv, N, d).  Returns (O double [n_bh, n_rows, d],
    underflow uint64 [n_bh, 2])."""
    B, Hq, Hkv, N, d = shape
    bl, rl = _lists(bh_list, rows)
    nbh = B * Hq if bl is None else len(bl)
    nr = N if rl is None else len(rl)
    O = np.empty((nbh, nr, d), np.float64)
    uf = np.zeros((nbh, 2), np.uint64)
    a = [np.ascontiguousarray(prep[x]) for x in ("q8", "k8", "v8", "q_descale", "k_descale", "v_descale")]
    _check(lib().orc_attn_quant(B, Hq, Hkv, N, d, flags, *[_p(t) for t in a], float(S), int(kv_order), int(causal),
                                int(kv_tile), int(k_sink), int(mode), _p(bl), nbh, _p(rl), nr, _p(O), _p(uf)))
    return O, uf


def attn_ponly(q, k, v, S: float, kv_order: int, causal: bool, kv_tile: int, k_sink: int = 4, mode: int = 0,
               bh_list=None, rows=None):
    """P-only emulation: float32 Q, K, V, only P cast. Returns (O double, underflow [n_bh, 2])."""
    q, k, v = (np.ascontiguousarray(a, dtype=np.float32) for a in (q, k, v))
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    bl, rl = _lists(bh_list, rows)
    nbh = B * Hq if bl is None else len(bl)
    nr = N if rl is None else len(rl)
    O = np.empty((nbh, nr, d), np.float64)
    uf = np.zeros((nbh, 2), np.uint64)
    _check(lib().orc_attn_ponly(B, Hq, Hkv, N, d, _p(q), _p(k), _p(v), float(S), int(kv_order), int(causal),
                                int(kv_tile), int(k_sink), int(mode), _p(bl), nbh, _p(rl), nr, _p(O), _p(uf)))
    return O, uf


def err(O, Oref) -> np.ndarray:
    """Per-head log1p(relative Frobenius error); O, Oref [n_heads, ...] as double."""
    O = np.ascontiguousarray(O, dtype=np.float64)
    Oref = np.ascontiguousarray(Oref, dtype=np.float64)
    nh = O.shape[0]
    n = O.size // nh
    e = np.empty(nh, np.float64)
    _check(lib().orc_err(nh, n, _p(O), _p(Oref), _p(e)))
    return e


def nonsink_in_mask(N: int, k_sink: int, causal: bool = True, rows=None) -> int:
    """Number of in-mask keys j >= k_sink summed over the given query rows."""
    r = np.arange(N) if rows is None else np.asarray(rows)
    if causal:
        return int(np.maximum(r + 1 - k_sink, 0).sum())
    return int(len(r) * max(N - k_sink, 0))
