"""ctypes binding of libattnq (include/attnq.h).  Argument marshalling only.

Tensor arguments are torch tensors on the current CUDA device (their data
pointers are passed through); `stream` defaults to torch's current stream.
Every function raises AttnqError on a non-OK status.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

ATTNQ_ROTATE = 1
ATTNQ_CENTER_K = 2
ATTNQ_VT_LAYOUT = 4
ATTNQ_TILE_SCALES = 8
ATTNQ_I8QK = 16
ATTNQ_SCALE_TILE = 128
ATTNQ_F32 = 0
ATTNQ_BF16 = 1
ATTNQ_KV_FORWARD = 0
ATTNQ_KV_REVERSE = 1

STATUS = {0: "ATTNQ_OK", 1: "ATTNQ_EINVAL", 2: "ATTNQ_EUNSUPPORTED", 3: "ATTNQ_ECUDA", 4: "ATTNQ_ENONFINITE",
          5: "ATTNQ_ETIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libattnq.so")
_lib = None


class AttnqError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class _Desc(C.Structure):
    _fields_ = [("B", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32), ("N", C.c_int32), ("d", C.c_int32),
                ("in_dtype", C.c_int32), ("flags", C.c_uint32), ("signs", C.c_void_p), ("stat_len", C.c_int32)]


class _Scales(C.Structure):
    _fields_ = [("q_descale", C.c_void_p), ("k_descale", C.c_void_p), ("v_descale", C.c_void_p),
                ("k_mean", C.c_void_p)]


@dataclass
class AttnqDesc:
    """Mirror of attnq_desc; `signs` is a device int8 tensor of d values or None;
    `stat_len` = P takes the mean key and the per-(batch, head) scales over the
    first P tokens (0: all N)."""
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    in_dtype: int = ATTNQ_BF16
    flags: int = ATTNQ_VT_LAYOUT
    signs: Optional[object] = None
    stat_len: int = 0

    def _c(self) -> _Desc:
        return _Desc(self.B, self.Hq, self.Hkv, self.N, self.d, self.in_dtype, self.flags,
                     None if self.signs is None else self.signs.data_ptr(), self.stat_len)


@dataclass
class AttnqScales:
    """Mirror of attnq_scales (device fp32 tensors; k_mean optional)."""
    q_descale: object
    k_descale: object
    v_descale: object
    k_mean: Optional[object] = None

    def _c(self) -> _Scales:
        return _Scales(self.q_descale.data_ptr(), self.k_descale.data_ptr(), self.v_descale.data_ptr(),
                       None if self.k_mean is None else self.k_mean.data_ptr())


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libattnq.so; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(python -m precision_attention_numerics_gb300._build)")
    L = C.CDLL(_LIB_PATH)
    P, i32, u32, i64, f32, sz = C.c_void_p, C.c_int32, C.c_uint32, C.c_int64, C.c_float, C.c_size_t
    L.attnq_version.restype = i32
    L.attnq_status_string.restype = C.c_char_p
    L.attnq_status_string.argtypes = [i32]
    L.attnq_vt_ld.restype = i64
    L.attnq_vt_ld.argtypes = [i32]
    L.attnq_scale_tiles.restype = i32
    L.attnq_scale_tiles.argtypes = [i32]
    L.attnq_hadamard_signs.restype = i32
    L.attnq_hadamard_signs.argtypes = [C.c_uint64, i32, P]
    L.attnq_prepare_workspace.restype = sz
    L.attnq_prepare_workspace.argtypes = [P]
    L.attnq_prepare.restype = i32
    L.attnq_prepare.argtypes = [P, P, P, P, P, P, P, P, P, sz, P]
    L.attnq_prepare_static.restype = i32
    L.attnq_prepare_static.argtypes = [P, P, P, P, P, P, P, P, P]
    L.attnq_fwd.restype = i32
    L.attnq_fwd.argtypes = [P, P, P, P, P, f32, i32, i32, i32, P, i32, P, i32, P]
    L.attnq_fwd_ponly.restype = i32
    L.attnq_fwd_ponly.argtypes = [P, P, P, P, f32, i32, i32, i32, P, P, i32, P]
    L.attnq_err.restype = i32
    L.attnq_err.argtypes = [P, P, i32, P, P, P]
    L.attnq_device_status.restype = i32
    L.attnq_device_status.argtypes = [P]
    L.attnq_set_wait_limit_ns.restype = C.c_uint64
    L.attnq_set_wait_limit_ns.argtypes = [C.c_uint64]
    L.attnq_ref_attention.restype = i32
    L.attnq_ref_attention.argtypes = [P, P, P, P, i32, P, P]
    L.attnq_harm_workspace.restype = sz
    L.attnq_harm_workspace.argtypes = [P]
    L.attnq_harm_report.restype = i32
    L.attnq_harm_report.argtypes = [P, P, P, P, f32, i32, i32, P, sz, P, P]
    L.attnq_host_pipeline_workspace.restype = sz
    L.attnq_host_pipeline_workspace.argtypes = [P, i32]
    L.attnq_attention_host.restype = i32
    L.attnq_attention_host.argtypes = [P, i32, P, P, P, f32, i32, i32, i32, P, i32, P, sz, P, P, P]
    _lib = L
    return L


def exported_symbols() -> list[str]:
    """Names declared in include/attnq.h (for the ABI test)."""
    import re
    hdr = os.path.join(os.path.dirname(_HERE), "include", "attnq.h")
    text = open(hdr).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(attnq_\w+)\s*\(", text, flags=re.M)))


def _stream(stream):
    if stream is not None:
        return C.c_void_p(int(stream))
    import torch
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _check(code: int, what: str):
    if code != 0:
        raise AttnqError(code, what)


def attnq_version() -> int:
    return int(load_library().attnq_version())


def attnq_status_string(code: int) -> str:
    return load_library().attnq_status_string(code).decode()


def attnq_vt_ld(N: int) -> int:
    return int(load_library().attnq_vt_ld(N))


def attnq_scale_tiles(N: int) -> int:
    return int(load_library().attnq_scale_tiles(N))


def attnq_hadamard_signs(seed: int, d: int) -> np.ndarray:
    out = np.empty(d, dtype=np.int8)
    _check(load_library().attnq_hadamard_signs(C.c_uint64(seed), d, out.ctypes.data_as(C.c_void_p)),
           "attnq_hadamard_signs")
    return out


def attnq_prepare_workspace(desc: AttnqDesc) -> int:
    d = desc._c()
    return int(load_library().attnq_prepare_workspace(C.byref(d)))


def attnq_prepare(desc: AttnqDesc, Q, K, V, q8, k8, v8, scales: AttnqScales, workspace, stream=None) -> None:
    d, s = desc._c(), scales._c()
    nbytes = workspace.numel() * workspace.element_size()
    _check(load_library().attnq_prepare(C.byref(d), _ptr(Q), _ptr(K), _ptr(V), _ptr(q8), _ptr(k8), _ptr(v8),
                                        C.byref(s), _ptr(workspace), nbytes, _stream(stream)), "attnq_prepare")


def attnq_prepare_static(desc: AttnqDesc, Q, K, V, q8, k8, v8, scales: AttnqScales, stream=None) -> None:
    """attnq_prepare with the library's fixed scratch array instead of a workspace
    (for callers that cannot allocate; calls must not overlap on the GPU)."""
    d, s = desc._c(), scales._c()
    _check(load_library().attnq_prepare_static(C.byref(d), _ptr(Q), _ptr(K), _ptr(V), _ptr(q8), _ptr(k8), _ptr(v8),
                                               C.byref(s), _stream(stream)), "attnq_prepare_static")


ATTNQ_STATIC_SCRATCH_BYTES = 4 << 20


def attnq_fwd(desc: AttnqDesc, q8, k8, v8, scales: AttnqScales, S: float, kv_order: int, causal: bool,
              kv_tile: int, O, underflow=None, k_sink: int = 4, stream=None) -> None:
    import torch
    d, s = desc._c(), scales._c()
    out_dtype = ATTNQ_BF16 if O.dtype == torch.bfloat16 else ATTNQ_F32
    _check(load_library().attnq_fwd(C.byref(d), _ptr(q8), _ptr(k8), _ptr(v8), C.byref(s), float(S), int(kv_order),
                                    int(bool(causal)), int(kv_tile), _ptr(O), out_dtype, _ptr(underflow),
                                    int(k_sink), _stream(stream)), "attnq_fwd")


def attnq_fwd_ponly(desc: AttnqDesc, Q, K, V, S: float, kv_order: int, causal: bool, kv_tile: int, O,
                    underflow=None, k_sink: int = 4, stream=None) -> None:
    d = desc._c()
    _check(load_library().attnq_fwd_ponly(C.byref(d), _ptr(Q), _ptr(K), _ptr(V), float(S), int(kv_order),
                                          int(bool(causal)), int(kv_tile), _ptr(O), _ptr(underflow), int(k_sink),
                                          _stream(stream)), "attnq_fwd_ponly")


def attnq_err(desc: AttnqDesc, O, O_ref, err_out, stream=None) -> None:
    import torch
    d = desc._c()
    o_dtype = ATTNQ_BF16 if O.dtype == torch.bfloat16 else ATTNQ_F32
    _check(load_library().attnq_err(C.byref(d), _ptr(O), o_dtype, _ptr(O_ref), _ptr(err_out), _stream(stream)),
           "attnq_err")


def attnq_device_status(stream=None) -> int:
    """Synchronise and return (and clear) the device status code (0 = OK)."""
    return int(load_library().attnq_device_status(_stream(stream)))


def attnq_ref_attention(desc: AttnqDesc, Q, K, V, causal: bool, O_ref, stream=None) -> None:
    """FP64 reference attention of the original inputs into O_ref (fp64 [B,Hq,N,d])."""
    d = desc._c()
    _check(load_library().attnq_ref_attention(C.byref(d), _ptr(Q), _ptr(K), _ptr(V), int(bool(causal)),
                                              _ptr(O_ref), _stream(stream)), "attnq_ref_attention")


def attnq_harm_workspace(desc: AttnqDesc) -> int:
    d = desc._c()
    return int(load_library().attnq_harm_workspace(C.byref(d)))


def attnq_harm_report(desc: AttnqDesc, Q, K, V, S: float, kv_order: int, kv_tile: int, workspace, err_out,
                      stream=None) -> None:
    """Per-head errors of the four conditions into err_out (fp64 [4, B*Hq])."""
    d = desc._c()
    _check(load_library().attnq_harm_report(C.byref(d), _ptr(Q), _ptr(K), _ptr(V), float(S), int(kv_order),
                                            int(kv_tile), _ptr(workspace), workspace.numel(), _ptr(err_out),
                                            _stream(stream)), "attnq_harm_report")


def attnq_set_wait_limit_ns(ns: int) -> int:
    """Set the limit of every wait inside the kernels (nanoseconds); returns the previous one."""
    return int(load_library().attnq_set_wait_limit_ns(int(ns)))


def attnq_host_pipeline_workspace(desc: AttnqDesc, out_dtype: int) -> int:
    d = desc._c()
    return int(load_library().attnq_host_pipeline_workspace(C.byref(d), int(out_dtype)))


def attnq_attention_host(desc: AttnqDesc, Q_host, K_host, V_host, S: float, kv_order: int, causal: bool,
                         kv_tile: int, O_host, out_dtype: int, workspace, compute, copy_in, copy_out) -> None:
    """Prepare + attention over n steps whose inputs and outputs live in host
    memory (lists of pinned CPU tensors of equal length); see include/attnq.h.
    `compute`, `copy_in`, `copy_out`: three torch.cuda.Stream objects."""
    n = len(Q_host)
    if not (len(K_host) == len(V_host) == len(O_host) == n):
        raise ValueError("Q_host, K_host, V_host and O_host must have one entry per step")
    arr = C.c_void_p * max(n, 1)
    qa, ka, va, oa = (arr(*[t.data_ptr() for t in ts]) for ts in (Q_host, K_host, V_host, O_host))
    d = desc._c()
    _check(load_library().attnq_attention_host(
        C.byref(d), n, qa, ka, va, float(S), int(kv_order), int(bool(causal)), int(kv_tile), oa, int(out_dtype),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(compute.cuda_stream),
        _stream(copy_in.cuda_stream), _stream(copy_out.cuda_stream)), "attnq_attention_host")
