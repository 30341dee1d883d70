"""Shared plumbing for the GPU parity tests: move the seeded numpy inputs to the
device, run the CUDA path through the C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import precision_attention_numerics_gb300 as aq

# Acceptance bars (stated for the forward pass): per-head relative Frobenius
# difference from the oracle's quantised emulation, and per-head error
# against FP64 within 5% of the oracle's.
REL_F_TOL = 2e-3
ERR_REL_TOL = 0.05


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def gpu_prepare(q, k, v, flags: int, signs=None, vt: bool = True, stat_len: int = 0):
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    in_dtype = aq.ATTNQ_BF16 if q.dtype == np.uint16 else aq.ATTNQ_F32
    st = None if signs is None else torch.from_numpy(np.ascontiguousarray(signs, dtype=np.int8)).cuda()
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, in_dtype, flags | (aq.ATTNQ_VT_LAYOUT if vt else 0), st, stat_len)
    bufs = aq.alloc_prepared(desc)
    Q, K, V = dev(q), dev(k), dev(v)
    aq.attnq_prepare(desc, Q, K, V, bufs.q8, bufs.k8, bufs.v8, bufs.scales, bufs.workspace)
    status = aq.attnq_device_status()
    return desc, bufs, status


def prepared_to_numpy(desc, bufs):
    """Device results in the oracle's layout (v8 untransposed)."""
    N = desc.N

    def codes(t):
        # INT8 codes held in bf16 come back as int8 (the values are exact integers)
        return t.float().cpu().numpy().astype(np.int8) if t.dtype == torch.bfloat16 else t.cpu().numpy()

    out = dict(q8=codes(bufs.q8), k8=codes(bufs.k8),
               q_descale=bufs.scales.q_descale.cpu().numpy(), k_descale=bufs.scales.k_descale.cpu().numpy(),
               v_descale=bufs.scales.v_descale.cpu().numpy(),
               k_mean=bufs.scales.k_mean.cpu().numpy() if bufs.scales.k_mean is not None else None)
    v8 = bufs.v8.cpu().numpy()
    if desc.flags & aq.ATTNQ_VT_LAYOUT:
        out["v8_pad"] = v8[..., N:]
        v8 = np.ascontiguousarray(np.swapaxes(v8[..., :N], -1, -2))
    out["v8"] = v8
    return out


def gpu_fwd(desc, bufs, S, order, causal, T, out_dtype=torch.float32, count=True, k_sink=4):
    O = torch.empty((desc.B, desc.Hq, desc.N, desc.d), dtype=out_dtype, device="cuda")
    uf = torch.zeros(desc.B * desc.Hq * 2, dtype=torch.int64, device="cuda") if count else None
    aq.attnq_fwd(desc, bufs.q8, bufs.k8, bufs.v8, bufs.scales, S, order, causal, T, O, uf, k_sink)
    status = aq.attnq_device_status()
    return O, (uf.cpu().numpy().reshape(-1, 2).astype(np.uint64) if count else None), status


def o_to_numpy(O: torch.Tensor) -> np.ndarray:
    if O.dtype == torch.bfloat16:
        return O.float().cpu().numpy().astype(np.float64)
    return O.cpu().numpy().astype(np.float64)


def rel_f(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Per-head relative Frobenius difference ||a - b|| / ||b|| over the last two axes."""
    a = a.reshape(-1, a.shape[-2] * a.shape[-1]) if a.ndim > 2 else a
    b = b.reshape(-1, b.shape[-2] * b.shape[-1]) if b.ndim > 2 else b
    return np.linalg.norm(a - b, axis=-1) / np.maximum(np.linalg.norm(b, axis=-1), 1e-300)


def oracle_bf16(O: np.ndarray) -> np.ndarray:
    import synth
    return synth.bf16_bits_to_f32(oracle.round_bf16(O)).astype(np.float64)
