"""Device buffers for one prepare/forward call (torch allocations only)."""
from __future__ import annotations

from dataclasses import dataclass

from .binding import (ATTNQ_I8QK, ATTNQ_TILE_SCALES, ATTNQ_VT_LAYOUT, AttnqDesc, AttnqScales, attnq_prepare_workspace,
                      attnq_scale_tiles, attnq_vt_ld)


@dataclass
class PreparedBuffers:
    q8: object
    k8: object
    v8: object
    scales: AttnqScales
    workspace: object


def alloc_prepared(desc: AttnqDesc, device="cuda", with_mean: bool = True) -> PreparedBuffers:
    """Operand tensors (E4M3 codes; Q and K as bf16-held INT8 codes with
    ATTNQ_I8QK), descales, optional mean key and workspace for `desc`."""
    import torch
    B, Hq, Hkv, N, d = desc.B, desc.Hq, desc.Hkv, desc.N, desc.d
    qk_dtype = torch.bfloat16 if desc.flags & ATTNQ_I8QK else torch.uint8
    q8 = torch.empty((B, Hq, N, d), dtype=qk_dtype, device=device)
    k8 = torch.empty((B, Hkv, N, d), dtype=qk_dtype, device=device)
    if desc.flags & ATTNQ_VT_LAYOUT:
        v8 = torch.empty((B, Hkv, d, attnq_vt_ld(N)), dtype=torch.uint8, device=device)
    else:
        v8 = torch.empty((B, Hkv, N, d), dtype=torch.uint8, device=device)
    nst = attnq_scale_tiles(N) if desc.flags & ATTNQ_TILE_SCALES else 1  # descales per Q/K slice
    scales = AttnqScales(torch.empty(B * Hq * nst, dtype=torch.float32, device=device),
                         torch.empty(B * Hkv * nst, dtype=torch.float32, device=device),
                         torch.empty(B * Hkv, dtype=torch.float32, device=device),
                         torch.empty(B * Hkv * d, dtype=torch.float32, device=device) if with_mean else None)
    ws = torch.empty(max(attnq_prepare_workspace(desc), 256), dtype=torch.uint8, device=device)
    return PreparedBuffers(q8, k8, v8, scales, ws)
