"""GB300 (sm_103a) causal FP8 attention with the numerics options of the
attention-numerics pages: optional random-sign Hadamard rotation of Q and K,
optional mean-key subtraction, per-(batch, head) max-based E4M3 scales, online
softmax over KV tiles in forward or reverse order, and a static P-cast scale S.

Further options: per-128-token-tile Q/K scales (ATTNQ_TILE_SCALES), mean key
and slice scales from the first stat_len tokens (AttnqDesc.stat_len), and
INT8 Q/K codes with FP8 P and V (ATTNQ_I8QK).

The compute lives in libattnq.so (hand-written CUDA kernels behind a C ABI,
include/attnq.h).  This package is a thin ctypes binding with the same names
as the C functions; it only marshals arguments.  There is no CPU fallback:
every call raises if the library has not been built.

Typical use (device tensors from torch; Q [B,Hq,N,d], K and V [B,Hkv,N,d] bf16):

    import precision_attention_numerics_gb300 as aq
    signs = torch.from_numpy(aq.attnq_hadamard_signs(seed, d)).cuda()
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16,
                        aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K | aq.ATTNQ_VT_LAYOUT, signs)
    bufs = aq.alloc_prepared(desc)
    aq.attnq_prepare(desc, Q, K, V, bufs.q8, bufs.k8, bufs.v8, bufs.scales, bufs.workspace)
    O = torch.empty(B, Hq, N, d, dtype=torch.bfloat16, device="cuda")
    aq.attnq_fwd(desc, bufs.q8, bufs.k8, bufs.v8, bufs.scales, 256.0, aq.ATTNQ_KV_REVERSE, True, 128, O)
    assert aq.attnq_device_status() == 0
"""
from .binding import (  # noqa: F401
    ATTNQ_BF16,
    ATTNQ_CENTER_K,
    ATTNQ_F32,
    ATTNQ_KV_FORWARD,
    ATTNQ_KV_REVERSE,
    ATTNQ_ROTATE,
    ATTNQ_SCALE_TILE,
    ATTNQ_TILE_SCALES,
    ATTNQ_I8QK,
    ATTNQ_VT_LAYOUT,
    AttnqDesc,
    AttnqError,
    AttnqScales,
    STATUS,
    attnq_attention_host,
    attnq_device_status,
    attnq_err,
    attnq_fwd,
    attnq_fwd_ponly,
    attnq_hadamard_signs,
    attnq_harm_report,
    attnq_harm_workspace,
    attnq_host_pipeline_workspace,
    attnq_prepare,
    attnq_prepare_static,
    ATTNQ_STATIC_SCRATCH_BYTES,
    attnq_prepare_workspace,
    attnq_ref_attention,
    attnq_scale_tiles,
    attnq_set_wait_limit_ns,
    attnq_status_string,
    attnq_version,
    attnq_vt_ld,
    exported_symbols,
    library_path,
    load_library,
)
from .buffers import PreparedBuffers, alloc_prepared  # noqa: F401
