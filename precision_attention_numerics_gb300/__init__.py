"""GB300 (sm_103a) causal FP8 attention with the numerics options of the
attention-numerics pages: optional random-sign Hadamard rotation of Q and K,
optional mean-key subtraction, per-(batch, head) max-based E4M3 scales, online
softmax over KV tiles in forward or reverse order, and a static P-cast scale S.

The compute lives in libattnq.so (hand-written CUDA kernels behind a C ABI,
include/attnq.h).  This package is a thin ctypes binding with the same names
as the C functions; it only marshals arguments.  There is no CPU fallback:
every call raises if the library has not been built.
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
