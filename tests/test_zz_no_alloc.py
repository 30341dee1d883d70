"""attnq_prepare_static: operand preparation for callers that cannot allocate
device memory at call time (a runtime plugin hook that must not allocate, a
process whose device memory belongs to another allocator).  It uses the
library's fixed scratch array instead of a caller workspace.

Checked through the C ABI against attnq_prepare (the existing entry point) on
two calls in a row with different inputs: the outputs must agree bit for bit,
the tolerance every prepare test uses.  The first call leaves a larger amax
in the shared array than the second one needs, so a second call that did not
clear it would get the wrong scales.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _outputs(bufs):
    return [bufs.q8, bufs.k8, bufs.v8, bufs.scales.q_descale, bufs.scales.k_descale, bufs.scales.v_descale,
            bufs.scales.k_mean]


def _both(q, k, v, flags, signs, stat_len=0):
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import dev
    B, Hq, N, d = q.shape
    in_dtype = aq.ATTNQ_BF16 if q.dtype == np.uint16 else aq.ATTNQ_F32
    sg = None if signs is None else torch.from_numpy(signs).cuda()
    desc = aq.AttnqDesc(B, Hq, k.shape[1], N, d, in_dtype, flags | aq.ATTNQ_VT_LAYOUT, sg, stat_len)
    Q, K, V = dev(q), dev(k), dev(v)
    ref = aq.alloc_prepared(desc)
    aq.attnq_prepare(desc, Q, K, V, ref.q8, ref.k8, ref.v8, ref.scales, ref.workspace)
    got = aq.alloc_prepared(desc)
    # the call under test goes straight through the C ABI, no workspace
    L = aq.load_library()
    d_c, s_c = desc._c(), got.scales._c()
    rc = L.attnq_prepare_static(C.byref(d_c), C.c_void_p(Q.data_ptr()), C.c_void_p(K.data_ptr()),
                                C.c_void_p(V.data_ptr()), C.c_void_p(got.q8.data_ptr()),
                                C.c_void_p(got.k8.data_ptr()), C.c_void_p(got.v8.data_ptr()), C.byref(s_c),
                                C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    assert aq.attnq_device_status() == 0
    for a, b in zip(_outputs(got), _outputs(ref)):
        assert torch.equal(a, b)
    return got


def test_static_scratch_matches_workspace_entry_point_twice():
    d = 128
    signs = synth.hadamard_signs(3, d)
    # first call: large values (a big shared key and outliers) so the amax words end high
    q1, k1, v1 = synth.qwen_like_inputs(1, 2, 8, 2, 1000, d, key_norm=400.0, key_channels=8, outlier_gain=200.0)
    _both(q1, k1, v1, 3, signs)
    # second call, right after: smaller values, other shape and flags
    q2, k2, v2 = synth.sink_inputs(2, 1, 4, 777, d, delta=6.0)
    k2, v2 = k2[:, :2].copy(), v2[:, :2].copy()
    _both(q2, k2, v2, 2, None)


def test_static_scratch_long_context_shape_fits():
    import precision_attention_numerics_gb300 as aq
    desc = aq.AttnqDesc(2, 32, 8, 32768, 128, aq.ATTNQ_BF16, aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K | aq.ATTNQ_VT_LAYOUT)
    assert aq.attnq_prepare_workspace(desc) <= aq.ATTNQ_STATIC_SCRATCH_BYTES


def test_static_scratch_rejects_too_large_before_launch():
    import precision_attention_numerics_gb300 as aq
    # 16 KV heads x 512 chunks of 128 tokens x 128 channels of fp32 partial
    # sums: just over 4 MiB, more than the array holds
    B, Hq, Hkv, N, d = 1, 16, 16, 65536, 128
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16, aq.ATTNQ_CENTER_K | aq.ATTNQ_VT_LAYOUT)
    assert aq.attnq_prepare_workspace(desc) > aq.ATTNQ_STATIC_SCRATCH_BYTES
    # every buffer is a real allocation of the size the descriptor implies,
    # so nothing passed here points outside memory this process owns
    bufs = aq.alloc_prepared(desc)
    Q = torch.zeros((B, Hq, N, d), dtype=torch.bfloat16, device="cuda")
    K = torch.zeros((B, Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    V = torch.zeros((B, Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    L = aq.load_library()
    d_c, s_c = desc._c(), bufs.scales._c()
    rc = L.attnq_prepare_static(C.byref(d_c), *(C.c_void_p(t.data_ptr()) for t in (Q, K, V, bufs.q8, bufs.k8,
                                                                                   bufs.v8)),
                                C.byref(s_c), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 2
    # nothing was launched: the outputs are as allocated and the device is clean
    assert aq.attnq_device_status() == 0


@pytest.mark.parametrize("flags,stat_len", [(3 | 16, 0), (3, 400), (3 | 16 | 8, 300)])
def test_static_scratch_with_other_forms(flags, stat_len):
    """INT8 Q/K codes, causal-prefix statistics and per-tile scales through the
    fixed scratch: bit for bit the workspace entry point's outputs."""
    d = 128
    q, k, v = synth.qwen_like_inputs(40 + stat_len, 1, 4, 2, 1000, d, key_norm=30.0, key_channels=4)
    _both(q, k, v, flags, synth.hadamard_signs(4, d), stat_len)
