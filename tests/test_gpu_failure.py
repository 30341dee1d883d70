"""Failure detection and out-of-bounds checks on the GPU, without a fault.

* Timeout path: with the wait limit at 0 every wait inside a kernel that is not
  already satisfied gives up; the kernel records ATTNQ_ETIMEOUT, drains its
  copies and tensor-core work (own one-second bound), frees tensor memory and
  returns.  The context stays usable: the next call with the normal limit
  succeeds and matches the oracle.
* Guard bands: outputs are written into the middle of larger buffers whose
  margins hold a known pattern; after prepare and forward the margins must be
  untouched (no write outside the tensor, including ragged tails)."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

ETIMEOUT = 5
GUARD = 4096  # bytes of margin on each side (a multiple of 256: keeps the alignment)


def _set_limit(ns):
    import precision_attention_numerics_gb300 as aq
    return aq.attnq_set_wait_limit_ns(ns)


def test_prepare_timeout_path_then_recovers():
    from tests.gpu_helpers import gpu_prepare, prepared_to_numpy
    q, k, v = synth.qwen_like_inputs(300, 2, 8, 2, 3000, 128, key_norm=30.0, key_channels=4)
    signs = synth.hadamard_signs(7, 128)
    codes = []
    prev = _set_limit(0)
    try:
        for _ in range(3):
            _, _, st = gpu_prepare(q, k, v, 3, signs)
            codes.append(st)
            if st == ETIMEOUT:
                break
    finally:
        _set_limit(prev)
    assert set(codes) <= {0, ETIMEOUT} and ETIMEOUT in codes, codes
    desc, bufs, st = gpu_prepare(q, k, v, 3, signs)
    assert st == 0
    got = prepared_to_numpy(desc, bufs)
    ref = oracle.prepare(q, k, v, flags=3, signs=signs)
    for name in ("q8", "k8", "v8"):
        assert np.array_equal(got[name], ref[name]), name


def test_fwd_timeout_path_then_recovers():
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, rel_f
    q, k, v = synth.qwen_like_inputs(301, 1, 4, 1, 2000, 128, key_norm=30.0, key_channels=4)
    desc, bufs, st = gpu_prepare(q, k, v, 0, None)
    assert st == 0
    codes = []
    prev = _set_limit(0)
    try:
        for _ in range(3):
            _, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, 128, count=False)
            codes.append(st)
            if st == ETIMEOUT:
                break
    finally:
        _set_limit(prev)
    assert set(codes) <= {0, ETIMEOUT} and ETIMEOUT in codes, codes
    O, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, 128, count=False)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=0)
    ref, _ = oracle.attn_quant(prep, (1, 4, 1, 2000, 128), 0, 256.0, 1, True, 128)
    assert rel_f(o_to_numpy(O).reshape(4, 2000, 128), ref).max() <= REL_F_TOL


def _guarded(shape, dtype, fill):
    """A tensor of `shape` inside a byte buffer with GUARD-byte margins set to `fill`."""
    es = torch.empty((), dtype=dtype).element_size()
    n = int(np.prod(shape)) * es
    raw = torch.full((GUARD + n + GUARD,), fill, dtype=torch.uint8, device="cuda")
    inner = raw[GUARD:GUARD + n].view(dtype).view(shape)
    return raw, inner


def _margins_intact(raw, n, fill):
    host = raw.cpu().numpy()
    return bool(np.all(host[:GUARD] == fill) and np.all(host[GUARD + n:] == fill))


@pytest.mark.parametrize("N,vt", [(1, True), (129, True), (257, False), (1000, True)])
def test_guard_bands_prepare_and_fwd(N, vt):
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import dev
    B, Hq, Hkv, d = 1, 4, 2, 128
    q, k, v = synth.qwen_like_inputs(310 + N, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    signs = torch.from_numpy(synth.hadamard_signs(8, d)).cuda()
    flags = aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K | (aq.ATTNQ_VT_LAYOUT if vt else 0)
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16, flags, signs)
    fill = 0xA5
    rq, q8 = _guarded((B, Hq, N, d), torch.uint8, fill)
    rk, k8 = _guarded((B, Hkv, N, d), torch.uint8, fill)
    vshape = (B, Hkv, d, aq.attnq_vt_ld(N)) if vt else (B, Hkv, N, d)
    rv, v8 = _guarded(vshape, torch.uint8, fill)
    scales = aq.AttnqScales(torch.empty(B * Hq, device="cuda"), torch.empty(B * Hkv, device="cuda"),
                            torch.empty(B * Hkv, device="cuda"), torch.empty(B * Hkv * d, device="cuda"))
    ws = torch.empty(max(aq.attnq_prepare_workspace(desc), 256), dtype=torch.uint8, device="cuda")
    aq.attnq_prepare(desc, dev(q), dev(k), dev(v), q8, k8, v8, scales, ws)
    assert aq.attnq_device_status() == 0
    checks = [(rq, q8), (rk, k8), (rv, v8)]
    if vt:  # the forward pass takes V in the transposed layout only
        ro, O = _guarded((B, Hq, N, d), torch.bfloat16, fill)
        aq.attnq_fwd(desc, q8, k8, v8, scales, 256.0, aq.ATTNQ_KV_REVERSE, True, 128, O)
        assert aq.attnq_device_status() == 0
        checks.append((ro, O))
    for raw, t in checks:
        assert _margins_intact(raw, t.numel() * t.element_size(), fill)
    ref = oracle.prepare(q, k, v, flags=flags & 3, signs=synth.hadamard_signs(8, d))
    assert np.array_equal(q8.cpu().numpy(), ref["q8"]) and np.array_equal(k8.cpu().numpy(), ref["k8"])


@pytest.mark.parametrize("mode", ["int8", "prefix"])
def test_timeout_path_of_the_other_instances_then_recovers(mode):
    """The INT8-QK and causal-prefix instances have their own code around the
    same waits (one staging buffer, one Q buffer, skipped items): each gives up
    with ETIMEOUT under a zero limit and works again afterwards."""
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, prepared_to_numpy, rel_f
    B, Hq, Hkv, N, d = 1, 4, 2, 3000, 128
    q, k, v = synth.qwen_like_inputs(320, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    signs = synth.hadamard_signs(9, d)
    flags, P = (3 | 16, 0) if mode == "int8" else (3, 1000)
    codes_p, codes_f = [], []
    desc, bufs, _ = gpu_prepare(q, k, v, flags, signs, stat_len=P)
    prev = _set_limit(0)
    try:
        for _ in range(3):
            _, _, st = gpu_prepare(q, k, v, flags, signs, stat_len=P)
            codes_p.append(st)
            _, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, 128, count=False)
            codes_f.append(st)
            if ETIMEOUT in codes_p and ETIMEOUT in codes_f:
                break
    finally:
        _set_limit(prev)
    for codes in (codes_p, codes_f):
        assert set(codes) <= {0, ETIMEOUT} and ETIMEOUT in codes, (codes_p, codes_f)
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs, stat_len=P)
    assert st == 0
    got = prepared_to_numpy(desc, bufs)
    ref = oracle.prepare(q, k, v, flags=flags, signs=signs, stat_len=P)
    for name in ("q8", "k8", "v8"):
        assert np.array_equal(got[name], ref[name]), name
    O, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, 128, count=False)
    assert st == 0
    emu, _ = oracle.attn_quant(ref, (B, Hq, Hkv, N, d), flags, 256.0, 1, True, 128)
    assert rel_f(o_to_numpy(O).reshape(B * Hq, N, d), emu).max() <= REL_F_TOL


@pytest.mark.parametrize("N", [1, 129, 1000])
def test_guard_bands_int8(N):
    """INT8 Q/K codes are bf16 rows of 2d bytes stored as 128-byte boxes: no
    write may leave the tensors, ragged tails included."""
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import dev
    B, Hq, Hkv, d = 1, 4, 2, 128
    q, k, v = synth.qwen_like_inputs(330 + N, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    signs = torch.from_numpy(synth.hadamard_signs(8, d)).cuda()
    flags = aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K | aq.ATTNQ_VT_LAYOUT | aq.ATTNQ_I8QK
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16, flags, signs)
    fill = 0x5A
    rq, q8 = _guarded((B, Hq, N, d), torch.bfloat16, fill)
    rk, k8 = _guarded((B, Hkv, N, d), torch.bfloat16, fill)
    rv, v8 = _guarded((B, Hkv, d, aq.attnq_vt_ld(N)), torch.uint8, fill)
    scales = aq.AttnqScales(torch.empty(B * Hq, device="cuda"), torch.empty(B * Hkv, device="cuda"),
                            torch.empty(B * Hkv, device="cuda"), torch.empty(B * Hkv * d, device="cuda"))
    ws = torch.empty(max(aq.attnq_prepare_workspace(desc), 256), dtype=torch.uint8, device="cuda")
    aq.attnq_prepare(desc, dev(q), dev(k), dev(v), q8, k8, v8, scales, ws)
    assert aq.attnq_device_status() == 0
    ro, O = _guarded((B, Hq, N, d), torch.bfloat16, fill)
    aq.attnq_fwd(desc, q8, k8, v8, scales, 256.0, aq.ATTNQ_KV_REVERSE, True, 128, O)
    assert aq.attnq_device_status() == 0
    for raw, t in ((rq, q8), (rk, k8), (rv, v8), (ro, O)):
        assert _margins_intact(raw, t.numel() * t.element_size(), fill)
    ref = oracle.prepare(q, k, v, flags=3 | 16, signs=synth.hadamard_signs(8, d))
    assert np.array_equal(q8.float().cpu().numpy().astype(np.int8), ref["q8"])
    assert np.array_equal(k8.float().cpu().numpy().astype(np.int8), ref["k8"])
