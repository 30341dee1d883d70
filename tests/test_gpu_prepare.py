"""GPU parity of attnq_prepare: E4M3 operands, descales and the mean key must
match the oracle bit for bit (centring, rotation, scales and the cast are
fixed-order IEEE arithmetic on both sides)."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


def _check_prepare(q, k, v, flags, signs, vt=True):
    from tests.gpu_helpers import gpu_prepare, prepared_to_numpy
    desc, bufs, status = gpu_prepare(q, k, v, flags, signs, vt=vt)
    assert status == 0
    got = prepared_to_numpy(desc, bufs)
    ref = oracle.prepare(q, k, v, flags=flags, signs=signs)
    for name in ("q_descale", "k_descale", "v_descale"):
        assert np.array_equal(got[name].view(np.uint32), ref[name].view(np.uint32)), name
    assert np.array_equal(got["k_mean"].view(np.uint32), ref["k_mean"].view(np.uint32))
    for name in ("q8", "k8", "v8"):
        bad = np.flatnonzero(got[name] != ref[name])
        assert bad.size == 0, (name, bad.size, bad[:8])
    if vt:
        assert np.all(got["v8_pad"] == 0)


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("d", [64, 128])
def test_prepare_bf16_qwen_like(flags, d):
    B, Hq, Hkv, N = 2, 6, 2, 300
    q, k, v = synth.qwen_like_inputs(7 + d + flags, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    _check_prepare(q, k, v, flags, synth.hadamard_signs(11, d))


@pytest.mark.parametrize("N", [1, 2, 3, 17, 63, 64, 65, 127, 129, 257])
def test_prepare_ragged_lengths(N):
    d = 128
    q, k, v = synth.qwen_like_inputs(100 + N, 1, 2, 1, N, d, key_norm=40.0, key_channels=8)
    _check_prepare(q, k, v, 3, synth.hadamard_signs(12, d))


@pytest.mark.parametrize("d", [64, 128])
def test_prepare_f32_sinks(d):
    q, k, v = synth.sink_inputs(5, 1, 3, 256, d, delta=7.0)
    _check_prepare(q, k, v, 0, None)
    _check_prepare(q, k, v, 3, synth.hadamard_signs(13, d))


def test_prepare_natural_v_layout():
    q, k, v = synth.qwen_like_inputs(9, 1, 4, 2, 130, 64, key_norm=30.0, key_channels=4)
    _check_prepare(q, k, v, 2, None, vt=False)


def test_prepare_long_mean_chunks():
    # many 128-token chunks plus a ragged one, bf16 with a large shared key
    q, k, v = synth.qwen_like_inputs(21, 1, 1, 1, 4096 + 77, 128, key_norm=40.0, key_channels=8)
    _check_prepare(q, k, v, 3, synth.hadamard_signs(14, 128))


def test_prepare_cast_covers_every_float_up_to_448():
    """With a slice whose amax is exactly 448 the scale is 1, so the cast sees
    the raw value: every non-negative float32 bit pattern up to 448 (and the
    negated copies) must encode exactly as the oracle's E4M3 encoder does."""
    from tests.gpu_helpers import gpu_prepare
    d = 128
    top = int(np.float32(448.0).view(np.uint32))
    chunk = 1 << 26
    for start in range(0, top + 1, chunk):
        n = min(chunk, top + 1 - start)
        bits = np.arange(start, start + n, dtype=np.uint64).astype(np.uint32)
        vals = bits.view(np.float32)
        rows = (n + d - 1) // d + 1
        flat = np.zeros(rows * d * 2, np.float32)
        flat[:n] = vals
        flat[rows * d: rows * d + n] = -vals
        flat[-1] = 448.0
        v = flat.reshape(1, 1, 2 * rows, d)
        q = np.ones((1, 1, 2 * rows, d), np.float32)
        desc, bufs, status = gpu_prepare(q, q, v, 0, None, vt=False)
        assert status == 0
        assert float(bufs.scales.v_descale[0]) == 1.0
        got = bufs.v8.cpu().numpy().reshape(-1)
        ref_pos = oracle.e4m3_encode_bits(start, n)
        assert np.array_equal(got[:n], ref_pos), start
        assert np.array_equal(got[rows * d: rows * d + n], ref_pos | np.uint8(0x80)), start


def test_prepare_cast_saturates_every_finite_float_above_448():
    """With statistics from a first token whose amax is 448 the scale is 1 and
    later tokens reach the cast unscaled: every finite float32 above 448 (and
    its negation) must encode as the oracle's encoder does, i.e. saturate."""
    from tests.gpu_helpers import gpu_prepare
    d = 128
    lo = int(np.float32(448.0).view(np.uint32)) + 1
    hi = int(np.float32(np.finfo(np.float32).max).view(np.uint32))
    chunk = 1 << 26
    for start in range(lo, hi + 1, chunk):
        n = min(chunk, hi + 1 - start)
        vals = np.arange(start, start + n, dtype=np.uint32).view(np.float32)
        rows = (n + d - 1) // d
        flat = np.zeros((1 + 2 * rows) * d, np.float32)
        flat[0] = 448.0  # the statistics token
        flat[d: d + n] = vals
        flat[(1 + rows) * d: (1 + rows) * d + n] = -vals
        v = flat.reshape(1, 1, 1 + 2 * rows, d)
        q = np.ones_like(v)
        desc, bufs, status = gpu_prepare(q, q, v, 0, None, vt=False, stat_len=1)
        assert status == 0
        assert float(bufs.scales.v_descale[0]) == 1.0
        got = bufs.v8.cpu().numpy().reshape(-1)
        ref_pos = oracle.e4m3_encode_bits(start, n)
        assert np.all(ref_pos == 0x7E)
        assert np.array_equal(got[d: d + n], ref_pos), start
        assert np.array_equal(got[(1 + rows) * d: (1 + rows) * d + n], ref_pos | np.uint8(0x80)), start


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_prepare_reports_nonfinite(bad):
    from tests.gpu_helpers import gpu_prepare
    q, k, v = synth.qkv_normal(3, 1, 2, 1, 64, 64)
    k[0, 0, 10, 3] = bad
    _, _, status = gpu_prepare(q, k, v, 0, None)
    assert status == 4
    _, _, status = gpu_prepare(q, k, v, 3, synth.hadamard_signs(1, 64))
    assert status == 4
    q2, k2, v2 = synth.qkv_normal(3, 1, 2, 1, 64, 64)
    _, _, status = gpu_prepare(q2, k2, v2, 3, synth.hadamard_signs(1, 64))
    assert status == 0       # the status word was cleared by the last read


def _bf16_inputs(qf, kf, vf):
    return tuple(synth.to_bf16_bits(np.ascontiguousarray(x, dtype=np.float32)) for x in (qf, kf, vf))


@pytest.mark.parametrize("case", ["near_ties", "late_outlier", "wide_range", "tiny", "small"])
def test_rotated_amax_edge_cases(case):
    """The amax of rotated, uncentred bf16 slices (d = 128) is the maximum of
    the exact butterfly outputs over all rows, whatever row or tile holds it;
    scales and codes must equal the oracle's bit for bit.  Cases: rows whose
    rotated maxima nearly tie (copies of one row, one element nudged by about
    a bf16 ulp), the slice maximum in a single late row, rows mixing
    magnitudes 2^20 and 2^-20, and slices of values near 1e-33 and 1e-28."""
    d, N = 128, 1000
    rng = np.random.default_rng(17)
    qf, kf, vf = (x.astype(np.float64) for x in synth.qkv_normal(31, 1, 4, 2, N, d))
    if case == "near_ties":
        base = qf[0, 0, 0].copy()
        for h in range(4):
            for t in range(N):
                row = base.copy()
                row[(7 * t + h) % d] *= 1.0 + 2.0 ** -7 * ((t % 3) - 1)
                qf[0, h, t] = row
    elif case == "late_outlier":
        qf[0, :, N - 3] *= 6.0
        kf[0, :, N - 1] *= 9.0
    elif case == "wide_range":
        scale = np.where(rng.random((1, 4, N, d)) < 0.5, 2.0 ** 20, 2.0 ** -20)
        qf = qf * scale
    elif case == "tiny":
        qf, kf = qf * 1e-33, kf * 1e-33
    elif case == "small":
        qf, kf = qf * 1e-28, kf * 1e-28
    q, k, v = _bf16_inputs(qf, kf, vf)
    _check_prepare(q, k, v, 1, synth.hadamard_signs(15, d))
