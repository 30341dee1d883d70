"""Pins for the oracle's INT8-QK / FP8-PV form (Q and K as symmetric INT8
codes, V and P as E4M3).

The "attention-numerics" page (method and kernel settings) names only the
formats.  The reading pinned here: the nearest integer with ties to even,
saturated to +-127, of fl32(x * qs) with qs = 127 / amax (one max-based scale
per (batch, head), or per 128-token tile, like the E4M3 path); q.k is an exact
integer sum.

Anchors: numpy's rint (round half to even) and clip, numpy float32
arithmetic on integer-valued inputs (where the transform is exact), and
float64 softmax attention on the dequantised operands.
"""
import numpy as np
import pytest
import scipy.linalg

import synth


def test_int8_encode_is_rint_with_saturation(orc):
    ties = np.arange(-140, 140, dtype=np.float32) + np.float32(0.5)
    dense = np.linspace(-200, 200, 400_001, dtype=np.float32)
    rnd = synth.normals(70, 100_000) * np.float32(60)
    for y in (ties, dense, rnd):
        want = np.clip(np.rint(y.astype(np.float64)), -127, 127).astype(np.int8)
        assert np.array_equal(orc.int8_encode(y), want)
    # ties go to the even neighbour
    assert np.array_equal(orc.int8_encode(np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5], np.float32)),
                          np.array([0, 2, 2, 0, -2, -2], np.int8))


@pytest.mark.parametrize("flags", [0, 1])
def test_int8_prepare_closed_form_on_integer_inputs(orc, flags):
    """Integer inputs: the FWHT is exact, so descale = fl32(amax / 127) and the
    codes are rint(fl32(x * fl32(127 / amax))) clipped, by numpy float32."""
    B, Hq, Hkv, N, d = 1, 2, 1, 200, 64
    q = ((synth.splitmix64(71, B * Hq * N * d) % np.uint64(61)).astype(np.float32) - 30).reshape(B, Hq, N, d)
    k = ((synth.splitmix64(72, B * Hkv * N * d) % np.uint64(41)).astype(np.float32) - 20).reshape(B, Hkv, N, d)
    v = synth.normals(73, B * Hkv * N * d).reshape(B, Hkv, N, d)
    signs = synth.hadamard_signs(74, d)
    p = orc.prepare(q, k, v, flags=flags | orc.I8QK, signs=signs)
    e = orc.prepare(q, k, v, flags=flags, signs=signs)
    assert np.array_equal(p["v8"], e["v8"]) and np.array_equal(p["v_descale"], e["v_descale"])
    H = scipy.linalg.hadamard(d).astype(np.int64)
    for name, x, ds in (("q8", q, p["q_descale"]), ("k8", k, p["k_descale"])):
        xi = x.astype(np.int64)
        if flags & orc.ROTATE:
            xi = (xi * signs.astype(np.int64)) @ H
        xf = xi.astype(np.float32).reshape(x.shape[0] * x.shape[1], -1)
        amax = np.abs(xf).max(-1)
        assert np.array_equal(ds, amax / np.float32(127))
        qs = np.float32(127) / amax
        y = (xf * qs[:, None]).astype(np.float32)
        want = np.clip(np.rint(y), -127, 127).astype(np.int8)
        assert p[name].dtype == np.int8
        assert np.array_equal(p[name].reshape(want.shape), want), name
        assert np.all(np.abs(p[name]).reshape(want.shape[0], -1).max(-1) == 127)


def test_int8_prepare_tile_and_prefix_scales(orc):
    """Per-tile INT8 scales are each tile's amax / 127; prefix statistics take the
    V scale and the mean from the first P tokens, as for E4M3 codes."""
    B, Hq, Hkv, N, d = 1, 2, 1, 300, 64
    qb, kb, vb = synth.qwen_like_inputs(75, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    p = orc.prepare(qb, kb, vb, flags=orc.I8QK | orc.TILE_SCALES)
    q = synth.bf16_bits_to_f32(qb)
    nt = 3
    ds = p["q_descale"].reshape(B * Hq, nt)
    for t in range(nt):
        amax = np.abs(q[0, :, t * 128:(t + 1) * 128]).reshape(Hq, -1).max(-1)
        assert np.array_equal(ds[:, t], amax / np.float32(127))
    P = 150
    pp = orc.prepare(qb, kb, vb, flags=orc.I8QK | orc.CENTER_K, stat_len=P)
    tt = orc.prepare(qb[:, :, :P], kb[:, :, :P], vb[:, :, :P], flags=orc.I8QK | orc.CENTER_K)
    for name in ("q8", "k8", "v8"):
        assert np.array_equal(pp[name][:, :, :P], tt[name]), name
    for name in ("q_descale", "k_descale", "v_descale", "k_mean"):
        assert np.array_equal(pp[name], tt[name]), name


@pytest.mark.parametrize("flags", [0, 1, 3])
@pytest.mark.parametrize("order", [0, 1])
def test_int8_emulation_without_pcast_is_attention_on_dequantised_operands(orc, flags, order):
    """Without the P cast the emulation is softmax attention on dq * q8, dk * k8,
    dv * v8 (float64; the FWHT's factor d divided out): the integer q.k, the
    127-based descales and the logit factor are all in it."""
    B, Hq, Hkv, N, d, T = 1, 2, 1, 150, 64, 64
    q, k, v = synth.qkv_normal(76, B, Hq, Hkv, N, d)
    q *= np.float32(3.0)
    signs = synth.hadamard_signs(77, d)
    fl = flags | orc.I8QK
    p = orc.prepare(q, k, v, flags=fl, signs=signs)
    O, _ = orc.attn_quant(p, (B, Hq, Hkv, N, d), fl, 256.0, order, True, T, mode=orc.NO_PCAST)
    table = orc.e4m3_decode_table()
    qd = p["q8"].astype(np.float64) * p["q_descale"].reshape(B, Hq, 1, 1)
    kd = p["k8"].astype(np.float64) * p["k_descale"].reshape(B, Hkv, 1, 1)
    vd = table[p["v8"]].astype(np.float64) * p["v_descale"].reshape(B, Hkv, 1, 1)
    scale = 1.0 / np.sqrt(d) / (d if flags & orc.ROTATE else 1)
    ref = np.empty((B * Hq, N, d))
    for h in range(Hq):
        s = qd[0, h] @ kd[0, 0].T * scale
        s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
        w = np.exp(s - s.max(-1, keepdims=True))
        ref[h] = (w / w.sum(-1, keepdims=True)) @ vd[0, 0]
    rel = np.linalg.norm(O.reshape(B * Hq, N, d) - ref, axis=(1, 2)) / np.linalg.norm(ref, axis=(1, 2))
    assert rel.max() < 2e-6, rel


def test_int8_dot_products_are_exact_at_full_range(orc):
    """Every q.k of full-range codes (|sum| up to 128 * 127^2 < 2^24) is exact:
    with one key per row the output is that key's dequantised value, and with
    two equal-logit keys the average of the two values."""
    B, Hq, Hkv, N, d, T = 1, 1, 1, 2, 128, 64
    q = np.full((B, Hq, N, d), 5.0, np.float32)
    k = np.full((B, Hkv, N, d), -3.0, np.float32)
    v = synth.normals(78, B * Hkv * N * d).reshape(B, Hkv, N, d)
    fl = orc.I8QK
    p = orc.prepare(q, k, v, flags=fl)
    assert np.all(p["q8"] == 127) and np.all(p["k8"] == -127)
    O, _ = orc.attn_quant(p, (B, Hq, Hkv, N, d), fl, 1.0, 0, True, T, mode=orc.NO_PCAST)
    table = orc.e4m3_decode_table()
    vd = table[p["v8"][0, 0]].astype(np.float64) * float(p["v_descale"][0])
    np.testing.assert_allclose(O[0, 0], vd[0], rtol=1e-7)
    np.testing.assert_allclose(O[0, 1], 0.5 * (vd[0] + vd[1]), rtol=1e-6)
