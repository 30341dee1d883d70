"""Pins for the oracle's operand preparation: the Hadamard rotation, the mean
key, the per-(batch, head) max-based scales and the cast.

Anchors: scipy's Sylvester Hadamard matrix, exact integer identities, the
orthogonality property the pages state ("rotation preserves dot products"),
float64 means from numpy, and the E4M3 error bound of a max-scaled cast.
"""
import numpy as np
import pytest
import scipy.linalg

import synth


@pytest.mark.parametrize("d", [8, 64, 128])
def test_fwht_is_sylvester_hadamard(orc, d):
    eye = np.eye(d, dtype=np.float32)
    H = orc.fwht(eye)             # row i = FWHT(e_i) = column i of H
    ref = scipy.linalg.hadamard(d)
    assert np.array_equal(H.T, ref.astype(np.float32))
    assert np.array_equal(H.astype(np.int64) @ H.astype(np.int64).T, d * np.eye(d, dtype=np.int64))


def test_rotation_preserves_dot_products(orc):
    d = 128
    rng_q = synth.normals(11, 16 * d).reshape(16, d)
    rng_k = synth.normals(12, 16 * d).reshape(16, d)
    s = synth.hadamard_signs(5, d).astype(np.float32)
    rq = orc.fwht(rng_q * s).astype(np.float64)
    rk = orc.fwht(rng_k * s).astype(np.float64)
    exact = rng_q.astype(np.float64) @ rng_k.astype(np.float64).T
    got = rq @ rk.T / d
    assert np.max(np.abs(got - exact)) <= 1e-5 * np.max(np.abs(exact))
    # float64 Hadamard on the float64 inputs: exact orthogonality to 1e-13
    H = scipy.linalg.hadamard(d).astype(np.float64)
    q64 = rng_q.astype(np.float64) * s
    k64 = rng_k.astype(np.float64) * s
    got64 = (q64 @ H) @ (k64 @ H).T / d
    assert np.max(np.abs(got64 - exact)) <= 1e-13 * np.max(np.abs(exact))


def test_fwht_sum_order_matches_stagewise_definition(orc):
    # Integer-valued inputs keep every float add exact, so the FWHT must equal
    # the integer matrix product exactly; a wrong pairing or a dropped stage
    # changes it.
    d = 64
    x = (synth.splitmix64(3, 4 * d) % np.uint64(2001)).astype(np.int64).reshape(4, d) - 1000
    got = orc.fwht(x.astype(np.float32))
    ref = x @ scipy.linalg.hadamard(d)
    assert np.array_equal(got.astype(np.int64), ref)


def test_mean_key_float_order_close_to_exact(orc):
    N, d = 1000, 64
    k = synth.normals(21, N * d).reshape(N, d) + np.float32(15.0)
    mu = orc.mean_key(k, orc.F32)
    ref = k.astype(np.float64).mean(axis=0)
    assert np.max(np.abs(mu - ref)) < 2e-5
    # integer-valued inputs: every partial sum exact, so the mean is exact
    ki = (synth.splitmix64(4, N * d) % np.uint64(64)).astype(np.float32).reshape(N, d)
    mui = orc.mean_key(ki, orc.F32)
    assert np.array_equal(mui, (ki.astype(np.float64).sum(0) / N).astype(np.float32))


def test_mean_key_bf16_matches_f32(orc):
    N, d = 300, 128
    kb = synth.to_bf16_bits(synth.normals(22, N * d).reshape(N, d))
    assert np.array_equal(orc.mean_key(kb, orc.BF16), orc.mean_key(synth.bf16_bits_to_f32(kb), orc.F32))


def _dequant(table, codes, ds, shape_bh):
    return table[codes].astype(np.float64) * ds.reshape(shape_bh + (1, 1)).astype(np.float64)


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_prepare_scales_and_cast(orc, flags):
    B, Hq, Hkv, N, d = 2, 4, 2, 200, 64
    qb, kb, vb = synth.qwen_like_inputs(31 + flags, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    signs = synth.hadamard_signs(77, d)
    p = orc.prepare(qb, kb, vb, flags=flags, signs=signs)
    table = orc.e4m3_decode_table()
    q = synth.bf16_bits_to_f32(qb).astype(np.float64)
    k = synth.bf16_bits_to_f32(kb).astype(np.float64)
    v = synth.bf16_bits_to_f32(vb).astype(np.float64)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    if flags & 2:
        mu = k.mean(axis=2, keepdims=True)
        assert np.max(np.abs(p["k_mean"].reshape(B, Hkv, 1, d) - mu)) < 1e-5
        k = k - p["k_mean"].reshape(B, Hkv, 1, d).astype(np.float64)
    else:
        assert np.all(p["k_mean"] == 0)
    if flags & 1:
        q = (q * signs) @ H
        k = (k * signs) @ H
    for name, x, ds, H_ in (("q8", q, p["q_descale"], Hq), ("k8", k, p["k_descale"], Hkv), ("v8", v, p["v_descale"], Hkv)):
        amax = np.abs(x).reshape(B, H_, -1).max(-1)
        # descale = amax / 448 (float32; float rounding of the transform allowed)
        np.testing.assert_allclose(ds.reshape(B, H_), amax / 448.0, rtol=1e-5)
        codes = p[name]
        # each slice reaches the saturation code exactly once or more
        assert np.all((np.abs(table[codes]).reshape(B, H_, -1) == 448.0).any(-1))
        deq = _dequant(table, codes, ds, (B, H_))
        # E4M3 RNE: relative error <= 2^-4 for normals, absolute <= 2^-10 * scale in the subnormal range
        err = np.abs(deq - x)
        bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * ds.reshape(B, H_, 1, 1)) + 1e-6 * np.abs(x)
        assert np.all(err <= bound), name


def test_prepare_rejects_nonfinite(orc):
    q, k, v = synth.qkv_normal(1, 1, 1, 1, 32, 64)
    q[0, 0, 3, 5] = np.inf
    with pytest.raises(orc.OracleError) as e:
        orc.prepare(q, k, v)
    assert e.value.code == 4
    q[0, 0, 3, 5] = np.nan
    with pytest.raises(orc.OracleError):
        orc.prepare(q, k, v)


def test_prepare_zero_slice_gives_unit_scale(orc):
    q, k, v = synth.qkv_normal(1, 1, 1, 1, 16, 64)
    v[:] = 0
    p = orc.prepare(q, k, v)
    assert p["v_descale"][0] == 1.0 and np.all(p["v8"] == 0)


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_prepare_tile_scales(orc, flags):
    """Per-tile scales: every 128-row tile of Q and K has descale = its own amax / 448
    (amax from an independent float64 transform), reaches the saturation code, and
    reconstructs within the E4M3 bound of its own scale; V keeps one scale per slice."""
    B, Hq, Hkv, N, d, TS = 1, 2, 2, 300, 64, 128
    nt = (N + TS - 1) // TS
    qb, kb, vb = synth.qwen_like_inputs(61 + flags, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    signs = synth.hadamard_signs(78, d)
    p = orc.prepare(qb, kb, vb, flags=flags | orc.TILE_SCALES, signs=signs)
    slice_p = orc.prepare(qb, kb, vb, flags=flags, signs=signs)
    assert p["q_descale"].shape == (B * Hq * nt,) and p["k_descale"].shape == (B * Hkv * nt,)
    assert np.array_equal(p["v8"], slice_p["v8"]) and np.array_equal(p["v_descale"], slice_p["v_descale"])
    table = orc.e4m3_decode_table()
    q = synth.bf16_bits_to_f32(qb).astype(np.float64)
    k = synth.bf16_bits_to_f32(kb).astype(np.float64)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    if flags & 2:
        k = k - p["k_mean"].reshape(B, Hkv, 1, d).astype(np.float64)
    if flags & 1:
        q = (q * signs) @ H
        k = (k * signs) @ H
    for name, x, ds, H_ in (("q8", q, p["q_descale"], Hq), ("k8", k, p["k_descale"], Hkv)):
        ds = ds.reshape(B, H_, nt)
        codes = p[name]
        for t in range(nt):
            xt = x[:, :, t * TS:(t + 1) * TS]
            ct = codes[:, :, t * TS:(t + 1) * TS]
            amax = np.abs(xt).reshape(B, H_, -1).max(-1)
            np.testing.assert_allclose(ds[:, :, t], amax / 448.0, rtol=1e-5)
            assert np.all((np.abs(table[ct]).reshape(B, H_, -1) == 448.0).any(-1))
            deq = table[ct].astype(np.float64) * ds[:, :, t].reshape(B, H_, 1, 1).astype(np.float64)
            bound = np.maximum(np.abs(xt) * 2.0 ** -4, 2.0 ** -10 * ds[:, :, t].reshape(B, H_, 1, 1)) + 1e-6 * np.abs(xt)
            assert np.all(np.abs(deq - xt) <= bound), (name, t)


def test_tile_scales_reduce_to_slice_scales_when_tiles_share_amax(orc):
    """If every tile holds the slice's largest magnitude, the per-tile scales all equal
    the slice scale and the codes are those of the full-sequence scaling."""
    B, Hq, Hkv, N, d = 1, 2, 1, 384, 64
    q, k, v = synth.qkv_normal(62, B, Hq, Hkv, N, d)
    for x in (q, k):
        x /= np.abs(x).max() * 1.01  # |x| < 1
        x[:, :, ::128, 0] = 3.0     # one entry of 3 in every 128-row tile
    p = orc.prepare(q, k, v, flags=orc.TILE_SCALES)
    s = orc.prepare(q, k, v, flags=0)
    assert np.array_equal(p["q8"], s["q8"]) and np.array_equal(p["k8"], s["k8"])
    assert np.all(p["q_descale"].reshape(B * Hq, -1) == s["q_descale"][:, None])
    assert np.all(p["k_descale"].reshape(B * Hkv, -1) == s["k_descale"][:, None])
