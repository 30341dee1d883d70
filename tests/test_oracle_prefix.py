"""Pins for the oracle's causal-prefix statistics (stat_len = P).

The "attention-numerics" page (limitations) notes that full-sequence means and
scales see future tokens.  The reading pinned here: the mean key and the
per-(batch, head) amax come from the first P tokens of each slice, every token
is centred and cast with them, and later values above the prefix amax
saturate at +-448.

Anchors: the full-sequence oracle on the truncated input (pinned in
test_oracle_prepare.py), numpy float32 arithmetic on integer-valued inputs
(every sum exact, one IEEE division), the saturation rule of the cast, and
row copies that must give identical codes.
"""
import numpy as np
import pytest

import synth


def _qkv(seed, B, Hq, Hkv, N, d):
    return synth.qwen_like_inputs(seed, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("P", [1, 77, 128, 200])
def test_prefix_statistics_equal_full_sequence_on_truncated_input(orc, flags, P):
    """The first P rows' codes, the descales and the mean key equal those of the
    full-sequence preparation of the first P tokens alone."""
    B, Hq, Hkv, N, d = 1, 2, 1, 300, 64
    qb, kb, vb = _qkv(40 + flags, B, Hq, Hkv, N, d)
    signs = synth.hadamard_signs(41, d)
    p = orc.prepare(qb, kb, vb, flags=flags, signs=signs, stat_len=P)
    t = orc.prepare(qb[:, :, :P], kb[:, :, :P], vb[:, :, :P], flags=flags, signs=signs)
    for name in ("q8", "k8", "v8"):
        assert np.array_equal(p[name][:, :, :P], t[name]), name
    for name in ("q_descale", "k_descale", "v_descale", "k_mean"):
        assert np.array_equal(p[name].view(np.uint32), t[name].view(np.uint32)), name


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_prefix_equal_to_n_is_the_full_sequence_preparation(orc, flags):
    B, Hq, Hkv, N, d = 1, 2, 1, 150, 64
    qb, kb, vb = _qkv(42 + flags, B, Hq, Hkv, N, d)
    signs = synth.hadamard_signs(43, d)
    full = orc.prepare(qb, kb, vb, flags=flags, signs=signs)
    for P in (0, N):
        p = orc.prepare(qb, kb, vb, flags=flags, signs=signs, stat_len=P)
        for name in full:
            assert np.array_equal(p[name].view(np.uint8), full[name].view(np.uint8)), (P, name)


def test_prefix_mean_and_scale_closed_form_on_integer_inputs(orc):
    """Integer-valued inputs keep every partial sum exact, so the mean is
    fl32(sum / P) and the V descale fl32(max |v| / 448), both over the first P
    tokens (numpy float32 division is the IEEE one)."""
    B, Hq, Hkv, N, d, P = 1, 2, 2, 333, 64, 129
    q = (synth.splitmix64(50, B * Hq * N * d) % np.uint64(17)).astype(np.float32).reshape(B, Hq, N, d) - 8
    k = (synth.splitmix64(51, B * Hkv * N * d) % np.uint64(64)).astype(np.float32).reshape(B, Hkv, N, d)
    v = (synth.splitmix64(52, B * Hkv * N * d) % np.uint64(201)).astype(np.float32).reshape(B, Hkv, N, d) - 100
    k[:, :, P:] += 1000.0   # later keys far from the prefix mean
    v[:, :, P + 5, 3] = 5000.0   # a later value far above the prefix amax
    p = orc.prepare(q, k, v, flags=orc.CENTER_K, stat_len=P)
    mu = k[:, :, :P].astype(np.float64).sum(axis=2).astype(np.float32) / np.float32(P)
    assert np.array_equal(p["k_mean"].reshape(B, Hkv, d), mu)
    amax_v = np.abs(v[:, :, :P]).reshape(B * Hkv, -1).max(-1)
    assert np.array_equal(p["v_descale"], amax_v / np.float32(448))
    amax_q = np.abs(q[:, :, :P]).reshape(B * Hq, -1).max(-1)
    assert np.array_equal(p["q_descale"], amax_q / np.float32(448))
    # the centred K amax is over the prefix too: |k - mu| <= 63 there, not ~1000
    kc = k[:, :, :P] - mu[:, :, None, :]
    amax_k = np.abs(kc).reshape(B * Hkv, -1).max(-1)
    assert np.array_equal(p["k_descale"], amax_k / np.float32(448))


@pytest.mark.parametrize("flags", [0, 1])
def test_later_values_above_the_prefix_amax_saturate(orc, flags):
    """Rows after the prefix scaled up by 4: where fl32(x * qs) exceeds 448 the
    code is +-448 with the sign of x; elsewhere it is the cast of fl32(x * qs)."""
    B, Hq, Hkv, N, d, P = 1, 1, 1, 256, 64, 128
    q, k, v = synth.qkv_normal(53, B, Hq, Hkv, N, d)
    for x in (q, k, v):
        x[:, :, P:] = x[:, :, :P] * np.float32(4.0)
    signs = synth.hadamard_signs(54, d)
    p = orc.prepare(q, k, v, flags=flags, signs=signs, stat_len=P)
    table = orc.e4m3_decode_table()
    for name, x, ds in (("q8", q, p["q_descale"]), ("k8", k, p["k_descale"]), ("v8", v, p["v_descale"])):
        x = x[0, 0]
        if flags & orc.ROTATE and name != "v8":
            x = orc.fwht(x * signs.astype(np.float32))
        amax = np.abs(x[:P]).max()
        qs = np.float32(448) / amax
        assert ds[0] == amax / np.float32(448)
        y = (x * qs).astype(np.float32)
        codes = p[name][0, 0]
        sat = np.abs(y) > 448
        assert sat[P:].sum() > sat[:P].sum()  # the prefix amax itself may round just above 448
        assert np.array_equal(table[codes[sat]], np.where(y[sat] > 0, 448.0, -448.0))
        assert np.array_equal(codes[~sat], orc.e4m3_encode(y[~sat]))


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_copied_rows_after_the_prefix_get_the_same_codes(orc, flags):
    """Statistics fixed by the prefix: a later token that repeats an earlier
    one is centred, rotated and cast exactly like it."""
    B, Hq, Hkv, N, d, P = 1, 2, 1, 260, 64, 130
    qb, kb, vb = _qkv(55 + flags, B, Hq, Hkv, N, d)
    for x in (qb, kb, vb):
        x[:, :, P:2 * P] = x[:, :, :P]
    signs = synth.hadamard_signs(56, d)
    p = orc.prepare(qb, kb, vb, flags=flags, signs=signs, stat_len=P)
    for name in ("q8", "k8", "v8"):
        assert np.array_equal(p[name][:, :, P:2 * P], p[name][:, :, :P]), name


def test_prefix_with_tile_scales_changes_only_v_scale_and_mean(orc):
    """Per-tile Q/K scales are local to their tile; the prefix sets the V scale and
    the mean key.  With P a multiple of the tile, the prefix tiles' Q/K descales and
    codes equal those of the truncated input."""
    B, Hq, Hkv, N, d, P = 1, 2, 2, 300, 64, 128
    qb, kb, vb = _qkv(57, B, Hq, Hkv, N, d)
    signs = synth.hadamard_signs(58, d)
    flags = orc.TILE_SCALES | orc.CENTER_K | orc.ROTATE
    p = orc.prepare(qb, kb, vb, flags=flags, signs=signs, stat_len=P)
    t = orc.prepare(qb[:, :, :P], kb[:, :, :P], vb[:, :, :P], flags=flags, signs=signs)
    nt = 3
    assert np.array_equal(p["q_descale"].reshape(-1, nt)[:, 0], t["q_descale"])
    assert np.array_equal(p["k_descale"].reshape(-1, nt)[:, 0], t["k_descale"])
    assert np.array_equal(p["v_descale"], t["v_descale"]) and np.array_equal(p["k_mean"], t["k_mean"])
    for name in ("q8", "k8", "v8"):
        assert np.array_equal(p[name][:, :, :P], t[name]), name
    # Q does not depend on the prefix at all under per-tile scales
    f = orc.prepare(qb, kb, vb, flags=flags, signs=signs)
    assert np.array_equal(p["q8"], f["q8"]) and np.array_equal(p["q_descale"], f["q_descale"])


def test_prefix_arguments_checked(orc):
    q, k, v = synth.qkv_normal(59, 1, 1, 1, 40, 64)
    for bad in (-1, 41):
        with pytest.raises(orc.OracleError) as e:
            orc.prepare(q, k, v, stat_len=bad)
        assert e.value.code == 1
    # a non-finite value after the prefix is still reported
    q[0, 0, 30, 2] = np.inf
    with pytest.raises(orc.OracleError) as e:
        orc.prepare(q, k, v, stat_len=10)
    assert e.value.code == 4
