"""Pins for the oracle's E4M3FN encode/decode.

Independent anchors: the format facts the pages print (tests/golden), PyTorch's
own float8_e4m3fn conversion (a separate implementation; it does not saturate,
so it is compared only where saturation cannot matter) and round-trip / tie
properties that follow from round-to-nearest-even.
"""
import numpy as np
import pytest
import torch

from tests.golden.pages import page_numbers

PAGE = page_numbers()


@pytest.fixture(scope="module")
def table(orc):
    return orc.e4m3_decode_table()


def test_decode_matches_torch(table):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(table))
    assert np.array_equal(ref[~nan], table[~nan])
    assert sorted(np.flatnonzero(nan).tolist()) == [0x7F, 0xFF]


def test_decode_page_facts(table):
    fin = table[np.isfinite(table)]
    assert fin.max() == PAGE["e4m3_max_finite"] and fin.min() == -PAGE["e4m3_max_finite"]
    assert not np.isinf(table).any()
    pos = table[:0x7F]
    assert np.all(np.diff(pos) > 0)                 # codes 0..0x7E ascend
    assert pos[1] == 2.0 ** -9                      # smallest subnormal
    assert pos[8] == PAGE["smallest_normal"]        # smallest normal is 2^-6
    assert np.array_equal(table[0x80:0xFF], -table[0:0x7F])
    assert len(np.unique(np.abs(fin))) == 127


def test_roundtrip_every_code(orc, table):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    vals = table[codes].astype(np.float32)
    vals[codes == 0x80] = np.float32(-0.0)
    assert np.array_equal(orc.e4m3_encode(vals), codes.astype(np.uint8))


def test_ties_to_even_and_neighbours(orc, table):
    pos = table[:0x7F]
    for k in range(126):
        mid = np.float32((pos[k] + pos[k + 1]) / 2)
        assert float(mid) == (pos[k] + pos[k + 1]) / 2      # midpoint is a float
        even = k if k % 2 == 0 else k + 1
        below = np.nextafter(mid, np.float32(-1))
        above = np.nextafter(mid, np.float32(1e9))
        got = orc.e4m3_encode(np.array([mid, below, above, -mid], dtype=np.float32))
        assert got.tolist() == [even, k, k + 1, 0x80 | even], k


def test_saturation_and_nan(orc):
    x = np.array([448, 460, 464, 470, 1e30, np.inf, -np.inf, -1e30, np.nan], dtype=np.float32)
    assert orc.e4m3_encode(x).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]


def test_round_to_zero_threshold(orc):
    t = np.float32(PAGE["round_to_zero_threshold"])
    assert t == np.float32(2.0 ** -10)
    x = np.array([t, np.nextafter(t, np.float32(1)), np.nextafter(t, np.float32(0)), -t, 1e-45, -0.0],
                 dtype=np.float32)
    assert orc.e4m3_encode(x).tolist() == [0x00, 0x01, 0x00, 0x80, 0x00, 0x80]


def test_encode_matches_torch_on_bit_pattern_sample(orc):
    """Every 61st float32 bit pattern, plus every pattern in the subnormal-to-
    normal region 2^-12 .. 2^-5, compared with PyTorch where |x| <= 464."""
    bits = np.arange(0, 1 << 32, 61, dtype=np.uint64).astype(np.uint32)
    lo = np.float32(2.0 ** -12).view(np.uint32)
    hi = np.float32(2.0 ** -5).view(np.uint32)
    dense = np.arange(lo, hi, dtype=np.uint32)
    bits = np.concatenate([bits, dense, dense | np.uint32(0x80000000)])
    x = bits.view(np.float32)
    keep = np.abs(x) <= 464
    x = x[keep]
    ours = orc.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.flatnonzero(ours != ref)
    assert bad.size == 0, (x[bad[:5]], ours[bad[:5]], ref[bad[:5]])


def test_encode_bits_range_matches_elementwise(orc):
    start = 0x3A7FFF00
    codes = orc.e4m3_encode_bits(start, 4096)
    x = np.arange(start, start + 4096, dtype=np.uint64).astype(np.uint32).view(np.float32)
    assert np.array_equal(codes, orc.e4m3_encode(x))
