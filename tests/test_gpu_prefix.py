"""Causal-prefix statistics (desc.stat_len = P) on the GPU against the oracle:
prepare bit-exact for prefixes that end inside a tile, on a tile edge, inside
and after the first 16-tile item, with every combination of rotation and
centring, both input types, both d, both V layouts and per-tile Q/K scales;
non-finite values after the prefix still reported; the forward pass on
prefix-scaled operands within the forward tolerance of the oracle."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

TILE = 8


def _inputs(seed, B, Hq, Hkv, N, d, kind, P):
    if kind == "bf16":
        q, k, v = synth.qwen_like_inputs(seed, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    else:
        q, k, v = synth.qkv_normal(seed, B, Hq, Hkv, N, d)
    # later tokens larger than the prefix's, so some of them saturate
    for x in (q, k, v):
        f = synth.bf16_bits_to_f32(x) if kind == "bf16" else x
        f[:, :, P:] *= 3.0
        if kind == "bf16":
            x[...] = oracle.round_bf16(f.astype(np.float64))
    return q, k, v


def _compare(q, k, v, flags, signs, P, vt=True):
    from tests.gpu_helpers import gpu_prepare, prepared_to_numpy
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs, vt=vt, stat_len=P)
    assert st == 0
    got = prepared_to_numpy(desc, bufs)
    ref = oracle.prepare(q, k, v, flags=flags, signs=signs, stat_len=P)
    for name in ("q8", "k8", "v8"):
        assert np.array_equal(got[name], ref[name]), name
    for name in ("q_descale", "k_descale", "v_descale"):
        assert np.array_equal(got[name].view(np.uint32), ref[name].view(np.uint32)), name
    if flags & 2:
        assert np.array_equal(got["k_mean"].view(np.uint32), ref["k_mean"].view(np.uint32))
    if vt:
        assert np.all(got["v8_pad"] == 0)


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("N,P", [(1, 1), (300, 1), (300, 127), (300, 128), (300, 129), (300, 299),
                                 (4500, 2048), (4500, 2049), (4500, 4499), (4500, 4500)])
def test_prepare_prefix_bit_exact(flags, N, P):
    B, Hq, Hkv, d = 1, 4, 2, 128
    q, k, v = _inputs(1200 + N + P + flags, B, Hq, Hkv, N, d, "bf16", P)
    _compare(q, k, v, flags, synth.hadamard_signs(93, d), P)


@pytest.mark.parametrize("flags", [0, 3])
@pytest.mark.parametrize("d,kind,vt", [(64, "bf16", True), (64, "f32", False), (128, "f32", True),
                                       (128, "bf16", False)])
def test_prepare_prefix_types_and_layouts(flags, d, kind, vt):
    B, Hq, Hkv, N, P = 2, 4, 2, 1000, 333
    q, k, v = _inputs(1300 + d + flags, B, Hq, Hkv, N, d, kind, P)
    _compare(q, k, v, flags, synth.hadamard_signs(94, d), P, vt=vt)


@pytest.mark.parametrize("flags", [0, 2, 3])
@pytest.mark.parametrize("P", [1, 200, 2176])
def test_prepare_prefix_with_tile_scales(flags, P):
    B, Hq, Hkv, N, d = 1, 4, 2, 2500, 128
    q, k, v = _inputs(1400 + P + flags, B, Hq, Hkv, N, d, "bf16", P)
    _compare(q, k, v, flags | TILE, synth.hadamard_signs(95, d), P)


def test_prepare_prefix_reports_nonfinite_after_the_prefix():
    from tests.gpu_helpers import gpu_prepare
    B, Hq, Hkv, N, d, P = 1, 2, 1, 700, 64, 130
    for flags, bad in ((0, np.inf), (3, np.nan), (3, -np.inf)):
        q, k, v = synth.qkv_normal(1500, B, Hq, Hkv, N, d)
        v[0, 0, 600, 7] = bad
        _, _, st = gpu_prepare(q, k, v, flags, synth.hadamard_signs(96, d), stat_len=P)
        assert st == 4, (flags, bad)
        q[0, 1, 140, 3] = bad
        v[0, 0, 600, 7] = 0.0
        _, _, st = gpu_prepare(q, k, v, flags, synth.hadamard_signs(96, d), stat_len=P)
        assert st == 4, (flags, bad)
    q, k, v = synth.qkv_normal(1501, B, Hq, Hkv, N, d)
    _, _, st = gpu_prepare(q, k, v, 3, synth.hadamard_signs(96, d), stat_len=P)
    assert st == 0


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("flags", [3, 3 | TILE])
def test_fwd_on_prefix_statistics_matches_oracle(order, flags):
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, rel_f
    B, Hq, Hkv, N, d, P, T = 1, 4, 2, 1000, 128, 256, 128
    q, k, v = _inputs(1600 + order + flags, B, Hq, Hkv, N, d, "bf16", P)
    signs = synth.hadamard_signs(97, d)
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs, stat_len=P)
    assert st == 0
    O, uf, st = gpu_fwd(desc, bufs, 256.0, order, True, T)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=flags, signs=signs, stat_len=P)
    ref, ufr = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags, 256.0, order, True, T)
    assert rel_f(o_to_numpy(O).reshape(B * Hq, N, d), ref).max() <= REL_F_TOL
    tot, totr = uf.sum(axis=0).astype(np.int64), ufr.sum(axis=0).astype(np.int64)
    assert np.all(np.abs(tot - totr) <= 0.001 * totr + 2), (tot, totr)


def test_prefix_long_context_full_size_sampled():
    """The long-context workload at full size with statistics from a 4096-token
    prompt: every operand byte, descale and the mean key against the oracle, and
    sampled output rows within the forward tolerance."""
    import torch
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, oracle_bf16, rel_f
    wl = synth.WORKLOADS["long_context"]
    B, Hq, Hkv, N, d, T = wl["B"], wl["Hq"], wl["Hkv"], wl["N"], wl["d"], wl["kv_tile"]
    P = 4096
    q, k, v = synth.long_context_inputs(5200, B, Hq, Hkv, N, d)
    signs = synth.hadamard_signs(17, d)
    flags = aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs, stat_len=P)
    assert st == 0
    O, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, T, out_dtype=torch.bfloat16, count=False)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=flags, signs=signs, stat_len=P)
    assert torch.equal(bufs.q8.cpu(), torch.from_numpy(prep["q8"]))
    assert torch.equal(bufs.k8.cpu(), torch.from_numpy(prep["k8"]))
    v8 = bufs.v8[..., :N].transpose(-1, -2).contiguous().cpu()
    assert torch.equal(v8, torch.from_numpy(prep["v8"]))
    for key, t in (("q_descale", bufs.scales.q_descale), ("k_descale", bufs.scales.k_descale),
                   ("v_descale", bufs.scales.v_descale), ("k_mean", bufs.scales.k_mean)):
        assert np.array_equal(t.cpu().numpy().view(np.uint32), prep[key].view(np.uint32)), key
    rows = np.array([0, 1, 127, 4095, 4096, 16384, 24577, 32767], dtype=np.int32)
    bh = [0, 7, 40, 63]
    emu, _ = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags, 256.0, 1, True, T, bh_list=bh, rows=rows)
    got = o_to_numpy(O).reshape(B * Hq, N, d)[bh][:, rows]
    assert rel_f(got, oracle_bf16(emu)).max() <= REL_F_TOL
