"""Per-tile Q/K scales (ATTNQ_TILE_SCALES) on the GPU against the oracle:
prepare bit-exact (codes and every tile's descale, ragged last tiles, with and
without rotation and centring, both input types), the forward pass within the
forward tolerance of the oracle's emulation with per-tile logit factors."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

TILE = 8


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("N,d,kind", [(1, 64, "bf16"), (129, 128, "bf16"), (300, 64, "f32"), (1000, 128, "bf16"),
                                      (2049, 128, "bf16")])
def test_prepare_tile_scales_bit_exact(flags, N, d, kind):
    from tests.gpu_helpers import gpu_prepare, prepared_to_numpy
    B, Hq, Hkv = 1, 4, 2
    if kind == "bf16":
        q, k, v = synth.qwen_like_inputs(900 + N + flags, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    else:
        q, k, v = synth.qkv_normal(900 + N + flags, B, Hq, Hkv, N, d)
    signs = synth.hadamard_signs(91, d)
    desc, bufs, st = gpu_prepare(q, k, v, flags | TILE, signs)
    assert st == 0
    got = prepared_to_numpy(desc, bufs)
    ref = oracle.prepare(q, k, v, flags=flags | TILE, signs=signs)
    for name in ("q8", "k8", "v8"):
        assert np.array_equal(got[name], ref[name]), name
    for name in ("q_descale", "k_descale", "v_descale"):
        assert np.array_equal(got[name].view(np.uint32), ref[name].view(np.uint32)), name
    assert np.all(got["v8_pad"] == 0)


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("T", [64, 128])
@pytest.mark.parametrize("N", [200, 1000])
def test_fwd_tile_scales_matches_oracle(order, T, N):
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, rel_f
    B, Hq, Hkv, d = 1, 4, 2, 128
    q, k, v = synth.qwen_like_inputs(950 + N, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    # tiles of very different magnitude, so their scales differ
    for x in (q, k):
        f = synth.bf16_bits_to_f32(x)
        f[:, :, 128:256] *= 16.0
        x[...] = oracle.round_bf16(f.astype(np.float64))
    signs = synth.hadamard_signs(92, d)
    flags = 3 | TILE
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs)
    assert st == 0
    O, uf, st = gpu_fwd(desc, bufs, 256.0, order, True, T)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=flags, signs=signs)
    ref, ufr = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags, 256.0, order, True, T)
    assert rel_f(o_to_numpy(O).reshape(B * Hq, N, d), ref).max() <= REL_F_TOL
    tot, totr = uf.sum(axis=0).astype(np.int64), ufr.sum(axis=0).astype(np.int64)
    assert np.all(np.abs(tot - totr) <= 0.001 * totr + 2), (tot, totr)


@pytest.mark.parametrize("i8", [False, True])
@pytest.mark.parametrize("T", [64, 128])
def test_tile_instance_with_equal_tile_scales_equals_slice_instance(i8, T):
    """Per-tile logit factors reduce to the per-slice one when every tile
    carries the slice's descale: the per-tile forward then gives the slice
    forward's output bit for bit."""
    import torch
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import gpu_fwd, gpu_prepare
    B, Hq, Hkv, N, d = 1, 4, 2, 1000, 128
    q, k, v = synth.qwen_like_inputs(990 + T + i8, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    signs = synth.hadamard_signs(93, d)
    flags = 3 | (aq.ATTNQ_I8QK if i8 else 0)
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs)
    assert st == 0
    O1, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, T, out_dtype=torch.float32, count=False)
    assert st == 0
    nt = aq.attnq_scale_tiles(N)
    tdesc = aq.AttnqDesc(B, Hq, Hkv, N, d, desc.in_dtype, desc.flags | TILE, desc.signs)
    bufs.scales = aq.AttnqScales(bufs.scales.q_descale.repeat_interleave(nt),
                                 bufs.scales.k_descale.repeat_interleave(nt), bufs.scales.v_descale, None)
    O2, _, st = gpu_fwd(tdesc, bufs, 256.0, 1, True, T, out_dtype=torch.float32, count=False)
    assert st == 0
    assert torch.equal(O1, O2)


def test_tile_scales_long_context_full_size_sampled():
    """The long-context workload at full size with per-tile Q/K scales (the
    shape runs the attention kernel's mirrored-pair schedule): every code and
    descale against the oracle, and sampled output rows within the forward
    tolerance."""
    import torch
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, oracle_bf16, rel_f
    wl = synth.WORKLOADS["long_context"]
    B, Hq, Hkv, N, d, T = wl["B"], wl["Hq"], wl["Hkv"], wl["N"], wl["d"], wl["kv_tile"]
    q, k, v = synth.long_context_inputs(5200, B, Hq, Hkv, N, d)
    signs = synth.hadamard_signs(17, d)
    flags = 3 | TILE
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs)
    assert st == 0
    O, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, T, out_dtype=torch.bfloat16, count=False)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=flags, signs=signs)
    assert torch.equal(bufs.q8.cpu(), torch.from_numpy(prep["q8"]))
    assert torch.equal(bufs.k8.cpu(), torch.from_numpy(prep["k8"]))
    v8 = bufs.v8[..., :N].transpose(-1, -2).contiguous().cpu()
    assert torch.equal(v8, torch.from_numpy(prep["v8"]))
    for key, t in (("q_descale", bufs.scales.q_descale), ("k_descale", bufs.scales.k_descale),
                   ("v_descale", bufs.scales.v_descale), ("k_mean", bufs.scales.k_mean)):
        assert np.array_equal(t.cpu().numpy().view(np.uint32), prep[key].view(np.uint32)), key
    rows = np.array([0, 1, 127, 128, 4095, 16383, 16384, 24577, 32640, 32767], dtype=np.int32)
    bh = [0, 5, 31, 32, 63]
    emu, _ = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags, 256.0, 1, True, T, bh_list=bh, rows=rows)
    got = o_to_numpy(O).reshape(B * Hq, N, d)[bh][:, rows]
    assert rel_f(got, oracle_bf16(emu)).max() <= REL_F_TOL
