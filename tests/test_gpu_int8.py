"""INT8-QK / FP8-PV (ATTNQ_I8QK) on the GPU against the oracle: prepare
bit-exact (INT8 Q/K codes held in bf16, their descales, E4M3 V) over ragged
lengths, both input types, both d, rotation and centring, per-tile scales and
causal-prefix statistics; the forward pass (S = Q K^T on the bf16 tensor path)
within the forward tolerance of the oracle's emulation with exact integer
q.k, underflow counts, and full-range codes whose dot products sit at
128 * 127^2."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

I8 = 16
TILE = 8


def _compare(q, k, v, flags, signs, P=0, vt=True):
    from tests.gpu_helpers import gpu_prepare, prepared_to_numpy
    desc, bufs, st = gpu_prepare(q, k, v, flags | I8, signs, vt=vt, stat_len=P)
    assert st == 0
    got = prepared_to_numpy(desc, bufs)
    ref = oracle.prepare(q, k, v, flags=flags | I8, signs=signs, stat_len=P)
    for name in ("q8", "k8", "v8"):
        assert np.array_equal(got[name], ref[name]), name
    for name in ("q_descale", "k_descale", "v_descale"):
        assert np.array_equal(got[name].view(np.uint32), ref[name].view(np.uint32)), name
    return desc, bufs


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("N,d,kind", [(1, 64, "bf16"), (129, 128, "bf16"), (300, 64, "f32"), (1000, 128, "bf16"),
                                      (2049, 128, "f32")])
def test_prepare_int8_bit_exact(flags, N, d, kind):
    B, Hq, Hkv = 1, 4, 2
    if kind == "bf16":
        q, k, v = synth.qwen_like_inputs(2000 + N + flags, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    else:
        q, k, v = synth.qkv_normal(2000 + N + flags, B, Hq, Hkv, N, d)
    _compare(q, k, v, flags, synth.hadamard_signs(98, d))


@pytest.mark.parametrize("flags", [0, 3])
@pytest.mark.parametrize("mode", ["tile", "prefix", "natural_v"])
def test_prepare_int8_with_other_options(flags, mode):
    B, Hq, Hkv, N, d = 2, 4, 2, 1000, 128
    q, k, v = synth.qwen_like_inputs(2100 + flags, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    signs = synth.hadamard_signs(99, d)
    if mode == "tile":
        _compare(q, k, v, flags | TILE, signs)
    elif mode == "prefix":
        _compare(q, k, v, flags, signs, P=300)
    else:
        _compare(q, k, v, flags, signs, vt=False)


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("d,T", [(128, 128), (128, 64), (64, 128), (64, 64)])
def test_fwd_int8_matches_oracle(order, d, T):
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, o_to_numpy, rel_f
    B, Hq, Hkv, N = 1, 4, 2, 1000
    q, k, v = synth.qwen_like_inputs(2200 + d + T + order, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    signs = synth.hadamard_signs(100, d)
    flags = 3
    desc, bufs = _compare(q, k, v, flags, signs)
    O, uf, st = gpu_fwd(desc, bufs, 256.0, order, True, T)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=flags | I8, signs=signs)
    ref, ufr = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags | I8, 256.0, order, True, T)
    assert rel_f(o_to_numpy(O).reshape(B * Hq, N, d), ref).max() <= REL_F_TOL
    tot, totr = uf.sum(axis=0).astype(np.int64), ufr.sum(axis=0).astype(np.int64)
    assert np.all(np.abs(tot - totr) <= 0.001 * totr + 2), (tot, totr)


@pytest.mark.parametrize("flags", [0, TILE])
def test_fwd_int8_tile_scales_and_bf16_output(flags):
    import torch
    from tests.gpu_helpers import gpu_fwd, o_to_numpy, oracle_bf16, rel_f
    B, Hq, Hkv, N, d, T = 2, 4, 2, 700, 128, 128
    q, k, v = synth.qwen_like_inputs(2300 + flags, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
    desc, bufs = _compare(q, k, v, flags, None)
    O, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, T, out_dtype=torch.bfloat16, count=False)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=flags | I8)
    ref, _ = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags | I8, 256.0, 1, True, T)
    assert rel_f(o_to_numpy(O).reshape(B * Hq, N, d), oracle_bf16(ref)).max() <= 1e-2


def test_fwd_int8_dot_products_are_exact_through_cancellation():
    """Scores that are small integers reached through partial sums near 10^6:
    q = (1, 127 x 64, -127 x 63) and key j = (j mod 128, 127 x 63, 0, 127 x 63)
    give q.k_j = j mod 128 exactly.  A tensor-core sum that dropped low bits at
    that magnitude would lose the first term and flatten the softmax weights
    2^(c j); the output must match the oracle's exact integer sums, and the
    flattened alternative must not."""
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, o_to_numpy, rel_f
    B, Hq, Hkv, N, d, T = 1, 2, 1, 256, 128, 128
    qrow = np.concatenate([[1.0], np.full(64, 127.0), np.full(63, -127.0)]).astype(np.float32)
    q = np.broadcast_to(qrow, (B, Hq, N, d)).copy()
    k = np.empty((B, Hkv, N, d), np.float32)
    k[..., 1:64] = 127.0
    k[..., 64] = 0.0
    k[..., 65:] = 127.0
    k[0, 0, :, 0] = np.arange(N) % 128
    v = synth.normals(2400, B * Hkv * N * d).reshape(B, Hkv, N, d)
    desc, bufs = _compare(q, k, v, 0, None)
    O, _, st = gpu_fwd(desc, bufs, 256.0, 0, True, T, count=False)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=I8)
    assert np.array_equal(prep["q8"][0, 0, 0], qrow.astype(np.int8))
    ref, _ = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), I8, 256.0, 0, True, T)
    got = o_to_numpy(O).reshape(B * Hq, N, d)
    assert rel_f(got, ref).max() <= REL_F_TOL
    flat = dict(prep)
    flat["k8"] = prep["k8"].copy()
    flat["k8"][..., 0] = 0  # every score 0: the sums without their small term
    ref_flat, _ = oracle.attn_quant(flat, (B, Hq, Hkv, N, d), I8, 256.0, 0, True, T)
    assert rel_f(ref_flat, ref).min() > 0.1


def test_int8_long_context_full_size_sampled():
    """The long-context workload at full size with INT8 Q/K: every operand byte and
    descale against the oracle, and sampled output rows within the forward tolerance."""
    import torch
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, oracle_bf16, rel_f
    wl = synth.WORKLOADS["long_context"]
    B, Hq, Hkv, N, d, T = wl["B"], wl["Hq"], wl["Hkv"], wl["N"], wl["d"], wl["kv_tile"]
    q, k, v = synth.long_context_inputs(5100, B, Hq, Hkv, N, d)
    signs = synth.hadamard_signs(17, d)
    flags = 3 | I8
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs)
    assert st == 0
    O, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, T, out_dtype=torch.bfloat16, count=False)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=flags, signs=signs)
    for name in ("q8", "k8"):
        # the codes are exact integers in bf16: compare their values
        assert torch.equal(getattr(bufs, name).float().cpu(), torch.from_numpy(prep[name]).float()), name
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


def test_int8_cast_of_every_finite_float():
    """With statistics from a first token whose amax is 127 the INT8 scale is 1,
    so later tokens reach the cast unscaled: every finite float32 (both signs)
    must give the oracle's code, nearest integer with ties to even, saturated."""
    import torch
    from tests.gpu_helpers import gpu_prepare
    d = 128
    hi = int(np.float32(np.finfo(np.float32).max).view(np.uint32))
    chunk = 1 << 26
    for start in range(0, hi + 1, chunk):
        n = min(chunk, hi + 1 - start)
        vals = np.arange(start, start + n, dtype=np.uint32).view(np.float32)
        rows = (n + d - 1) // d
        flat = np.zeros((1 + 2 * rows) * d, np.float32)
        flat[0] = 127.0  # the statistics token
        flat[d: d + n] = vals
        flat[(1 + rows) * d: (1 + rows) * d + n] = -vals
        q = flat.reshape(1, 1, 1 + 2 * rows, d)
        ones = np.ones_like(q)
        desc, bufs, status = gpu_prepare(q, ones, ones, I8, None, vt=False, stat_len=1)
        assert status == 0
        assert float(bufs.scales.q_descale[0]) == 1.0
        got = bufs.q8.to(torch.int8).cpu().numpy().reshape(-1)
        want = oracle.int8_encode(vals)
        assert np.array_equal(got[d: d + n], want), start
        assert np.array_equal(got[(1 + rows) * d: (1 + rows) * d + n], oracle.int8_encode(-vals)), start
