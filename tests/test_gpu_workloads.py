"""The pages' workloads (synthetic stand-ins) end to end on the GPU, checked
against the oracle:

* one layer of each Qwen-shaped workload in all four conditions (unrotated,
  rotated, centred, centred + rotated): forward parity with the quantised
  emulation (rel-F <= 2e-3) and each head's log1p error against FP64 within
  5% of the oracle's (attnq_err with the oracle's exact attention as O_ref);
* the P-cast sweep at its full size (N = 4096, 8 heads, P-only mode) for all
  six (order, S) pairs at delta in {0, 4, 7, 10, 12}: outputs within rel-F
  2e-3 of the oracle and underflow counts within 0.1% + 2;
* every layer of both Qwen-shaped workloads (24 and 28) in all four
  conditions (marked slow: about five minutes of oracle time);
* the long-context workload at full size in the configuration bench.py times
  (B=2, Hq=32, Hkv=8, N=32768, d=128, rotation + centring, reverse, S=256,
  bf16 output): every E4M3 operand byte, descale and mean-key value, and the
  outputs of sampled rows of sampled heads;
* a shape on the attention kernel's mirrored-pair schedule with an odd GQA
  group, 64-key tiles, forward order and ragged N (sampled rows).
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

CONDS = list(synth.CONDITIONS.items())


def _flags(rotate, center):
    return (1 if rotate else 0) | (2 if center else 0)


def _qwen_layer_all_conditions(name, layer):
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import ERR_REL_TOL, REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, rel_f
    wl = synth.WORKLOADS[name]
    B, Hq, Hkv, N, d, T = wl["B"], wl["Hq"], wl["Hkv"], wl["N"], wl["d"], wl["kv_tile"]
    q, k, v = synth.qwen_layer_inputs(name, layer)
    signs = synth.qwen_signs(name)
    exact = oracle.attn_exact(q, k, v)
    Oref = torch.from_numpy(exact.reshape(B, Hq, N, d)).cuda()
    errs = {}
    for cond, (rot, cen) in CONDS:
        flags = _flags(rot, cen)
        desc, bufs, st = gpu_prepare(q, k, v, flags, signs)
        assert st == 0
        O, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, T, count=False)
        assert st == 0
        prep = oracle.prepare(q, k, v, flags=flags, signs=signs)
        emu, _ = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags, 256.0, 1, True, T)
        got = o_to_numpy(O).reshape(B * Hq, N, d)
        assert rel_f(got, emu).max() <= REL_F_TOL, cond
        err = torch.empty(B * Hq, dtype=torch.float64, device="cuda")
        aq.attnq_err(desc, O, Oref, err)
        e_gpu = err.cpu().numpy()
        e_orc = oracle.err(emu, exact)
        assert np.all(np.abs(e_gpu - e_orc) <= ERR_REL_TOL * e_orc), (cond, e_gpu, e_orc)
        errs[cond] = e_gpu.reshape(B, Hq).mean(axis=0)    # mean over the "texts" (batch)
    # the harm score of every head is defined and finite
    harm = errs["rotated"] - errs["unrotated"]
    assert np.all(np.isfinite(harm))


@pytest.mark.parametrize("name", ["qwen05b", "qwen15b"])
def test_qwen_shaped_layer_all_conditions(name):
    _qwen_layer_all_conditions(name, 0)


@pytest.mark.slow
@pytest.mark.parametrize("name,layer", [("qwen05b", x) for x in range(1, synth.WORKLOADS["qwen05b"]["layers"])]
                         + [("qwen15b", x) for x in range(1, synth.WORKLOADS["qwen15b"]["layers"])])
def test_qwen_shaped_every_layer(name, layer):
    """Layers 1.. of both Qwen-shaped workloads (layer 0 is the test above)."""
    _qwen_layer_all_conditions(name, layer)


@pytest.mark.parametrize("delta", [0.0, 4.0, 7.0, 10.0, 12.0])
@pytest.mark.parametrize("order,S", [(0, 1.0), (0, 256.0), (0, 448.0), (1, 1.0), (1, 256.0), (1, 448.0)])
def test_pcast_sweep_full_size(order, S, delta):
    from tests.gpu_helpers import rel_f
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import dev
    wl = synth.WORKLOADS["pcast_sweep"]
    B, H, N, d, T = wl["B"], wl["Hq"], wl["N"], wl["d"], wl["kv_tile"]
    q, k, v = synth.pcast_sweep_inputs(delta)
    desc = aq.AttnqDesc(B, H, H, N, d, aq.ATTNQ_F32, 0, None)
    O = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    uf = torch.zeros(B * H * 2, dtype=torch.int64, device="cuda")
    aq.attnq_fwd_ponly(desc, dev(q), dev(k), dev(v), S, order, True, T, O, uf)
    assert aq.attnq_device_status() == 0
    got = O.cpu().numpy().astype(np.float64).reshape(B * H, N, d)
    ref, uref = oracle.attn_ponly(q, k, v, S, order, True, T)
    assert rel_f(got, ref).max() <= 2e-3
    u = uf.cpu().numpy().reshape(-1, 2)
    assert np.all(np.abs(u - uref.astype(np.int64)) <= 0.001 * uref + 2)


def test_long_context_full_size_sampled():
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, oracle_bf16, rel_f
    wl = synth.WORKLOADS["long_context"]
    B, Hq, Hkv, N, d, T = wl["B"], wl["Hq"], wl["Hkv"], wl["N"], wl["d"], wl["kv_tile"]
    q, k, v = synth.long_context_inputs(5000, B, Hq, Hkv, N, d)
    signs = synth.hadamard_signs(17, d)
    flags = aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs)
    assert st == 0
    O, _, st = gpu_fwd(desc, bufs, 256.0, 1, True, T, out_dtype=torch.bfloat16, count=False)
    assert st == 0
    # operands: every byte
    prep = oracle.prepare(q, k, v, flags=flags, signs=signs)
    assert torch.equal(bufs.q8.cpu(), torch.from_numpy(prep["q8"]))
    assert torch.equal(bufs.k8.cpu(), torch.from_numpy(prep["k8"]))
    v8 = bufs.v8[..., :N].transpose(-1, -2).contiguous().cpu()
    assert torch.equal(v8, torch.from_numpy(prep["v8"]))
    for key, t in (("q_descale", bufs.scales.q_descale), ("k_descale", bufs.scales.k_descale),
                   ("v_descale", bufs.scales.v_descale), ("k_mean", bufs.scales.k_mean)):
        assert np.array_equal(t.cpu().numpy().view(np.uint32), prep[key].view(np.uint32)), key
    # outputs of sampled rows (first tile, tile edges, middle, the longest rows)
    rows = np.array([0, 1, 127, 128, 4095, 16383, 16384, 24577, 32640, 32767], dtype=np.int32)
    bh = [0, 5, 31, 32, 63]
    emu, _ = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags, 256.0, 1, True, T, bh_list=bh, rows=rows)
    got = o_to_numpy(O).reshape(B * Hq, N, d)[bh][:, rows]
    assert rel_f(got, oracle_bf16(emu)).max() <= REL_F_TOL


def test_mirrored_pair_schedule_sampled():
    """A shape whose unit count puts the attention kernel on its mirrored-pair
    schedule on a 152-SM GPU (causal, 380 query tiles: 760 items of two
    mirrored query tiles, five full rounds), with the cases that schedule must
    still get right: a GQA group of three query heads (its second pair has one
    head), 64-key tiles, forward KV order, ragged N.  Every operand byte
    against the oracle, and the outputs of sampled rows (both ends of the
    sequence, the mirrored tiles' edges, the ragged tail)."""
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import REL_F_TOL, gpu_fwd, gpu_prepare, o_to_numpy, oracle_bf16, rel_f
    B, Hq, Hkv, d, T = 1, 6, 2, 64, 64
    N = 380 * 128 - 37
    q, k, v = synth.long_context_inputs(5101, B, Hq, Hkv, N, d)
    signs = synth.hadamard_signs(5102, d)
    flags = aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K
    desc, bufs, st = gpu_prepare(q, k, v, flags, signs)
    assert st == 0
    O, _, st = gpu_fwd(desc, bufs, 448.0, 0, True, T, out_dtype=torch.bfloat16, count=False)
    assert st == 0
    prep = oracle.prepare(q, k, v, flags=flags, signs=signs)
    assert torch.equal(bufs.q8.cpu(), torch.from_numpy(prep["q8"]))
    assert torch.equal(bufs.k8.cpu(), torch.from_numpy(prep["k8"]))
    v8 = bufs.v8[..., :N].transpose(-1, -2).contiguous().cpu()
    assert torch.equal(v8, torch.from_numpy(prep["v8"]))
    rows = np.array([0, 127, 128, 255, 24191, 24192, 48255, 48256, 48500, N - 1], dtype=np.int32)
    bh = [0, 2, 3, 5]
    emu, _ = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags, 448.0, 0, True, T, bh_list=bh, rows=rows)
    got = o_to_numpy(O).reshape(B * Hq, N, d)[bh][:, rows]
    assert rel_f(got, oracle_bf16(emu)).max() <= REL_F_TOL
