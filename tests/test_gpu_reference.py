"""The FP64 reference attention and the batched four-condition report on the
GPU, against the oracle: the reference equals the oracle's exact attention
(two-pass, double) up to double rounding; the report's per-head errors equal
the oracle's quantised emulation measured against its exact attention, per
condition, within the forward pass's error bar."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

# double rounding of sums of at most N*d terms, relative to the output norm
REF_TOL = 1e-12


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,kind", [
    (1, 2, 1, 1, 64, True, "bf16"),
    (1, 3, 1, 77, 64, True, "bf16"),
    (2, 4, 2, 300, 128, True, "bf16"),
    (1, 2, 2, 257, 128, False, "f32"),
    (1, 6, 3, 129, 64, True, "f32"),
])
def test_reference_attention_matches_oracle(B, Hq, Hkv, N, d, causal, kind):
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import dev
    if kind == "bf16":
        q, k, v = synth.qwen_like_inputs(400 + N, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
        dt = aq.ATTNQ_BF16
    else:
        q, k, v = synth.sink_inputs(400 + N, B, Hq, N, d, delta=6.0)
        k, v = k[:, :Hkv], v[:, :Hkv]
        dt = aq.ATTNQ_F32
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, dt, 0, None)
    O = torch.empty((B, Hq, N, d), dtype=torch.float64, device="cuda")
    aq.attnq_ref_attention(desc, dev(q), dev(k), dev(v), causal, O)
    assert aq.attnq_device_status() == 0
    ref = oracle.attn_exact(q, k, v, causal=causal).reshape(B, Hq, N, d)
    got = O.cpu().numpy()
    err = np.linalg.norm((got - ref).reshape(B * Hq, -1), axis=1) / np.linalg.norm(ref.reshape(B * Hq, -1), axis=1)
    assert err.max() <= REF_TOL, err


def test_harm_report_matches_oracle_pipeline():
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import ERR_REL_TOL, dev
    wl = synth.WORKLOADS["qwen05b"]
    B, Hq, Hkv, N, d, T = wl["B"], wl["Hq"], wl["Hkv"], 512, wl["d"], wl["kv_tile"]
    q, k, v = synth.qwen_like_inputs(4100, B, Hq, Hkv, N, d, key_norm=wl["key_norm"],
                                     key_channels=wl["key_channels"])
    signs = synth.hadamard_signs(4101, d)
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16, 0, torch.from_numpy(signs).cuda())
    ws = torch.empty(aq.attnq_harm_workspace(desc), dtype=torch.uint8, device="cuda")
    err = torch.empty((4, B * Hq), dtype=torch.float64, device="cuda")
    aq.attnq_harm_report(desc, dev(q), dev(k), dev(v), 256.0, aq.ATTNQ_KV_REVERSE, T, ws, err)
    assert aq.attnq_device_status() == 0
    got = err.cpu().numpy()
    exact = oracle.attn_exact(q, k, v)
    for c, flags in enumerate((0, 1, 2, 3)):
        prep = oracle.prepare(q, k, v, flags=flags, signs=signs)
        emu, _ = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), flags, 256.0, 1, True, T)
        want = oracle.err(emu, exact)
        assert np.all(np.abs(got[c] - want) <= ERR_REL_TOL * want), (c, got[c], want)
    harm = (got[1] - got[0]).reshape(B, Hq).mean(axis=0)
    assert np.all(np.isfinite(harm))


def test_harm_report_rejects_missing_signs():
    import precision_attention_numerics_gb300 as aq
    desc = aq.AttnqDesc(1, 2, 1, 64, 64, aq.ATTNQ_BF16, 0, None)
    x = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(aq.attnq_harm_workspace(desc), dtype=torch.uint8, device="cuda")
    err = torch.empty((4, 2), dtype=torch.float64, device="cuda")
    with pytest.raises(aq.AttnqError) as e:
        aq.attnq_harm_report(desc, x, x[:, :1], x[:, :1], 256.0, 1, 128, ws, err)
    assert e.value.code == 1
