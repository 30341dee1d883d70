"""The host-buffer pipeline (attnq_attention_host): several steps of
prepare + attention whose inputs and outputs live in pinned host memory, with
the copies overlapping the kernels.  Each step's output must equal, bit for
bit, the device path (attnq_prepare + attnq_fwd) on the same inputs: the
pipeline only moves data, the kernels are the same deterministic launches."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _pipeline_vs_device(steps, N, out_bf16, extra_flags=0, stat_len=0):
    import precision_attention_numerics_gb300 as aq
    B, Hq, Hkv, d, T = 1, 4, 2, 128, 128
    flags = aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K | aq.ATTNQ_VT_LAYOUT | extra_flags
    signs = torch.from_numpy(synth.hadamard_signs(21, d)).cuda()
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16, flags, signs, stat_len)
    odt = aq.ATTNQ_BF16 if out_bf16 else aq.ATTNQ_F32
    tdt = torch.bfloat16 if out_bf16 else torch.float32
    hosts = []
    for i in range(steps):
        q, k, v = synth.qwen_like_inputs(700 + i, B, Hq, Hkv, N, d, key_norm=30.0, key_channels=4)
        hosts.append(tuple(torch.from_numpy(x).view(torch.bfloat16).pin_memory() for x in (q, k, v)))
    outs = [torch.full((B, Hq, N, d), float("nan"), dtype=tdt).pin_memory() for _ in range(steps)]
    ws = torch.empty(aq.attnq_host_pipeline_workspace(desc, odt), dtype=torch.uint8, device="cuda")
    compute, cin, cout = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    aq.attnq_attention_host(desc, [h[0] for h in hosts], [h[1] for h in hosts], [h[2] for h in hosts], 256.0,
                            aq.ATTNQ_KV_REVERSE, True, T, outs, odt, ws, compute, cin, cout)
    compute.synchronize()
    assert aq.attnq_device_status(compute.cuda_stream) == 0
    bufs = aq.alloc_prepared(desc)
    for i in range(steps):
        Q, K, V = (x.cuda() for x in hosts[i])
        O = torch.empty((B, Hq, N, d), dtype=tdt, device="cuda")
        aq.attnq_prepare(desc, Q, K, V, bufs.q8, bufs.k8, bufs.v8, bufs.scales, bufs.workspace)
        aq.attnq_fwd(desc, bufs.q8, bufs.k8, bufs.v8, bufs.scales, 256.0, aq.ATTNQ_KV_REVERSE, True, T, O)
        torch.cuda.synchronize()
        got = outs[i].view(torch.int16 if out_bf16 else torch.int32).numpy()
        want = O.cpu().view(torch.int16 if out_bf16 else torch.int32).numpy()
        assert np.array_equal(got, want), i


@pytest.mark.parametrize("steps,N,out_bf16", [(1, 300, True), (3, 1000, False), (5, 257, True)])
def test_host_pipeline_matches_device_path(steps, N, out_bf16):
    _pipeline_vs_device(steps, N, out_bf16)


@pytest.mark.parametrize("extra,stat_len", [("i8", 0), ("tile", 300), ("i8+tile", 200), ("i8", 777)])
def test_host_pipeline_other_options(extra, stat_len):
    """INT8 Q/K codes take two bytes in the pipeline's operand buffers, per-tile
    scales one descale per tile, prefix statistics change only the kernels'
    arguments: every variant still equals the device path bit for bit."""
    import precision_attention_numerics_gb300 as aq
    f = {"i8": aq.ATTNQ_I8QK, "tile": aq.ATTNQ_TILE_SCALES, "i8+tile": aq.ATTNQ_I8QK | aq.ATTNQ_TILE_SCALES}[extra]
    _pipeline_vs_device(3, 1000, True, f, stat_len)


def test_host_pipeline_rejects_bad_arguments():
    import precision_attention_numerics_gb300 as aq
    desc = aq.AttnqDesc(1, 2, 1, 64, 64, aq.ATTNQ_BF16, aq.ATTNQ_VT_LAYOUT, None)
    x = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16).pin_memory()
    o = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(aq.attnq_host_pipeline_workspace(desc, aq.ATTNQ_BF16), dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with pytest.raises(aq.AttnqError) as e:  # the same stream twice
        aq.attnq_attention_host(desc, [x], [x[:, :1]], [x[:, :1]], 256.0, 1, True, 128, [o], aq.ATTNQ_BF16, ws,
                                s1, s1, s2)
    assert e.value.code == 1
    nat = aq.AttnqDesc(1, 2, 1, 64, 64, aq.ATTNQ_BF16, 0, None)
    with pytest.raises(aq.AttnqError) as e:  # the forward pass needs the transposed V layout
        aq.attnq_attention_host(nat, [x], [x[:, :1]], [x[:, :1]], 256.0, 1, True, 128, [o], aq.ATTNQ_BF16, ws,
                                torch.cuda.Stream(), s1, s2)
    assert e.value.code == 2
    with pytest.raises(aq.AttnqError) as e:  # workspace too small
        aq.attnq_attention_host(desc, [x], [x[:, :1]], [x[:, :1]], 256.0, 1, True, 128, [o], aq.ATTNQ_BF16,
                                ws[:256], torch.cuda.Stream(), s1, s2)
    assert e.value.code == 1


@pytest.mark.parametrize("B,Hq,Hkv,N,d,T,f32_in,order", [(2, 6, 2, 333, 64, 64, True, 0), (1, 3, 3, 129, 128, 64, False, 1),
                                                         (3, 5, 1, 700, 64, 128, True, 1)])
def test_host_pipeline_shapes(B, Hq, Hkv, N, d, T, f32_in, order):
    """Other shapes, fp32 inputs, 64-key tiles and the forward order through the
    pipeline: its buffer sizes follow the shape and input type, and every step
    equals the device path bit for bit."""
    import precision_attention_numerics_gb300 as aq
    steps = 3
    flags = aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K | aq.ATTNQ_VT_LAYOUT
    signs = torch.from_numpy(synth.hadamard_signs(23, d)).cuda()
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_F32 if f32_in else aq.ATTNQ_BF16, flags, signs)
    hosts = []
    for i in range(steps):
        q, k, v = synth.qkv_normal(7100 + i, B, Hq, Hkv, N, d)
        if f32_in:
            hosts.append(tuple(torch.from_numpy(x).pin_memory() for x in (q, k, v)))
        else:
            hosts.append(tuple(torch.from_numpy(synth.to_bf16_bits(x)).view(torch.bfloat16).pin_memory()
                               for x in (q, k, v)))
    outs = [torch.full((B, Hq, N, d), float("nan"), dtype=torch.float32).pin_memory() for _ in range(steps)]
    ws = torch.empty(aq.attnq_host_pipeline_workspace(desc, aq.ATTNQ_F32), dtype=torch.uint8, device="cuda")
    compute, cin, cout = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    aq.attnq_attention_host(desc, [h[0] for h in hosts], [h[1] for h in hosts], [h[2] for h in hosts], 448.0,
                            order, True, T, outs, aq.ATTNQ_F32, ws, compute, cin, cout)
    compute.synchronize()
    assert aq.attnq_device_status(compute.cuda_stream) == 0
    bufs = aq.alloc_prepared(desc)
    for i in range(steps):
        Q, K, V = (x.cuda() for x in hosts[i])
        O = torch.empty((B, Hq, N, d), dtype=torch.float32, device="cuda")
        aq.attnq_prepare(desc, Q, K, V, bufs.q8, bufs.k8, bufs.v8, bufs.scales, bufs.workspace)
        aq.attnq_fwd(desc, bufs.q8, bufs.k8, bufs.v8, bufs.scales, 448.0, order, True, T, O)
        torch.cuda.synchronize()
        assert np.array_equal(outs[i].view(torch.int32).numpy(), O.cpu().view(torch.int32).numpy()), i
