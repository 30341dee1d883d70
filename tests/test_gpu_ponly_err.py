"""GPU parity of attnq_fwd_ponly (P-only mode) and attnq_err."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _ponly(q, k, v, S, order, causal, T):
    import precision_attention_numerics_gb300 as aq
    from tests.gpu_helpers import dev
    B, Hq, N, d = q.shape
    desc = aq.AttnqDesc(B, Hq, k.shape[1], N, d, aq.ATTNQ_F32, 0, None)
    O = torch.empty((B, Hq, N, d), dtype=torch.float32, device="cuda")
    uf = torch.zeros(B * Hq * 2, dtype=torch.int64, device="cuda")
    aq.attnq_fwd_ponly(desc, dev(q), dev(k), dev(v), S, order, causal, T, O, uf)
    assert aq.attnq_device_status() == 0
    return O.cpu().numpy().astype(np.float64).reshape(B * Hq, N, d), uf.cpu().numpy().reshape(-1, 2)


@pytest.mark.parametrize("delta", [0.0, 7.0, 12.0])
@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("S", [1.0, 256.0, 448.0])
def test_ponly_pcast_sweep_shape(delta, order, S):
    """P-cast sweep shape (H=8, d=128, T=128) at N=1024."""
    from tests.gpu_helpers import rel_f
    q, k, v = synth.sink_inputs(2000 + int(delta), 1, 8, 1024, 128, delta=delta)
    got, uf = _ponly(q, k, v, S, order, True, 128)
    ref, uref = oracle.attn_ponly(q, k, v, S, order, True, 128)
    assert rel_f(got, ref).max() <= 2e-3
    assert np.all(np.abs(uf - uref.astype(np.int64)) <= 0.001 * uref + 2), (uf, uref)


@pytest.mark.parametrize("T", [16, 48, 64])
@pytest.mark.parametrize("N", [1, 33, 130])
def test_ponly_tiles_and_ragged(T, N):
    from tests.gpu_helpers import rel_f
    q, k, v = synth.sink_inputs(2100 + N + T, 1, 2, N, 64, delta=4.0)
    for causal in (True, False):
        got, uf = _ponly(q, k, v, 256.0, 1, causal, T)
        ref, uref = oracle.attn_ponly(q, k, v, 256.0, 1, causal, T)
        assert rel_f(got, ref).max() <= 2e-3


@pytest.mark.parametrize("o_dtype", [torch.float32, torch.bfloat16])
def test_err_matches_oracle(o_dtype):
    import precision_attention_numerics_gb300 as aq
    B, Hq, N, d = 2, 3, 257, 64
    ref = synth.normals(3000, B * Hq * N * d).reshape(B, Hq, N, d).astype(np.float64) * 1.7
    noise = synth.normals(3001, B * Hq * N * d).reshape(B, Hq, N, d).astype(np.float64)
    scale = np.array([1e-3, 1e-2, 0.3, 0.0, 2.0, 1e-5]).reshape(B, Hq, 1, 1)
    O = (ref + noise * scale).astype(np.float32)
    Ot = torch.from_numpy(O).cuda().to(o_dtype)
    Oref = torch.from_numpy(ref).cuda()
    err = torch.empty(B * Hq, dtype=torch.float64, device="cuda")
    desc = aq.AttnqDesc(B, Hq, Hq, N, d, aq.ATTNQ_F32, 0, None)
    aq.attnq_err(desc, Ot, Oref, err)
    got = err.cpu().numpy()
    O64 = Ot.float().cpu().numpy().astype(np.float64).reshape(B * Hq, -1)
    want = oracle.err(O64, ref.reshape(B * Hq, -1))
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-15)


def test_err_zero_reference():
    import precision_attention_numerics_gb300 as aq
    O = torch.zeros((1, 2, 16, 64), device="cuda")
    O[0, 1, 3, 3] = 1.0
    Oref = torch.zeros((1, 2, 16, 64), dtype=torch.float64, device="cuda")
    err = torch.empty(2, dtype=torch.float64, device="cuda")
    aq.attnq_err(aq.AttnqDesc(1, 2, 2, 16, 64, aq.ATTNQ_F32, 0, None), O, Oref, err)
    e = err.cpu().numpy()
    assert e[0] == 0.0 and np.isinf(e[1])
