"""The seeded input generators shared by both sides."""
import numpy as np

import synth


def test_splitmix64_published_vector():
    # first outputs of SplitMix64 seeded with 1234567 (the test vector that
    # accompanies public ports of Steele-Lea-Flood's generator)
    assert synth.splitmix64(1234567, 5).tolist() == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]
    assert np.array_equal(synth.splitmix64(1234567, 3, offset=2), synth.splitmix64(1234567, 5)[2:])


def test_normals_moments_and_chunking():
    x = synth.normals(9, 400001, chunk=1 << 12)
    y = synth.normals(9, 400001)
    assert np.array_equal(x, y)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_bf16_rounding_ties_to_even():
    f = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, -2.5], np.float32)
    b = synth.to_bf16_bits(f)
    assert synth.bf16_bits_to_f32(b).tolist() == [1.0, 1.0 + 2 * 2.0 ** -7, 1.0, -2.5]


def test_sink_construction_shifts_logits():
    d, N, delta = 64, 32, 7.0
    q, k, v = synth.sink_inputs(3, 1, 1, N, d, delta)
    logits = q[0, 0] @ k[0, 0].T / np.sqrt(d)
    base = q[0, 0, :, :-1] @ k[0, 0, :, :-1].T / np.sqrt(d)
    shift = logits - base
    assert np.allclose(shift[:, :4], delta, atol=1e-5) and np.allclose(shift[:, 4:], 0.0)


def test_qwen_like_shared_key_vector():
    qb, kb, vb = synth.qwen_like_inputs(5, 1, 4, 2, 64, 64, key_norm=30.0, key_channels=4)
    k = synth.bf16_bits_to_f32(kb).astype(np.float64)
    mean = k.mean(axis=2)                        # [1, 2, 64]
    big = np.sort(np.abs(mean), axis=-1)[..., -4:]
    assert np.all(big > 13.0) and np.linalg.norm(big, axis=-1).min() > 27.0
    assert synth.hadamard_signs(1, 128).dtype == np.int8
