"""Seeded synthetic inputs shaped like the workloads of the attention-numerics pages.

This module draws random numbers and builds input tensors; it holds none of the
attention method's arithmetic (no quantisation, rotation, softmax or scaling).
Both the CPU oracle's tests and the CUDA path's tests and benchmark take their
inputs from here, so the two sides always see identical bits.

Random source: SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used as a counter-based
generator: output i (1-based) of stream `seed` is mix(seed + i * 0x9E3779B97F4A7C15).
Normals come from the Box-Muller transform on pairs of 53-bit uniforms.

bf16 tensors are carried as uint16 bit patterns (numpy has no bf16 type); the
conversion from float32 is round-to-nearest-even on the bit pattern.

Workload recipes (the pages' workloads are private captures of Qwen models on
three books; these shapes stand in for them):

* sink probe / P-cast sweep (page "Technische Samenvatting: P-Cast Precisie in
  FP8 Attention", sections 2 and 4): i.i.d. N(0,1) Q, K, V; the last channel
  is reserved for k sink keys (tokens 0..k-1): Q[:, d-1] = K[:k, d-1] =
  sqrt(delta * sqrt(d)), K[k:, d-1] = 0, so each query's sink logits
  q.k/sqrt(d) exceed the others by delta while keeping the N(0,1) spread of
  the remaining d-1 channels.
* Qwen-shaped layers (page "attention-numerics", loss and head-transfer
  sections): bf16 N(0,1) Q, K, V plus a key vector shared by every token of a
  KV head (norm `key_norm` spread evenly over `key_channels` seeded channels)
  and `q_outliers` seeded channels per query head multiplied by 20.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset+1 .. offset+n of the SplitMix64 stream started at `seed`."""
    idx = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniforms(seed: int, n: int) -> np.ndarray:
    """n float64 uniforms in [0, 1) with 53 random bits each."""
    return (splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normals_block(seed: int, out: np.ndarray, pair0: int, m: int, n: int) -> None:
    z = splitmix64(seed, 2 * m, offset=2 * pair0)
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    del z
    r = np.sqrt(-2.0 * np.log(u1))
    th = (2.0 * math.pi) * u2
    pair = np.empty(2 * m, dtype=np.float64)
    pair[0::2] = r * np.cos(th)
    pair[1::2] = r * np.sin(th)
    lo = 2 * pair0
    hi = min(n, lo + 2 * m)
    out[lo:hi] = pair[: hi - lo]


def normals(seed: int, n: int, chunk: int = 1 << 22, threads: int | None = None) -> np.ndarray:
    """n standard normals (float32) by Box-Muller on SplitMix64 pairs.

    Pair p uses stream outputs 2p+1 and 2p+2, so the result does not depend
    on the chunking or the thread count; chunks run on a thread pool (numpy
    releases the GIL inside its loops).
    """
    out = np.empty(n, dtype=np.float32)
    pairs_total = (n + 1) // 2
    starts = list(range(0, pairs_total, chunk))
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    if len(starts) <= 1 or threads <= 1:
        for p0 in starts:
            _normals_block(seed, out, p0, min(chunk, pairs_total - p0), n)
        return out
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda p0: _normals_block(seed, out, p0, min(chunk, pairs_total - p0), n), starts))
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def hadamard_signs(seed: int, d: int) -> np.ndarray:
    """Random +-1 signs (int8, length d): bit 63 of SplitMix64 output i selects -1."""
    z = splitmix64(seed, d)
    return np.where((z >> np.uint64(63)) == np.uint64(1), -1, 1).astype(np.int8)


def pick_channels(seed: int, d: int, k: int, exclude: tuple[int, ...] = ()) -> np.ndarray:
    """k distinct channels in [0, d) chosen by a seeded partial Fisher-Yates shuffle."""
    pool = [c for c in range(d) if c not in exclude]
    z = splitmix64(seed, k)
    for t in range(k):
        r = t + int(z[t] % np.uint64(len(pool) - t))
        pool[t], pool[r] = pool[r], pool[t]
    return np.array(sorted(pool[:k]), dtype=np.int64)


# ---------------------------------------------------------------------------
# workload builders
# ---------------------------------------------------------------------------

def qkv_normal(seed: int, B: int, Hq: int, Hkv: int, N: int, d: int):
    """Independent N(0,1) float32 Q [B,Hq,N,d], K and V [B,Hkv,N,d]."""
    q = normals(seed * 3 + 0, B * Hq * N * d).reshape(B, Hq, N, d)
    k = normals(seed * 3 + 1, B * Hkv * N * d).reshape(B, Hkv, N, d)
    v = normals(seed * 3 + 2, B * Hkv * N * d).reshape(B, Hkv, N, d)
    return q, k, v


def sink_inputs(seed: int, B: int, H: int, N: int, d: int, delta: float, k_sink: int = 4):
    """float32 Q, K, V with k_sink sink keys whose logits exceed the others by delta."""
    q, k, v = qkv_normal(seed, B, H, H, N, d)
    a = np.float32(math.sqrt(delta * math.sqrt(d)))
    q[..., d - 1] = a
    k[..., d - 1] = 0.0
    k[:, :, :k_sink, d - 1] = a
    return q, k, v


def qwen_like_inputs(seed: int, B: int, Hq: int, Hkv: int, N: int, d: int,
                     key_norm: float, key_channels: int, q_outliers: int = 2,
                     outlier_gain: float = 20.0):
    """bf16 bit patterns of Q, K, V shaped like a Qwen attention layer.

    K gets a shared vector (every token of a KV head) of norm `key_norm` spread
    evenly over `key_channels` seeded channels; each query head gets
    `q_outliers` seeded channels multiplied by `outlier_gain`.
    """
    q, k, v = qkv_normal(seed, B, Hq, Hkv, N, d)
    per = np.float32(key_norm / math.sqrt(key_channels))
    for g in range(Hkv):
        ch = pick_channels(seed * 7919 + 17 + g, d, key_channels)
        k[:, g, :, ch] += per
    for h in range(Hq):
        ch = pick_channels(seed * 7919 + 1009 + h, d, q_outliers)
        q[:, h, :, ch] *= np.float32(outlier_gain)
    return to_bf16_bits(q), to_bf16_bits(k), to_bf16_bits(v)


def long_context_inputs(seed: int, B: int = 2, Hq: int = 32, Hkv: int = 8, N: int = 32768, d: int = 128):
    """bf16 bit patterns of i.i.d. N(0,1) Q, K, V (the long-context throughput workload)."""
    q, k, v = qkv_normal(seed, B, Hq, Hkv, N, d)
    return to_bf16_bits(q), to_bf16_bits(k), to_bf16_bits(v)


# The five workloads, by name. Sizes follow the pages' descriptions; seeds are
# 1000 * workload index + sub-index.
WORKLOADS = {
    "sink_probe": dict(B=1, Hq=1, Hkv=1, N=256, d=64, kv_tile=64, deltas=(7.0,), S=(1.0, 256.0),
                       orders=("forward",), rotate=False, center=False, dtype="f32"),
    "pcast_sweep": dict(B=1, Hq=8, Hkv=8, N=4096, d=128, kv_tile=128, deltas=tuple(float(x) for x in range(13)),
                        S=(1.0, 256.0, 448.0), orders=("forward", "reverse"), dtype="f32"),
    "qwen05b": dict(B=3, Hq=14, Hkv=2, N=1024, d=64, kv_tile=128, layers=24, key_norm=30.0, key_channels=4,
                    S=(256.0,), orders=("reverse",), dtype="bf16"),
    "qwen15b": dict(B=3, Hq=12, Hkv=2, N=1024, d=128, kv_tile=128, layers=28, key_norm=40.0, key_channels=8,
                    S=(256.0,), orders=("reverse",), dtype="bf16"),
    "long_context": dict(B=2, Hq=32, Hkv=8, N=32768, d=128, kv_tile=128, S=(256.0,), orders=("reverse",),
                         rotate=True, center=True, dtype="bf16"),
}

CONDITIONS = {  # name -> (rotate, center_k)
    "unrotated": (False, False),
    "rotated": (True, False),
    "centred": (False, True),
    "centred_rotated": (True, True),
}


# Seeds of the workloads' instances: 1000 * workload index + sub-index.
SEED_BASE = {"sink_probe": 1000, "pcast_sweep": 2000, "qwen05b": 3000, "qwen15b": 4000, "long_context": 5000}


def sink_probe_inputs():
    """The sink probe's one instance (delta = 7)."""
    wl = WORKLOADS["sink_probe"]
    return sink_inputs(SEED_BASE["sink_probe"] + 1, wl["B"], wl["Hq"], wl["N"], wl["d"], delta=wl["deltas"][0])


def pcast_sweep_inputs(delta: float, N: int | None = None):
    """One delta of the P-cast sweep (float32, 8 heads); N defaults to the sweep's 4096."""
    wl = WORKLOADS["pcast_sweep"]
    return sink_inputs(SEED_BASE["pcast_sweep"] + int(delta), wl["B"], wl["Hq"], wl["N"] if N is None else N,
                       wl["d"], delta=float(delta))


def qwen_layer_inputs(name: str, layer: int):
    """Layer `layer` of a Qwen-shaped workload ("qwen05b" or "qwen15b"): bf16 bit patterns."""
    wl = WORKLOADS[name]
    return qwen_like_inputs(SEED_BASE[name] + layer, wl["B"], wl["Hq"], wl["Hkv"], wl["N"], wl["d"],
                            key_norm=wl["key_norm"], key_channels=wl["key_channels"])


def qwen_signs(name: str):
    """The fixed Hadamard sign vector of a Qwen-shaped workload (one for all its layers)."""
    return hadamard_signs(SEED_BASE[name] + 1, WORKLOADS[name]["d"])
