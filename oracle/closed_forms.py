"""Closed forms from the P-cast page ("Technische Samenvatting: P-Cast Precisie
in FP8 Attention", sections 2 and 3).  Test infrastructure, like the rest of
oracle/.

* Phi: standard normal CDF.
* ROUND_TO_ZERO_NATS = 10 ln 2: an E4M3 value at or below 2^-10 rounds to
  zero; in natural-log units the threshold sits 10 ln 2 (printed as 6.93)
  below the running maximum.
* delta_k(k): expected maximum of k standard normals (printed as about 1.0
  for k = 4), by quadrature of x * k phi(x) Phi(x)^(k-1).
* underflow_fraction F(delta, S) = Phi(delta + delta_k - 10 ln 2 - ln S):
  predicted share of non-sink P values cast to zero under forward iteration
  (section 2, "Theoretisch Kader").
* underflow_fraction_spread(delta, S, k, var): the same model without
  replacing the sink maximum by its mean: P(x - M <= delta - 10 ln 2 - ln S)
  with x ~ N(0, var) a non-sink logit and M the maximum of k N(0, var) sink
  logit residues, by quadrature.  F above is this with M fixed at its mean;
  the spread of M (sd ~0.70 for k = 4) is why F is off by up to ~0.046 in its
  tails (max over z of |Phi(z) - Phi(z / sqrt(1 + 0.49))|).
* critical_delta = 10 ln 2 + ln S - delta_k: onset of the collapse
  (section 3, item 1).
* reverse_bound(N, S): with reverse iteration the running max before the sink
  block is the maximum of about N standard normals, near sqrt(2 ln N); a
  non-sink P underflows with probability Phi(sqrt(2 ln N) - 10 ln 2 - ln S)
  (section 2, "Optimalisatie 1").
* d_p(S, table): the largest E4M3 quantisation step met by P*S for P in
  (0, 1], divided by S (section 2, "Optimalisatie 2", item 2); computed by
  brute force over the oracle's decode table.
* normal_coverage(S) = 2^-6 / S: smallest P whose P*S is an E4M3 normal
  (item 3).
"""
from __future__ import annotations

import math

import numpy as np

ROUND_TO_ZERO_NATS = 10.0 * math.log(2.0)


def Phi(x: float) -> float:
    return 0.5 * math.erfc(-x / math.sqrt(2.0))


def delta_k(k: int) -> float:
    from scipy import integrate

    def f(x):
        phi = math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)
        return x * k * phi * Phi(x) ** (k - 1)

    val, _ = integrate.quad(f, -12.0, 12.0, epsabs=1e-13, epsrel=1e-12, limit=200)
    return val


def underflow_fraction(delta: float, S: float, k: int = 4) -> float:
    return Phi(delta + delta_k(k) - ROUND_TO_ZERO_NATS - math.log(S))


def underflow_fraction_spread(delta: float, S: float, k: int = 4, var: float = 1.0) -> float:
    from scipy import integrate

    sd = math.sqrt(var)
    c = ROUND_TO_ZERO_NATS + math.log(S)

    def f(m):
        z = m / sd
        dens = k * math.exp(-0.5 * z * z) / (math.sqrt(2.0 * math.pi) * sd) * Phi(z) ** (k - 1)
        return Phi((delta - c + m) / sd) * dens

    val, _ = integrate.quad(f, -12.0 * sd, 12.0 * sd, epsabs=1e-13, epsrel=1e-11, limit=200)
    return val


def critical_delta(S: float, k: int = 4) -> float:
    return ROUND_TO_ZERO_NATS + math.log(S) - delta_k(k)


def reverse_bound(N: int, S: float) -> float:
    return Phi(math.sqrt(2.0 * math.log(N)) - ROUND_TO_ZERO_NATS - math.log(S))


def d_p(S: float, table: np.ndarray) -> float:
    """Largest gap between consecutive positive E4M3 values v_k < S, over S."""
    pos = np.sort(table[np.isfinite(table) & (table >= 0.0)])
    pos = np.unique(pos)
    gaps = np.diff(pos)
    lower = pos[:-1]
    return float(gaps[lower < S].max() / S)


def normal_coverage(S: float, table: np.ndarray) -> float:
    """Smallest P with P*S an E4M3 normal: (smallest normal) / S."""
    codes = np.arange(256)
    normal = ((codes >> 3) & 15) > 0
    vals = table[normal & (codes < 128) & np.isfinite(table)]
    return float(vals.min() / S)
