"""Attention-mass dilution diagnostic for SharpDraft's query scaling.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: nothing on the
product path imports it.  It is the diagnostic that comes before SharpDraft's
exact top-k mass correction, whose derivation the pages do not print.

"SharpDraft: Accelerating Long-Context Speculative Decoding with
Cardinality-Aware Query Scaling", Abstract: as the softmax normalises over more
visible keys, the probability mass on the highest-scoring keys can fall
(attention-mass dilution); the method scales the query, and with it every
logit, by a closed-form fixed-slope function of the number of visible keys.
The scale used here is the library's reading of that function,
gamma(n) = max(1, 1 + beta * ln(n / N_ref)) (``draft_attn_oracle.sharp_gamma``).

What this module measures, in float64 on synthetic logits:

* ``topk_mass(logits, k)``: the softmax mass of the k largest logits.
* ``dilution_curve``: for a query with k relevant keys whose logits sit
  ``gap`` above a background of n - k keys drawn from N(0, sigma^2), the mean
  top-k mass over draws as n grows, with the logits as they are and with
  SharpDraft's scale applied.
"""
from __future__ import annotations

import math

import numpy as np

from oracle.draft_attn_oracle import sharp_gamma


def topk_mass(logits, k: int) -> float:
    """Softmax probability of the k largest entries of `logits` (float64)."""
    s = np.asarray(logits, dtype=np.float64).ravel()
    if k <= 0 or s.size == 0:
        return 0.0
    k = min(k, s.size)
    m = s.max()
    e = np.exp(s - m)
    top = np.partition(e, s.size - k)[s.size - k:]
    return float(top.sum() / e.sum())


def synthetic_logits(n: int, k: int, gap: float, sigma: float, rng) -> np.ndarray:
    """k relevant keys at `gap` above a background of n - k N(0, sigma^2) logits."""
    s = rng.normal(0.0, sigma, size=n)
    s[:k] = gap
    return s


def dilution_curve(ns, k: int = 8, gap: float = 6.0, sigma: float = 1.0, beta: float = 0.05,
                   n_ref: int = 4096, draws: int = 16, seed: int = 0) -> list[dict]:
    """Mean top-k mass at each n in `ns`, unscaled and with gamma(n) applied."""
    rng = np.random.default_rng(seed)
    rows = []
    for n in ns:
        g = sharp_gamma(n, beta, n_ref)
        plain, scaled = [], []
        for _ in range(draws):
            s = synthetic_logits(n, k, gap, sigma, rng)
            plain.append(topk_mass(s, k))
            scaled.append(topk_mass(g * s, k))
        rows.append({"n": int(n), "gamma": g, "topk_mass": float(np.mean(plain)),
                     "topk_mass_sharp": float(np.mean(scaled))})
    return rows


if __name__ == "__main__":
    ns = [4096, 32768, 131072, 524288, 1048576]
    print("n, gamma, top-8 mass, top-8 mass with SharpDraft scale (k=8, gap=6, sigma=1, "
          "beta=0.05, N_ref=4096, 16 draws)")
    for r in dilution_curve(ns):
        print(f"{r['n']}, {r['gamma']:.4f}, {r['topk_mass']:.4f}, {r['topk_mass_sharp']:.4f}")
