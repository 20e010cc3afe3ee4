"""Closed forms the pages give around the verification step (fp64, plain Python).

TEST INFRASTRUCTURE ONLY (imported by tests and by the benchmark's report of
the speedup model, never by the CUDA path).

  expected_tokens   E[N] = (1 - a^(g+1)) / (1 - a)
                    ("Speculative Decoding in Large Language Models", section 2,
                    "Theoretical Speedup Equation")
  cycle_speedup     S = E[N] / (1 + g c)            (same section)
  measured_speedup  T_verif(B) AL / (T_verif(B (1 + D)) + T_draft(B, D))
                    ("Co-Designing AI Models Using Speculative Decoding",
                    "What is speculative decoding?")
  acceptance_beta   beta = sum_y min(q(y), p(y))   (section 2, "Proof of
                    Distributional Invariance")
  mean_accept_length  E[AL] = sum_{k=0}^{K} prod_{j<k} beta_j for independent
                    per-position acceptance with probabilities beta_j; with all
                    beta_j = a it is the E[N] above.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np


def expected_tokens(alpha: float, gamma: int) -> float:
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def cycle_speedup(alpha: float, gamma: int, c: float) -> float:
    return expected_tokens(alpha, gamma) / (1.0 + gamma * c)


def measured_speedup(t_verif_b: float, t_verif_b1d: float, t_draft: float, al: float) -> float:
    return t_verif_b * al / (t_verif_b1d + t_draft)


def acceptance_beta(p: np.ndarray, q: np.ndarray) -> float:
    return float(np.minimum(np.asarray(p, np.float64), np.asarray(q, np.float64)).sum())


def mean_accept_length(betas: Sequence[float]) -> float:
    total, run = 1.0, 1.0
    for b in betas:
        run *= b
        total += run
    return total
