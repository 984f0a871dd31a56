"""Acceptance analytics over the verification step's outputs (host side, numpy).

What a serving loop needs to choose the draft length from what `spec_verify`
already returns.  The formulas are the pages':
  * expected tokens per round with an i.i.d. acceptance rate alpha,
    (1 - alpha^(gamma+1)) / (1 - alpha), and the walltime speedup
    (1 - alpha^(gamma+1)) / ((1 - alpha)(gamma c + 1)) with c the drafter's cost
    relative to the target's, and the operations increase
    (1 - alpha)(gamma c_hat + gamma + 1) / (1 - alpha^(gamma+1))
    ("Fast Inference from Transformers via Speculative Decoding" review page,
    section Analysis: expected tokens, speedup, operations, optimal gamma);
  * the acceptance length with position-dependent rates,
    tau = 1 + sum_k prod_{i<=k} alpha_i ("Speculative decoding: the art of
    guessing well", section on how many tokens a round yields).
For fixed rows the acceptance of draft i (given the earlier ones were accepted)
has probability alpha_i = sum_x min(p_i, q_i), the per-position `alpha` the
step returns, so tau of a sequence is exact for its rows.
"""
from __future__ import annotations

import numpy as np


def expected_tokens(alpha, gamma):
    """E[#tokens per round] = (1 - alpha^(gamma+1)) / (1 - alpha); gamma + 1 at alpha = 1."""
    a = np.asarray(alpha, dtype=np.float64)
    g = np.asarray(gamma, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (1.0 - a ** (g + 1)) / (1.0 - a)
    return np.where(a == 1.0, g + 1.0, v)


def walltime_speedup(alpha, gamma, c):
    """(1 - alpha^(gamma+1)) / ((1 - alpha)(gamma c + 1))."""
    return expected_tokens(alpha, gamma) / (np.asarray(gamma, dtype=np.float64) * c + 1.0)


def operations_increase(alpha, gamma, c_hat=0.0):
    """(1 - alpha)(gamma c_hat + gamma + 1) / (1 - alpha^(gamma+1))."""
    g = np.asarray(gamma, dtype=np.float64)
    return (g * c_hat + g + 1.0) / expected_tokens(alpha, gamma)


def optimal_gamma(alpha: float, c: float, gamma_max: int = 256) -> int:
    """The integer gamma in [1, gamma_max] that maximises the walltime speedup (the
    smallest one on ties)."""
    g = np.arange(1, gamma_max + 1)
    return int(g[np.argmax(walltime_speedup(alpha, g, c))])


def acceptance_length(alpha_rows, num_draft=None):
    """tau_b = 1 + sum_{k <= gamma_b} prod_{i <= k} alpha_{b,i} for every sequence of a
    batch: alpha_rows [B, G] (the step's `alpha`; entries past gamma_b are ignored),
    num_draft [B] or None (all G).  Returns [B] float64, the expected number of
    tokens each sequence's round emits."""
    a = np.asarray(alpha_rows, dtype=np.float64)
    B, G = a.shape
    nd = np.full(B, G) if num_draft is None else np.asarray(num_draft).reshape(B)
    mask = np.arange(G)[None, :] < nd[:, None]
    prods = np.cumprod(np.where(mask, a, 1.0), axis=1)
    return 1.0 + np.where(mask, prods, 0.0).sum(axis=1)


def position_rates(alpha_rows, num_draft=None):
    """Mean acceptance rate at each draft position over the sequences that have it:
    [G] float64 (NaN where no sequence drafts that far)."""
    a = np.asarray(alpha_rows, dtype=np.float64)
    B, G = a.shape
    nd = np.full(B, G) if num_draft is None else np.asarray(num_draft).reshape(B)
    mask = np.arange(G)[None, :] < nd[:, None]
    cnt = mask.sum(axis=0)
    with np.errstate(invalid="ignore"):
        return np.where(cnt > 0, np.where(mask, a, 0.0).sum(axis=0) / np.maximum(cnt, 1), np.nan)
