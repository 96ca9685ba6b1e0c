"""Closed forms the pages print, used to pin the oracle's acceptance rule.

TEST INFRASTRUCTURE ONLY (see oracle/verify_step.py).

* Expected tokens per verify pass with independent acceptance alpha and
  gamma drafts: E = (1 - alpha^(gamma+1)) / (1 - alpha) ("Speculative
  Decoding at High Batch Size", section "What does one speculative iteration
  actually cost?"; printed: 4.16 at alpha 0.8, gamma 7).
* The same expectation with position-dependent conditional acceptance
  alpha_1, alpha_2, ...: E = sum_{j=0..gamma} prod_{k<=j} alpha_k; the pages'
  decaying model starts at 0.94 and loses 0.07 per position (section "Why
  should you not trust an independent-acceptance model for long drafts?";
  printed: 4.49 at gamma 7, and 0.33 more tokens going from gamma 5 to 8).
"""
from __future__ import annotations


def expected_tokens(alpha: float, gamma: int) -> float:
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def decaying_alphas(gamma: int, first: float = 0.94, step: float = 0.07):
    return [first - step * k for k in range(gamma)]


def expected_tokens_conditional(alphas) -> float:
    total, run = 1.0, 1.0
    for a in alphas:
        run *= a
        total += run
    return total
