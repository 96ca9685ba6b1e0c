"""Roofline and speedup model of a speculative verify step, and its fit to measurements.

The model ("Speculative Decoding at High Batch Size: Where the 3x Speedup Turns
Into a Tax", sections "What does one speculative iteration actually cost?" and
"How does the roofline model work?"): a step over B sequences of n tokens each
costs the larger of its memory time and its compute time,

    t_step(B, n, frac) = max(t_w * frac + B * k,  c * frac * B * n)

with t_w the time to read the weights once, k the time to read one sequence's
KV cache, c the compute time of one token, and frac the share of the weights a
pass touches (the pages charge a drafter pass 4 % of the target's).  One
speculative iteration verifies gamma + 1 tokens per sequence and drafts gamma,
and yields E tokens per sequence:

    speedup(B, gamma) = E * t_step(B, 1) / (t_step(B, gamma + 1) + t_step(B, gamma, 0.04))

The verify pass turns compute-bound at B* = t_w / ((gamma + 1) c - k).

``fit`` (least squares on the max() form) and ``fit_regimes`` (each parameter
from the regime that exposes it) recover t_w, k and c from measured step
times, so the same questions
(where the pass turns compute-bound, the best draft length per batch size,
where speculation stops paying) can be asked of this GPU instead of the
pages' illustrative H100-class numbers.  Host-side arithmetic only.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable, Iterable, Sequence

DRAFT_FRAC = 0.04  # a drafter pass costs this share of a target pass


@dataclass(frozen=True)
class StepModel:
    t_w: float  # weight-read time per step
    k: float    # KV-read time per sequence
    c: float    # compute time per token

    def t_step(self, B: float, n: float, frac: float = 1.0) -> float:
        return max(self.t_w * frac + B * self.k, self.c * frac * B * n)

    def b_star(self, gamma: int) -> float:
        """Batch size at which verifying gamma + 1 tokens per sequence turns compute-bound."""
        d = (gamma + 1) * self.c - self.k
        return math.inf if d <= 0 else self.t_w / d

    def speedup(self, B: float, gamma: int, expected: float) -> float:
        base = self.t_step(B, 1)
        spec = self.t_step(B, gamma + 1) + self.t_step(B, gamma, DRAFT_FRAC)
        return expected * base / spec

    def rows_budget(self, B: float = 0.0) -> float:
        """Verify rows (B times tokens per sequence) that still hide under the
        memory time of a pass over B sequences: (t_w + B k) / c."""
        return (self.t_w + B * self.k) / self.c


def expected_tokens_iid(alpha: float, gamma: int) -> float:
    """E = (1 - alpha^(gamma+1)) / (1 - alpha): tokens per pass, independent acceptance."""
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def expected_tokens_conditional(alphas: Sequence[float]) -> float:
    """Tokens per pass when draft position j is accepted with conditional probability alphas[j]."""
    total, run = 1.0, 1.0
    for a in alphas:
        run *= a
        total += run
    return total


def decaying(gamma: int, first: float = 0.94, step: float = 0.07) -> float:
    """The pages' decaying acceptance (94 % at the first position, 7 points less per
    position, each conditional on the previous): tokens per pass."""
    return expected_tokens_conditional([first - step * j for j in range(gamma)])


def best_gamma(model: StepModel, B: float, expected: Callable[[int], float],
               gammas: Iterable[int] = range(1, 9)) -> int:
    """The draft length with the highest speedup at batch size B."""
    return max(gammas, key=lambda g: model.speedup(B, g, expected(g)))


def break_even(model: StepModel, gamma: int, expected: float, limit: int = 100000) -> int | None:
    """The smallest batch size at which speculation of length gamma is slower than plain decoding."""
    for B in range(1, limit + 1):
        if model.speedup(B, gamma, expected) < 1.0:
            return B
    return None


def fit(points: Iterable[tuple[float, float, float]], iters: int = 60) -> StepModel:
    """Fit (t_w, k, c) to measured steps (B, tokens per sequence n, step time).

    Points whose compute estimate exceeds their memory estimate are assigned to
    the compute branch, the rest to the memory branch; each branch is a linear
    least-squares problem (t = t_w + B k, and t = c B n through the origin), and
    the assignment is iterated to a fixed point.
    """
    pts = [(float(B), float(n), float(t)) for B, n, t in points]
    if len(pts) < 3:
        raise ValueError("need at least three measured steps")
    # start: every point memory-bound except the largest B n
    order = sorted(range(len(pts)), key=lambda i: pts[i][0] * pts[i][1])
    comp = {order[-1]}
    model = None
    for _ in range(iters):
        mem = [p for i, p in enumerate(pts) if i not in comp]
        cmp_ = [p for i, p in enumerate(pts) if i in comp]
        t_w, k = _line(mem) if len(mem) >= 2 else (min(p[2] for p in pts), 0.0)
        c = (sum(p[0] * p[1] * p[2] for p in cmp_) / sum((p[0] * p[1]) ** 2 for p in cmp_)) if cmp_ else 0.0
        model = StepModel(t_w=t_w, k=max(k, 0.0), c=max(c, 0.0))
        new = {i for i, (B, n, _) in enumerate(pts) if model.c * B * n > model.t_w + B * model.k}
        if not new:
            new = {order[-1]}
        if new == comp:
            break
        comp = new
    return model


def fit_regimes(points: Iterable[tuple[float, float, float]], compute_rows: float | None = None) -> StepModel:
    """Each parameter from the regime that exposes it (the pages' advice: use the
    model for the shape of the curve, with your own measured rates):

      t_w: the step time at the fewest rows (one sequence, one token);
      k:   the slope over B of the steps that verify one token per sequence;
      c:   time per row, least squares through the origin, over the steps with
           at least ``compute_rows`` rows (default: the largest quarter of B n).
    """
    pts = [(float(B), float(n), float(t)) for B, n, t in points]
    if len(pts) < 3:
        raise ValueError("need at least three measured steps")
    first = min(pts, key=lambda p: (p[0] * p[1], p[2]))
    t_w = first[2]
    ones = [p for p in pts if p[1] == 1.0]
    k = max(_line(ones)[1], 0.0) if len({p[0] for p in ones}) >= 2 else 0.0
    rows = sorted(p[0] * p[1] for p in pts)
    lim = compute_rows if compute_rows is not None else rows[(3 * len(rows)) // 4]
    big = [p for p in pts if p[0] * p[1] >= lim]
    c = sum(p[0] * p[1] * p[2] for p in big) / sum((p[0] * p[1]) ** 2 for p in big)
    return StepModel(t_w=t_w, k=k, c=c)


def _line(pts):
    """Least squares t = a + b B."""
    n = len(pts)
    sx = sum(p[0] for p in pts)
    sy = sum(p[2] for p in pts)
    sxx = sum(p[0] * p[0] for p in pts)
    sxy = sum(p[0] * p[2] for p in pts)
    den = n * sxx - sx * sx
    if den == 0:
        return sy / n, 0.0
    b = (n * sxy - sx * sy) / den
    return (sy - b * sx) / n, b


def report(model: StepModel, expected: Callable[[int], float] = decaying,
           batches: Sequence[int] = (1, 8, 16, 32, 64, 128)) -> dict:
    """B* at gamma 3 and 7, the best gamma per batch size and break-even batch sizes."""
    return {
        "t_w": model.t_w, "k": model.k, "c": model.c,
        "b_star": {g: model.b_star(g) for g in (3, 7)},
        "best_gamma": {B: best_gamma(model, B, expected) for B in batches},
        "speedup_at_best": {B: model.speedup(B, best_gamma(model, B, expected),
                                             expected(best_gamma(model, B, expected))) for B in batches},
        "break_even": {g: break_even(model, g, expected(g)) for g in (3, 7, 8)},
        "rows_budget_B1": model.rows_budget(1),
    }
