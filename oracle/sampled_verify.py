"""Oracle for stochastic (lossless) tree verification.

TEST INFRASTRUCTURE ONLY: the test suite and the benchmark's CPU baseline use it; the
product path never imports it.  Plain Python and numpy in fp64, sharing no code with the
CUDA kernels.

What is verified.  The JetFlow pages call draft-then-verify lossless (qxai.app commentary
on JetFlow, "まず、何が問題なのか" and "慎重に見るべき点"; explainer §1 Problem): the
output must follow the target model's own distribution.  They give no rule.  The reading
taken here is the multi-step speculative sampling of SpecInfer (Miao et al., "SpecInfer:
Accelerating Generative LLM Serving with Tree-based Speculative Inference and
Verification", ASPLOS 2024) for drafts that are deterministic: the draft tree's children
of a node are fixed candidate tokens (the top-K of a depth, explainer §2 tree
construction), i.e. each trial's draft distribution is a point mass on its token, so the
residual after rejecting token x is the target distribution with x removed.  At node u:

    p = softmax(logits[u] / T)                     (the target's next-token distribution)
    r = p; for the children c of u in increasing node id (best-first order):
        accept c iff uniform[c] * sum(r) < r[draft[c]]         (probability r(x) / sum r)
        on acceptance continue at c; on rejection set r[draft[c]] = 0
    if no child is accepted (or u has none): the bonus token is the smallest y with
        cumsum(r)[y] > bonus_uniform * sum(r)                  (a sample of r / sum r)

Every emitted token is then distributed exactly as the target's p at its position (the
chain rule: token x_i is emitted with probability prod_{j<i}(1 - p(x_j)/R_j) * p(x_i)/R_i
= p(x_i), R_i the residual mass; the rest with p(y)), which is what lossless means.
The random numbers are inputs: uniform[b][c] is the one drawn when child c is tested
(each node is tested at most once; entry 0 is unused) and bonus_uniform[b] the one drawn
for the bonus token, all in [0, 1).
"""
from __future__ import annotations

import numpy as np


def _rows_f64(logits: np.ndarray, dtype: str) -> np.ndarray:
    """bf16 bit patterns (uint16) or fp32 values -> float64, exactly."""
    if dtype == "bf16":
        bits = np.asarray(logits, dtype=np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(logits, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def target_probs(row: np.ndarray, temperature: float) -> np.ndarray:
    """softmax(row / T) in fp64 (row already float64)."""
    x = row / float(temperature)
    e = np.exp(x - x.max())
    return e / e.sum()


def tree_verify_sampled(logits, dtype: str, draft, parent, uniform, bonus_uniform,
                        temperature: float):
    """Stochastic verification of B trees (see the module docstring).

    logits [B][N][V] (bf16 bits or fp32), draft / parent int [B][N], uniform float [B][N],
    bonus_uniform float [B].  Returns (accept_len int32 [B], path int32 [B][N] (-1 padded),
    bonus int32 [B], margins) where margins[b] lists, for every decision taken, the distance
    between the drawn threshold and the decision boundary relative to the residual mass:
    ("accept" or "reject", node, margin) and ("bonus", y, margin) -- a decision whose margin
    is below the floating-point error of a kernel may legitimately come out the other way."""
    rows = _rows_f64(logits, dtype)
    draft = np.asarray(draft, dtype=np.int64)
    parent = np.asarray(parent, dtype=np.int64)
    uniform = np.asarray(uniform, dtype=np.float64)
    bonus_uniform = np.asarray(bonus_uniform, dtype=np.float64)
    B, N, V = rows.shape
    acc = np.zeros(B, dtype=np.int32)
    path = np.full((B, N), -1, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int32)
    margins = []
    for b in range(B):
        children = [[] for _ in range(N)]
        for c in range(1, N):
            children[int(parent[b, c])].append(c)
        u, walk, mb = 0, [0], []
        while True:
            r = target_probs(rows[b, u], temperature)
            nxt = None
            for c in children[u]:
                x = int(draft[b, c])
                mass = r.sum()
                thr = uniform[b, c] * mass
                if thr < r[x]:
                    mb.append(("accept", c, (r[x] - thr) / mass))
                    nxt = c
                    break
                mb.append(("reject", c, (thr - r[x]) / mass))
                r[x] = 0.0
            if nxt is None:
                mass = r.sum()
                target = bonus_uniform[b] * mass
                cdf = np.cumsum(r)
                y = int(np.searchsorted(cdf, target, side="right"))
                if y >= V:                       # rounding at the very top: last live token
                    y = int(np.flatnonzero(r > 0)[-1])
                lo = cdf[y - 1] if y > 0 else 0.0
                mb.append(("bonus", y, min(target - lo, cdf[y] - target) / mass))
                bonus[b] = y
                break
            walk.append(nxt)
            u = nxt
        acc[b] = len(walk) - 1
        path[b, :len(walk)] = walk
        margins.append(mb)
    return acc, path, bonus, margins
