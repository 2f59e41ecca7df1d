"""Oracle for best-first draft-tree construction from per-depth draft logits.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU
baseline use it; the product path never imports it.  Plain Python and numpy, sharing no
code with the CUDA kernels.

Follows the JetFlow explainer ("JetFlow: Breaking the Scaling Ceiling of Speculative
Decoding with Parallel Tree Drafting"), technical summary §2 "Method", tree
construction: the draft head produces logits for all tree depths in one pass, nodes are
ranked by the cumulative draft log-probability, and a best-first expansion builds the
tree up to the budget.  Readings where the pages are silent: the candidates of a depth
are its K most likely tokens (lower token id on ties); every node of depth d has the
depth-(d+1) candidates as children; the cumulative log-probability is the exact sum of
the path's log-probabilities (the pages fix no precision, so it is taken in fp64 like
every other oracle quantity); ties in the expansion order go to the shallower node, then
to the smaller rank path.
"""
from __future__ import annotations

import heapq

import numpy as np


def depth_candidates(logits_row: np.ndarray, K: int):
    """Log-softmax of one depth's logits (fp64) and its K most likely tokens.

    Returns (tokens int64[K], logp float64[K]): tokens by decreasing logit, lower id first
    among equal logits; logp = logit - log(sum(exp(logits)))."""
    x = np.asarray(logits_row, dtype=np.float64)
    m = x.max()
    lse = m + np.log(np.exp(x - m).sum())
    remaining = x.copy()
    tokens = []
    for _ in range(K):                       # K passes of "largest remaining, first index"
        best = int(np.argmax(remaining))     # argmax returns the first of equal maxima
        remaining[best] = -np.inf
        tokens.append(best)
    tokens = np.array(tokens, dtype=np.int64)
    return tokens, x[tokens] - lse


def candidates(draft_logits: np.ndarray, K: int):
    """depth_candidates for every (sequence, depth): ([B][Dmax][K] tokens, fp64 logp)."""
    B, Dmax, _ = draft_logits.shape
    tok = np.empty((B, Dmax, K), dtype=np.int64)
    lp = np.empty((B, Dmax, K), dtype=np.float64)
    for b in range(B):
        for d in range(Dmax):
            tok[b, d], lp[b, d] = depth_candidates(draft_logits[b, d], K)
    return tok, lp


def best_first_tree(cand_token: np.ndarray, cand_logp: np.ndarray, N: int, root_token: int = -1):
    """Best-first expansion of one sequence's candidate lattice to N nodes.

    cand_token / cand_logp: [Dmax][K]; scores accumulate in fp64 from the root (score 0),
    child score = parent score + cand_logp[depth][rank].  A priority queue holds the
    frontier keyed by (-score, depth, rank path); each pop becomes the next node id and
    pushes its K children.  Returns (parent, draft, depth, score[float64], rank path) with
    N entries each; rank path i is the tuple of candidate ranks from the root to node i."""
    Dmax, K = cand_token.shape
    lp = np.asarray(cand_logp, dtype=np.float64)
    heap = [(-0.0, 0, (), -1)]
    parent, draft, depth, score, paths = [], [], [], [], []
    while heap and len(parent) < N:
        neg, d, ranks, par = heapq.heappop(heap)
        node = len(parent)
        s = -neg
        parent.append(par)
        depth.append(d)
        score.append(s)
        paths.append(ranks)
        draft.append(root_token if d == 0 else int(cand_token[d - 1, ranks[-1]]))
        if d < Dmax:
            for r in range(K):
                heapq.heappush(heap, (-(s + float(lp[d, r])), d + 1, ranks + (r,), node))
    return (np.array(parent, np.int32), np.array(draft, np.int32), np.array(depth, np.int32),
            np.array(score, np.float64), paths)


def path_score(cand_logp: np.ndarray, ranks) -> float:
    """fp64 cumulative log-probability of the node with this rank path (root: 0), summed
    from the root in the same order as best_first_tree."""
    s = 0.0
    for d, r in enumerate(ranks):
        s = s + float(cand_logp[d, r])
    return s
