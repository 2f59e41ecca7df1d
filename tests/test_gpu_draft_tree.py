"""GPU parity for best-first draft-tree construction (jf_build_draft_tree through the C ABI).

Everything expected comes from the fp64 oracle run on the logits alone: no value the
kernel produced is fed back into the oracle.

Candidates: tokens bit-exact, log-probabilities within 5e-5 of fp64 (the kernel's
log-sum-exp is fp32).  Tree: the kernel orders nodes by fp32 cumulative scores, the
oracle by fp64 ones, so two nodes whose exact scores lie within the scores' error bound
may legitimately come out in either order.  The test therefore
  - checks that the GPU tree is well formed (parents earlier, depths, each node's token
    is the candidate of its rank at its depth, no rank path twice),
  - recomputes every GPU node's exact score from its rank path and the oracle's fp64
    log-probs, and checks the GPU's score against it,
  - checks that the GPU's node order and node set are best-first under the exact scores
    up to swaps of nodes closer than the error bound,
  - cuts the oracle's ranking into near-tie clusters (runs of consecutive exact scores
    within the bound) and requires the GPU to hold exactly the oracle's nodes at each
    cluster's positions, in any order, and at the cluster that straddles the budget only
    nodes of that cluster; where a cluster's scores are exactly equal in fp64 and in the
    kernel's fp32, the tie rule (depth, then rank path) must give the GPU's order.
Score error bound per node: 6e-5 x depth (each candidate log-prob within 5e-5, plus fp32
rounding of a running sum of at most 16 terms of magnitude below 100)."""
import numpy as np
import pytest
import torch

from oracle import draft_tree as odt
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
LOGP_ATOL = 5e-5
SCORE_TOL_PER_DEPTH = 6e-5


@pytest.fixture(scope="module")
def jf():
    from tree_speculative_decoding_jf_gb300 import build
    build.build()
    from tree_speculative_decoding_jf_gb300 import jf as mod
    return mod


def run(jf, logits_np, dtype, K, N, roots):
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(logits_np).view(np.int16)).view(torch.bfloat16).cuda()
        ref_in = wl.bf16_bits_to_f32(logits_np)
    else:
        t = torch.from_numpy(np.ascontiguousarray(logits_np, np.float32)).cuda()
        ref_in = logits_np
    rt = torch.tensor(roots, dtype=torch.int32, device="cuda")
    parent, draft, depth, score, ctok, clp = jf.build_draft_tree(t, K, N, root_token=rt)
    torch.cuda.synchronize()
    return ([x.cpu().numpy() for x in (parent, draft, depth, score, ctok, clp)], ref_in)


def tol(d):
    return SCORE_TOL_PER_DEPTH * max(int(d), 1)


def gpu_rank_paths(parent, draft, depth, rtok, root):
    """Rank path of every GPU node, rebuilt from its parent and token against the oracle's
    candidate lists; asserts the tree is well formed on the way."""
    N = len(parent)
    assert parent[0] == -1 and depth[0] == 0 and draft[0] == root
    paths = [()]
    for i in range(1, N):
        p = int(parent[i])
        assert 0 <= p < i, f"node {i}: parent {p}"
        assert depth[i] == depth[p] + 1 and depth[i] <= rtok.shape[0]
        hits = np.flatnonzero(rtok[depth[i] - 1] == draft[i])
        assert len(hits) == 1, f"node {i}: token {draft[i]} is not a depth-{depth[i]} candidate"
        paths.append(paths[p] + (int(hits[0]),))
    assert len(set(paths)) == N, "a rank path occurs twice"
    return paths


def check_tree(parent, draft, depth, score, rtok, rlp, N, root):
    """Returns the number of positions pinned to the oracle's tree (see the module doc)."""
    Dmax, K = rtok.shape
    paths = gpu_rank_paths(parent, draft, depth, rtok, root)
    exact = np.array([odt.path_score(rlp, p) for p in paths])
    err = np.abs(score.astype(np.float64) - exact)
    assert all(err[i] <= tol(depth[i]) for i in range(N)), f"score error {err.max():.2e}"
    # order: best-first up to near-ties
    for i in range(1, N - 1):
        assert exact[i] >= exact[i + 1] - tol(depth[i]) - tol(depth[i + 1]), f"order at {i}"
    # set: no frontier node beats a chosen one by more than the bound
    chosen = set(paths)
    front = [p + (r,) for p in paths if len(p) < Dmax for r in range(K) if p + (r,) not in chosen]
    if front and N > 1:
        fs = np.array([odt.path_score(rlp, p) for p in front])
        fb = int(fs.argmax())
        worst = int(np.argmin(exact[1:])) + 1
        assert fs[fb] <= exact[worst] + tol(len(front[fb])) + tol(depth[worst]), "not best-first"
    # Near-tie clusters of the oracle's ranking (consecutive exact scores within the bound),
    # taken past the budget until the cluster at the boundary is complete.
    extra = 64
    while True:
        _, _, rdep, rs, rpaths = odt.best_first_tree(rtok, rlp, N + extra, root_token=root)
        near = [rs[i] - rs[i + 1] <= tol(rdep[i]) + tol(rdep[i + 1]) for i in range(len(rs) - 1)]
        j = N - 1
        while j < len(near) and near[j]:
            j += 1
        if j < len(near) or len(rs) < N + extra:
            break
        extra *= 2
    assert paths[0] == rpaths[0] == ()
    pinned, a = 1, 1
    while a < N:
        b = a + 1
        while b < len(rs) and near[b - 1]:
            b += 1
        if b <= N:       # a cluster inside the budget: the same nodes, in any order
            assert set(paths[a:b]) == set(rpaths[a:b]), f"positions {a}..{b - 1} hold other nodes"
            pinned += b - a
            # exactly tied in fp64 and in the kernel's fp32: the tie rule decides the order
            if b - a > 1 and len(set(rs[a:b])) == 1 and len(set(score[a:b].tolist())) == 1:
                keys = [(len(p), p) for p in paths[a:b]]
                assert keys == sorted(keys), f"tie order at {a}..{b - 1}"
        else:            # the cluster at the budget boundary: any of its nodes may be chosen
            assert set(paths[a:N]) <= set(rpaths[a:b]), f"positions {a}..{N - 1} outside the boundary cluster"
        a = b
    return pinned


def check(jf, logits_np, dtype, K, N, min_pinned=0.0):
    B = logits_np.shape[0]
    roots = list(range(100, 100 + B))
    (parent, draft, depth, score, ctok, clp), ref_in = run(jf, logits_np, dtype, K, N, roots)
    rtok, rlp = odt.candidates(ref_in, K)
    assert (ctok == rtok).all(), "candidate tokens differ"
    assert np.abs(clp.astype(np.float64) - rlp).max() <= LOGP_ATOL
    pinned = 0
    for b in range(B):
        pinned += check_tree(parent[b], draft[b], depth[b], score[b], rtok[b], rlp[b], N, roots[b])
    assert pinned >= min_pinned * B * N, f"only {pinned} of {B * N} positions pinned exactly"


def test_budget_256_vocab_151936_bf16(jf):
    check(jf, wl.draft_logits(2, 16, 151936, seed=1), "bf16", 8, 256, min_pinned=0.8)


@pytest.mark.parametrize("B,Dmax,V,K,N,seed", [(3, 5, 1000, 4, 60, 2), (2, 16, 4096, 8, 200, 3),
                                               (1, 9, 333, 3, 100, 4)])
def test_shapes_fp32(jf, B, Dmax, V, K, N, seed):
    check(jf, wl.draft_logits(B, Dmax, V, dtype="f32", seed=seed), "f32", K, N, min_pinned=0.8)


def test_chain_and_star(jf):
    check(jf, wl.draft_logits(1, 16, 5000, seed=5), "bf16", 1, 17)      # K = 1: a chain
    check(jf, wl.draft_logits(2, 1, 300, seed=6), "bf16", 8, 9)         # Dmax = 1: a star


def test_equal_logits_and_scores_tie_break(jf):
    """Integer logits in [-2, 2]: many equal tokens and equal cumulative scores."""
    rng = np.random.default_rng(8)
    x = rng.integers(-2, 3, size=(2, 6, 700)).astype(np.float32)
    check(jf, x, "f32", 6, 150)


@pytest.mark.parametrize("V", [704, 700])
def test_equal_bf16_logits_tie_break(jf, V):
    """The same integer logits as bf16: rows of 704 logits start on 16-byte boundaries and
    take the packed passes (whole vectors tie at the threshold), rows of 700 do not."""
    rng = np.random.default_rng(18)
    x = rng.integers(-2, 3, size=(3, 6, V)).astype(np.float32)
    check(jf, wl.to_bf16_bits(x), "bf16", 6, 150)


@pytest.mark.parametrize("B,Dmax,V,K,N,dtype", [(2, 6, 3000, 5, 200, "bf16"), (1, 10, 2000, 3, 256, "f32"),
                                                (3, 16, 8192, 7, 256, "bf16")])
def test_levels_with_many_candidates(jf, B, Dmax, V, K, N, dtype):
    """Levels with more than 64 candidates from parent counts that are not powers of two
    (25 parents of 5 children, 27 of 3, 49 of 7): their children are merged as sorted runs
    before the chosen set is updated."""
    check(jf, wl.draft_logits(B, Dmax, V, sigma=1.0, dtype=dtype, seed=30 + K), dtype, K, N, min_pinned=0.8)


@pytest.mark.parametrize("B,N", [(20, 64), (8, 256), (32, 64)])
def test_many_rows_bf16(jf, B, N):
    """16 depths for 20 (8, 32) sequences: 320 (128, 512) logit rows, so rows run one CTA
    each (three CTAs per row) instead of eight-CTA clusters; 512 rows are more than one
    wave at three CTAs per SM and take the two-per-SM instantiation."""
    V = 151936 if B < 32 else 8192
    check(jf, wl.draft_logits(B, 16, V, seed=9 + B), "bf16", 8, N, min_pinned=0.8)


@pytest.mark.parametrize("B,Dmax,V", [(2, 4, 20000), (20, 16, 3000)])
def test_two_valued_logits_overflow_the_filter(jf, B, Dmax, V):
    """Logits in {0, 1}: about half of every slice ties at the threshold, more than the
    candidate buffer holds, so the exact per-warp ranking runs (in clusters and with one
    CTA per row)."""
    rng = np.random.default_rng(B * 100 + V)
    x = rng.integers(0, 2, size=(B, Dmax, V)).astype(np.float32)
    check(jf, x, "f32", 8, 30)


def test_lattice_smaller_than_budget_is_rejected(jf):
    x = torch.zeros((1, 2, 10), dtype=torch.float32, device="cuda")
    with pytest.raises(RuntimeError):
        jf.build_draft_tree(x, 2, 8)                 # 1 + 2 + 4 = 7 < 8 nodes


@pytest.mark.parametrize("B,Dmax,V,K,N,dtype", [(4, 16, 32000, 8, 64, "bf16"),
                                                 (6, 12, 151936, 8, 256, "bf16"),
                                                 (3, 5, 1000, 4, 40, "f32")])
def test_ragged_budgets_are_prefixes_of_the_full_tree(jf, B, Dmax, V, K, N, dtype):
    """Best-first expansion pops nodes in an order that does not depend on the budget, so
    the tree of budget n is the first n nodes of the tree of budget N: with per-sequence
    budgets, sequence b's nodes 0 .. n_b - 1 must equal the fixed-size call's bit for bit
    (same candidates: same call shape) and the rest be padding.  Budgets outside [1, N]
    are reported and clamped."""
    rng = np.random.default_rng(B * 100 + N)
    logits = wl.draft_logits(B, Dmax, V, seed=N + V % 13, dtype=dtype)
    t = (torch.from_numpy(np.ascontiguousarray(logits).view(np.int16)).view(torch.bfloat16)
         if dtype == "bf16" else torch.from_numpy(np.ascontiguousarray(logits, np.float32))).cuda()
    rt = torch.from_numpy(rng.integers(0, V, B).astype(np.int32)).cuda()
    full = jf.build_draft_tree(t, K, N, root_token=rt)
    budgets = rng.integers(1, N + 1, B).astype(np.int32)
    budgets[0], budgets[-1] = 0, N + 5                   # out of range: clamped to 1 and N
    want = np.clip(budgets, 1, N)
    out = dict(cand_token=torch.empty((B, Dmax, K), dtype=torch.int32, device="cuda"),
               cand_logp=torch.empty((B, Dmax, K), dtype=torch.float32, device="cuda"),
               parent=torch.full((B, N), 7, dtype=torch.int32, device="cuda"),
               draft=torch.full((B, N), 7, dtype=torch.int32, device="cuda"),
               depth=torch.full((B, N), 7, dtype=torch.int32, device="cuda"),
               score=torch.zeros((B, N), dtype=torch.float32, device="cuda"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    jf.jf_build_draft_tree_ragged(t, K, N, torch.from_numpy(budgets).cuda(), out["cand_token"],
                                  out["cand_logp"], out["parent"], out["draft"], out["depth"],
                                  root_token=rt, score=out["score"], dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == jf.DEVERR_BAD_TREE_LEN
    f_par, f_dr, f_dep, f_sc, f_tok, f_lp = [x.cpu().numpy() for x in full]
    g = {k: v.cpu().numpy() for k, v in out.items()}
    assert (g["cand_token"] == f_tok).all() and (g["cand_logp"] == f_lp).all()
    for b, n in enumerate(want):
        assert (g["parent"][b, :n] == f_par[b, :n]).all(), b
        assert (g["draft"][b, :n] == f_dr[b, :n]).all() and (g["depth"][b, :n] == f_dep[b, :n]).all()
        assert (g["score"][b, :n] == f_sc[b, :n]).all()
        assert (g["parent"][b, n:] == -1).all() and (g["draft"][b, n:] == -1).all()
        assert (g["depth"][b, n:] == -1).all() and np.isneginf(g["score"][b, n:]).all()
