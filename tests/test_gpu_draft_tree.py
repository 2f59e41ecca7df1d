"""GPU parity for best-first draft-tree construction (jf_build_draft_tree through the C ABI).

Candidates: tokens bit-exact against the fp64 oracle, log-probabilities within 5e-5
(the kernel's log-sum-exp is fp32).  Tree: the expansion decides integers (node order,
parents) from fp32 scores, so the oracle expands the kernel's own fp32 candidate
log-probabilities in fp32, and parent, draft, depth and score must match exactly."""
import numpy as np
import pytest
import torch

from oracle import draft_tree as odt
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
LOGP_ATOL = 5e-5


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


def check(jf, logits_np, dtype, K, N):
    B = logits_np.shape[0]
    roots = list(range(100, 100 + B))
    (parent, draft, depth, score, ctok, clp), ref_in = run(jf, logits_np, dtype, K, N, roots)
    rtok, rlp = odt.candidates(ref_in, K)
    assert (ctok == rtok).all(), "candidate tokens differ"
    assert np.abs(clp.astype(np.float64) - rlp).max() <= LOGP_ATOL
    for b in range(B):
        rp, rd, rdep, rs = odt.best_first_tree(ctok[b], clp[b], N, root_token=roots[b])
        assert (parent[b] == rp).all() and (draft[b] == rd).all()
        assert (depth[b] == rdep).all() and (score[b] == rs).all()


def test_budget_256_vocab_151936_bf16(jf):
    check(jf, wl.draft_logits(2, 16, 151936, seed=1), "bf16", 8, 256)


@pytest.mark.parametrize("B,Dmax,V,K,N,seed", [(3, 5, 1000, 4, 60, 2), (2, 16, 4096, 8, 200, 3),
                                               (1, 9, 333, 3, 100, 4)])
def test_shapes_fp32(jf, B, Dmax, V, K, N, seed):
    check(jf, wl.draft_logits(B, Dmax, V, dtype="f32", seed=seed), "f32", K, N)


def test_chain_and_star(jf):
    check(jf, wl.draft_logits(1, 16, 5000, seed=5), "bf16", 1, 17)      # K = 1: a chain
    check(jf, wl.draft_logits(2, 1, 300, seed=6), "bf16", 8, 9)         # Dmax = 1: a star


def test_equal_logits_and_scores_tie_break(jf):
    """Integer logits in [-2, 2]: many equal tokens and equal cumulative scores."""
    rng = np.random.default_rng(8)
    x = rng.integers(-2, 3, size=(2, 6, 700)).astype(np.float32)
    check(jf, x, "f32", 6, 150)


@pytest.mark.parametrize("B,N", [(20, 64), (8, 256)])
def test_many_rows_bf16(jf, B, N):
    """16 depths for 20 (8) sequences: 320 (128) logit rows, so rows run one CTA each
    (three CTAs per row) instead of eight-CTA clusters."""
    check(jf, wl.draft_logits(B, 16, 151936, seed=9 + B), "bf16", 8, N)


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
