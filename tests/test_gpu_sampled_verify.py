"""GPU parity for lossless (stochastic) tree verification (jf_tree_verify_sampled through
the C ABI) against the fp64 oracle, on the same seeded logits, trees and random numbers.

Each decision compares a drawn threshold with a probability.  The kernel's probabilities
carry a relative error of about 1e-6 (fp32 chunk sums of exponentials), and its residual
CDF an absolute error below about 1e-6 of the residual mass.  So:
  - when every accept/reject decision of a sequence lies further than 1e-5 (relative to
    the residual mass) from its boundary, the accepted length and path must equal the
    oracle's;
  - the bonus token must then equal the oracle's when its draw lies further than 1e-5 from
    a CDF step, and otherwise (common over 151936 tokens, where one token holds about 7e-6
    of the mass) lie in the right place: the drawn threshold inside the token's exact fp64
    CDF interval, widened by 1e-6;
  - a sequence with a closer accept/reject decision (rare) is checked for validity only."""
import numpy as np
import pytest
import torch

from oracle import sampled_verify as osv
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
MARGIN = 1e-5


@pytest.fixture(scope="module")
def jf():
    from tree_speculative_decoding_jf_gb300 import build
    build.build()
    from tree_speculative_decoding_jf_gb300 import jf as mod
    return mod


def logits_tensor(x, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()


def check(jf, logits, dtype, draft, parent, T, seed, min_exact=0.9):
    B, N = parent.shape
    u, bu = wl.sampling_uniforms(B, N, seed)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, path, bonus = jf.tree_verify_sampled(
        logits_tensor(logits, dtype), torch.from_numpy(np.ascontiguousarray(draft, np.int32)).cuda(),
        torch.from_numpy(np.ascontiguousarray(parent, np.int32)).cuda(), torch.from_numpy(u).cuda(),
        torch.from_numpy(bu).cuda(), T, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    acc, path, bonus = acc.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy()
    racc, rpath, rbonus, margins = osv.tree_verify_sampled(logits, dtype, draft, parent, u, bu, T)
    rows = osv._rows_f64(logits, dtype)
    V = logits.shape[-1]
    exact = 0
    for b in range(B):
        walk = [m for k, _, m in margins[b] if k != "bonus"]
        bonus_margin = [m for k, _, m in margins[b] if k == "bonus"][0]
        if not walk or min(walk) > MARGIN:
            assert acc[b] == racc[b] and (path[b] == rpath[b]).all(), b
            exact += 1
            if bonus_margin > MARGIN:
                assert bonus[b] == rbonus[b], b
            else:                               # the draw sits within a CDF step of y
                f = path[b, acc[b]]
                r = osv.target_probs(rows[b, f], T)
                for c in np.flatnonzero(parent[b] == f):
                    r[draft[b, c]] = 0.0
                cdf = np.cumsum(r)
                y = int(bonus[b])
                target = float(bu[b]) * r.sum()
                lo = cdf[y - 1] if y > 0 else 0.0
                tol = 1e-6 * r.sum()
                assert r[y] > 0 and lo - tol <= target <= cdf[y] + tol, (b, y, rbonus[b])
        else:                                   # a near-boundary decision: validity only
            n = acc[b]
            assert path[b, 0] == 0 and (path[b, n + 1:] == -1).all()
            assert all(parent[b, path[b, k + 1]] == path[b, k] for k in range(n))
            assert 0 <= bonus[b] < V
    assert exact >= min_exact * B, f"only {exact} of {B} sequences decided away from boundaries"
    return racc


@pytest.mark.parametrize("T", [0.7, 1.0, 2.5])
def test_small_vocab_mixed_decisions(jf, T):
    """V = 8, each child's token drawn from its parent's target distribution: acceptances
    and rejections mix, paths chain, and the residual bonus draw matters."""
    rng = np.random.default_rng(int(T * 10))
    B, N, V = 32, 48, 8
    parent = np.stack([np.array([-1] + [rng.integers(max(0, i - 5), i) for i in range(1, N)])
                       for _ in range(B)]).astype(np.int32)
    logits = (rng.standard_normal((B, N, V)) * 1.5).astype(np.float32)
    draft = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            p = osv.target_probs(logits[b, parent[b, c]].astype(np.float64), T)
            draft[b, c] = rng.choice(V, p=p)
    racc = check(jf, logits, "f32", draft, parent, T, seed=int(T * 10))
    assert racc.max() >= 2


@pytest.mark.parametrize("V,dtype", [(1001, "bf16"), (8195, "f32"), (20000, "bf16"), (16384, "f32")])
def test_vocab_shapes_mixed_decisions(jf, V, dtype):
    """Vocabularies of one to three 8192-token chunks, with a ragged last chunk and with
    rows that do not start on a 16-byte boundary (1001 bf16, 8195 fp32): children drawn
    from their parent's target distribution, so acceptances, rejections and residual bonus
    draws across the chunks all occur."""
    rng = np.random.default_rng(V)
    B, N, T = 6, 24, 1.0
    parent = np.stack([np.array([-1] + [rng.integers(max(0, i - 4), i) for i in range(1, N)])
                       for _ in range(B)]).astype(np.int32)
    x = (rng.standard_normal((B, N, V)) * 2.0).astype(np.float32)
    logits = wl.to_bf16_bits(x) if dtype == "bf16" else x
    rows = osv._rows_f64(logits, dtype)
    draft = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            draft[b, c] = rng.choice(V, p=osv.target_probs(rows[b, parent[b, c]], T))
    check(jf, logits, dtype, draft, parent, T, seed=V)


@pytest.mark.parametrize("dtype,V", [("f32", 1001), ("bf16", 1000)])
def test_largest_trees(jf, dtype, V):
    """4096 nodes (the most a call takes): the walk's shared memory is at its largest."""
    rng = np.random.default_rng(V)
    B, N, T = 2, 4096, 1.0
    parent = np.stack([np.array([-1] + [rng.integers(max(0, i - 6), i) for i in range(1, N)])
                       for _ in range(B)]).astype(np.int32)
    x = (rng.standard_normal((B, N, V)) * 2.0).astype(np.float32)
    logits = wl.to_bf16_bits(x) if dtype == "bf16" else x
    rows = osv._rows_f64(logits, dtype)
    draft = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            draft[b, c] = rng.choice(V, p=osv.target_probs(rows[b, parent[b, c]], T))
    check(jf, logits, dtype, draft, parent, T, seed=V)


@pytest.mark.parametrize("name", ["c1_tiny_random16", "c3_qwen3_8b_tree256"])
def test_workloads_forced_drafts(jf, name):
    """Workload logits with half the children's tokens planted as their parent's maximum
    (probability close to 1): long accepted paths, then a bonus drawn from the residual of
    the full vocabulary (151936 bf16 logits on workload 3)."""
    w = wl.config(name, forcing="half")
    racc = check(jf, w.logits, w.logits_dtype, w.draft, w.parent, 1.0, seed=3)
    assert racc.max() >= 1


def test_chain_with_five_planted_acceptances(jf):
    w = wl.config("c2_qwen3_8b_chain16")
    racc = check(jf, w.logits, w.logits_dtype, w.draft, w.parent, 1.0, seed=4)
    assert (racc == 5).all()


def test_low_temperature_is_the_greedy_walk(jf):
    """T -> 0: the stochastic rule accepts exactly the children whose token is the parent's
    argmax and the bonus is the argmax (distinct sibling tokens)."""
    w = wl.config("c1_tiny_random16", forcing="half")
    logits = w.logits.astype(np.float32)
    B, N = w.parent.shape
    draft = w.draft.copy()
    for b in range(B):
        for p_ in range(N):
            kids = np.flatnonzero(w.parent[b] == p_)
            seen = set()
            for c in kids:
                while int(draft[b, c]) in seen:
                    draft[b, c] = (draft[b, c] + 1) % w.V
                seen.add(int(draft[b, c]))
    u, bu = wl.sampling_uniforms(B, N, 5)
    acc, path, bonus = jf.tree_verify_sampled(
        logits_tensor(logits, "f32"), torch.from_numpy(draft).cuda(),
        torch.from_numpy(w.parent).cuda(), torch.from_numpy(np.clip(u, 0.01, 0.99)).cuda(),
        torch.from_numpy(np.clip(bu, 0.01, 0.99)).cuda(), 1e-4)
    am, gacc, gpath, gbonus = jf.tree_verify(logits_tensor(logits, "f32"), torch.from_numpy(draft).cuda(),
                                             torch.from_numpy(w.parent).cuda())
    torch.cuda.synchronize()
    assert (acc.cpu() == gacc.cpu()).all() and (path.cpu() == gpath.cpu()).all()
    assert (bonus.cpu() == gbonus.cpu()).all()


def test_reports_bad_tokens(jf):
    lg = torch.randn(1, 4, 50, device="cuda")
    par = torch.tensor([[-1, 0, 0, 1]], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    u = torch.full((1, 4), 0.5, device="cuda")
    jf.tree_verify_sampled(lg, torch.tensor([[0, 3, 99, 1]], dtype=torch.int32, device="cuda"), par,
                           u, torch.full((1,), 0.5, device="cuda"), 1.0, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == jf.DEVERR_BAD_TOKEN


# ----------------------------------------------------------------------------- ragged / packed

@pytest.mark.parametrize("V,dtype,T", [(1000, "f32", 1.0), (151936, "bf16", 0.7), (4097, "bf16", 1.3)])
def test_ragged_and_packed_equal_the_per_sequence_calls(jf, V, dtype, T):
    """Per-sequence tree sizes: the ragged call (padded arrays, hostile padding) and the
    packed call (cu_seqlens) give every sequence exactly what jf_tree_verify_sampled gives
    on that sequence's first n_b nodes with the same random numbers (same arithmetic per
    row, so bit for bit); the fixed-size call is itself checked against the oracle above."""
    B, N = 5, 40
    w = wl.make_workload(f"sr{V}", B, N, 1, 1, 64, V, 8, tree="random_depth_limited",
                         logits_dtype=dtype, forcing="half", seed=V % 97)
    tree_len = [1, 2, 17, 39, 40]
    u, bu = wl.sampling_uniforms(B, N, 5)
    draft, parent = w.draft.copy(), w.parent.copy()
    uni = u.copy()
    for b, n in enumerate(tree_len):             # padding: out of range, never read
        draft[b, n:] = -3
        parent[b, n:] = 10 ** 6
        uni[b, n:] = np.nan
    lg = logits_tensor(w.logits, dtype)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()   # noqa: E731
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.empty((B, N), dtype=torch.int32, device="cuda")
    bonus = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(jf.jf_tree_verify_workspace_size(B, N, V), dtype=torch.uint8, device="cuda")
    jf.jf_tree_verify_sampled_ragged(lg, dev(draft), dev(parent), dev(np.array(tree_len, np.int32)),
                                     dev(uni), dev(bu), T, acc, path, bonus, ws, err)
    # packed
    cu = np.concatenate([[0], np.cumsum(tree_len)]).astype(np.int32)
    Tn = int(cu[-1])
    pk = lambda a: np.ascontiguousarray(np.concatenate([a[b, :n] for b, n in enumerate(tree_len)]))  # noqa: E731
    acc_p = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    path_p = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    bonus_p = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ws_p = torch.empty(jf.jf_tree_verify_packed_workspace_size(Tn, V), dtype=torch.uint8,
                       device="cuda")
    jf.jf_tree_verify_sampled_packed(logits_tensor(pk(w.logits), dtype), dev(pk(draft)),
                                     dev(pk(parent)), dev(cu), N, dev(pk(uni)), dev(bu), T, acc_p,
                                     path_p, bonus_p, ws_p, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(acc, acc_p) and torch.equal(path, path_p) and torch.equal(bonus, bonus_p)
    acc, path, bonus = acc.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy()
    for b, n in enumerate(tree_len):
        r_acc, r_path, r_bonus = jf.tree_verify_sampled(
            logits_tensor(w.logits[b:b + 1, :n], dtype), dev(draft[b:b + 1, :n]),
            dev(parent[b:b + 1, :n]), dev(u[b:b + 1, :n]), dev(bu[b:b + 1]), T)
        assert acc[b] == r_acc.item() and bonus[b] == r_bonus.item(), b
        assert (path[b, :n] == r_path.cpu().numpy()[0]).all() and (path[b, n:] == -1).all()
    assert acc.max() >= 1


def test_packed_bad_span_is_reported_and_not_read(jf):
    B, N, V = 2, 8, 300
    w = wl.make_workload("sbad", B, N, 1, 1, 64, V, 8, tree="random_depth_limited",
                         logits_dtype="f32", forcing="half", seed=3)
    cu = torch.tensor([0, 9, 11], dtype=torch.int32, device="cuda")     # 9 > N_max: bad
    Tn = 11
    lg = torch.from_numpy(np.ascontiguousarray(w.logits.reshape(B * N, V)[:Tn])).cuda()
    u, bu = wl.sampling_uniforms(B, N, 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    bonus = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    par = np.concatenate([w.parent[0], [0], w.parent[1, :2]]).astype(np.int32)
    dr = np.concatenate([w.draft[0], [0], w.draft[1, :2]]).astype(np.int32)
    ws = torch.empty(jf.jf_tree_verify_packed_workspace_size(Tn, V), dtype=torch.uint8,
                     device="cuda")
    jf.jf_tree_verify_sampled_packed(lg, torch.from_numpy(dr).cuda(), torch.from_numpy(par).cuda(),
                                     cu, N, torch.from_numpy(u.reshape(-1)[:Tn].copy()).cuda(),
                                     torch.from_numpy(bu).cuda(), 1.0, acc, path, bonus, ws, err)
    torch.cuda.synchronize()
    assert err.item() & jf.DEVERR_BAD_TREE_LEN
    assert acc[0].item() == 0 and bonus[0].item() == -1
    assert path[0, 0].item() == 0 and (path[0, 1:] == -1).all()
    assert 0 <= bonus[1].item() < V and path[1, 0].item() == 0
