"""Seeded random attention shapes against the fp64 oracle, through the C ABI.

The planner picks among several dispatches (one CTA per unit, key splits merged in a
cluster or by the combine kernel, longest-first order, stream-K ranges) from B, N, G, Hkv,
D and the prefix lengths; fixed test shapes reach each of them once.  These cases draw the
shapes at random (fixed seeds) so that the dispatch boundaries, odd row counts, mixed
prefix lengths (including empty ones) and deep or flat trees meet in combinations nobody
picked by hand.  Every row is compared when there are few, else a sample that includes
each sequence's root, last and deepest node.

JF_FUZZ_SCALE=k (default 1) runs k times as many cases of each kind: the first cases are
the default ones, the rest new seeds."""
import os

import numpy as np
import pytest
import torch

import oracle
from tree_speculative_decoding_jf_gb300 import workloads as wl
from test_gpu_parity import assert_attention_close, gpu_attention, jf, sample_rows  # noqa: F401 (fixture)

pytestmark = pytest.mark.gpu

SCALE = max(1, int(os.environ.get("JF_FUZZ_SCALE", "1")))
N_CASES = 48 * SCALE


def draw(case):
    rng = np.random.default_rng(9000 + case)
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    B = int(rng.choice([1, 2, 3, 5, 8, 13, 24, 40]))
    N = int(rng.choice([1, 7, 16, 33, 64, 100, 200, 256]))
    while B * N * G * Hkv > 120000:                      # keep the oracle's share small
        B = max(1, B // 2)
        N = max(1, N // 2)
    prefix = rng.integers(0, 3000, B).astype(np.int32)
    prefix[rng.random(B) < 0.15] = 0                     # some sequences without prefix
    prefix[rng.random(B) < 0.15] = rng.integers(1, 4)    # and some of 1..3 keys
    kind = rng.choice(["window", "chain", "star", "deep"])
    parents = []
    for _ in range(B):
        if kind == "chain":
            par = np.arange(-1, N - 1)
        elif kind == "star":
            par = np.array([-1] + [0] * (N - 1))
        else:
            width = 2 if kind == "deep" else int(rng.integers(2, 9))
            par = np.array([-1] + [rng.integers(max(0, i - width), i) for i in range(1, N)])
        parents.append(par.astype(np.int32))
    parent = np.stack(parents)
    w = wl.make_workload(f"fuzz{case}", B, N, G * Hkv, Hkv, D, 64, prefix, tree="chain",
                         parent=parent, permute_pages=bool(rng.random() < 0.7), seed=case,
                         with_logits=False)
    return w


@pytest.mark.parametrize("case", range(N_CASES))
def test_attention_random_shapes(jf, case):
    w = draw(case)
    out, lse, err = gpu_attention(jf, w)
    assert err == 0
    assert np.isfinite(out).all()
    nrows = w.B * w.N * w.Hq
    rows = oracle.all_rows(w) if nrows <= 6144 else sample_rows(w, 1536, seed=case)
    assert_attention_close(w, out, lse, rows)


def test_fuzz_shapes_cover_the_dispatches():
    """The draw reaches stream-K-sized calls (units >= 152 with two or more row-tile groups
    per kv-head), single-unit calls and both head dims (checked on the shapes alone)."""
    shapes = [draw(c) for c in range(N_CASES)]
    def units(w):
        mt = -(-w.N * (w.Hq // w.Hkv) // 128)
        groups = -(-mt // 2) if mt >= 2 else mt
        return w.B * w.Hkv * groups, groups
    assert any(units(w)[0] >= 152 and units(w)[1] >= 2 for w in shapes)
    assert any(units(w)[0] == 1 for w in shapes) or any(units(w)[0] < 8 for w in shapes)
    assert {w.D for w in shapes} == {64, 128}


# ----------------------------------------------------------------------------- ragged

N_RAGGED = 16 * SCALE


@pytest.mark.parametrize("case", range(N_RAGGED))
def test_ragged_attention_random_shapes(jf, case):
    """Random shapes again, now with a random tree size per sequence (some one-node, some
    full) and hostile padding (out-of-range parents, NaN K/V in the padding slots, -1 block
    table past the needed pages); rows of the first n_b nodes against the oracle run on
    each sequence's slice."""
    from test_gpu_ragged import check_rows, poison_padding, ragged_attention
    w = draw(100 + case)
    rng = np.random.default_rng(7000 + case)
    tree_len = [int(x) for x in rng.integers(1, w.N + 1, w.B)]
    tree_len[0] = w.N
    if w.B > 1:
        tree_len[-1] = 1
    w = poison_padding(w, tree_len)
    out, lse, err = ragged_attention(jf, w, tree_len)
    assert err == 0
    check_rows(w, tree_len, out, lse, rows_per_seq=24 if w.B > 8 else 96, seed=case)


# ----------------------------------------------------------------------------- verify

N_VERIFY = 24 * SCALE


@pytest.mark.parametrize("case", range(N_VERIFY))
def test_verify_random_shapes(jf, case):
    """Greedy verification on random trees, vocabularies (odd sizes: unaligned rows and
    chunk tails), both logit types, with about half of the nodes forced to be accepted
    (their draft token is the parent's planted maximum): argmax, accepted length, path and
    bonus bit-exact against the oracle."""
    from test_gpu_parity import assert_verify_matches
    rng = np.random.default_rng(5000 + case)
    V = int(rng.choice([7, 33, 1000, 4097, 32001, 151936]))
    N = int(rng.choice([1, 2, 16, 64, 100, 256, 700]))
    B = int(rng.choice([1, 2, 5, 16]))
    while B * N * V > 60_000_000:
        if B > 1:
            B //= 2
        else:
            N = max(1, N // 2)
    width = int(rng.integers(1, 10))
    parent = np.stack([np.array([-1] + [rng.integers(max(0, i - width), i) for i in range(1, N)],
                                np.int32) for _ in range(B)])
    w = wl.make_workload(f"vfuzz{case}", B, N, 1, 1, 64, V, 8, tree="chain", parent=parent,
                         logits_dtype=str(rng.choice(["bf16", "f32"])), forcing="half",
                         seed=300 + case)
    assert_verify_matches(jf, w)


# ----------------------------------------------------------------------------- draft tree

N_DRAFT = 24 * SCALE


@pytest.mark.parametrize("case", range(N_DRAFT))
def test_draft_tree_random_shapes(jf, case):
    """Best-first draft trees on random shapes (batch, depths, vocabulary, K, budget, dtype,
    logit spread), checked against the oracle as in test_gpu_draft_tree: candidates exact,
    the tree equal to the oracle's up to swaps of near-tied nodes."""
    from test_gpu_draft_tree import check
    rng = np.random.default_rng(4000 + case)
    K = int(rng.integers(1, 9))
    Dmax = int(rng.integers(1, 17))
    lattice, level = 1, 1
    for _ in range(Dmax):
        level *= K
        lattice += level
    N = int(min(lattice, rng.choice([2, 9, 33, 64, 129, 256]), 4096 // (K + 1)))
    B = int(rng.choice([1, 2, 3, 8, 21]))
    V = int(rng.choice([K + 3, 500, 4099, 32000, 151936]))
    while B * Dmax * V > 40_000_000 and B > 1:
        B //= 2
    dtype = str(rng.choice(["bf16", "f32"]))
    sigma = float(rng.choice([0.5, 3.0, 8.0]))
    x = wl.draft_logits(B, Dmax, V, sigma=sigma, dtype=dtype, seed=600 + case)
    check(jf, x, dtype, K, N)


# ----------------------------------------------------------------------------- packed

N_PACKED = 12 * SCALE


@pytest.mark.parametrize("case", range(N_PACKED))
def test_packed_attention_random_shapes(jf, case):
    """Random shapes and tree sizes in the packed (cu_seqlens) layout: masks, outputs and
    LSEs equal the ragged call's bit for bit, rows against the oracle's slices."""
    from test_gpu_packed import ragged_vs_packed_attention
    from test_gpu_ragged import check_rows, poison_padding
    w = draw(200 + case)
    rng = np.random.default_rng(7500 + case)
    tree_len = [int(x) for x in rng.integers(1, w.N + 1, w.B)]
    w = poison_padding(w, tree_len)
    out, lse = ragged_vs_packed_attention(jf, w, tree_len)
    check_rows(w, tree_len, out, lse, rows_per_seq=24 if w.B > 8 else 64, seed=case)


# ----------------------------------------------------------------------------- vocabulary shards

N_SHARD = 12 * SCALE


@pytest.mark.parametrize("case", range(N_SHARD))
def test_sharded_verify_random_shapes(jf, case):
    """Greedy verification with the vocabulary cut into 2-8 random ranges (keys per range,
    merged walk): argmax, accepted length, path and bonus bit-exact against the oracle."""
    from test_gpu_shard_verify import cuts, sharded
    rng = np.random.default_rng(6000 + case)
    V = int(rng.choice([9, 33, 1000, 4097, 32001, 151936]))
    N = int(rng.choice([1, 2, 16, 64, 100, 256]))
    B = int(rng.choice([1, 2, 5, 16]))
    while B * N * V > 40_000_000:
        if B > 1:
            B //= 2
        else:
            N = max(1, N // 2)
    S = int(min(rng.integers(2, 9), V))
    width = int(rng.integers(1, 10))
    parent = np.stack([np.array([-1] + [rng.integers(max(0, i - width), i) for i in range(1, N)],
                                np.int32) for _ in range(B)])
    dtype = str(rng.choice(["bf16", "f32"]))
    w = wl.make_workload(f"sfuzz{case}", B, N, 1, 1, 64, V, 8, tree="chain", parent=parent,
                         logits_dtype=dtype, forcing="half", seed=600 + case)
    lg = (torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16) if dtype == "bf16"
          else torch.from_numpy(w.logits)).cuda()
    ranges = cuts(V, S, rng, ragged=bool(rng.random() < 0.7))
    keys, _ = sharded(jf, lg, ranges, rng.permutation(len(ranges)).tolist())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    am, acc, path, bonus = jf.tree_verify_from_keys(keys, V, torch.from_numpy(w.draft).cuda(),
                                                    torch.from_numpy(w.parent).cuda(), dev_err=err)
    ram = oracle.argmax(w.logits, dtype)
    racc, rpath, rbonus = oracle.tree_walk(ram, w.draft, w.parent)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert (am.cpu().numpy() == ram).all()
    assert (acc.cpu().numpy() == racc).all() and (path.cpu().numpy() == rpath).all()
    assert (bonus.cpu().numpy() == rbonus).all()


# ----------------------------------------------------------------------------- ragged lossless verify

N_SAMPLED_RAGGED = 8 * SCALE


@pytest.mark.parametrize("case", range(N_SAMPLED_RAGGED))
def test_sampled_ragged_and_packed_random_shapes(jf, case):
    """Lossless verification with random tree sizes: the ragged and packed calls give each
    sequence what the fixed-size call gives on its slice, bit for bit."""
    rng = np.random.default_rng(8800 + case)
    V = int(rng.choice([50, 1000, 8193, 32001, 151936]))
    N = int(rng.choice([1, 5, 16, 40, 64, 100]))
    B = int(rng.choice([1, 2, 3, 6]))
    T = float(rng.choice([0.5, 1.0, 1.5]))
    while B * N * V > 30_000_000:
        if B > 1:
            B //= 2
        else:
            N = max(1, N // 2)
    dtype = str(rng.choice(["bf16", "f32"]))
    width = int(rng.integers(1, 8))
    parent = np.stack([np.array([-1] + [rng.integers(max(0, i - width), i) for i in range(1, N)],
                                np.int32) for _ in range(B)])
    w = wl.make_workload(f"srf{case}", B, N, 1, 1, 64, V, 8, tree="chain", parent=parent,
                         logits_dtype=dtype, forcing="half", seed=880 + case)
    tree_len = rng.integers(1, N + 1, B)
    u, bu = wl.sampling_uniforms(B, N, case)
    draft, par = w.draft.copy(), w.parent.copy()
    for b, n in enumerate(tree_len):
        draft[b, n:] = -1
        par[b, n:] = -7
    to_dev = (lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()) \
        if dtype == "bf16" else (lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda())
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()   # noqa: E731
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.empty((B, N), dtype=torch.int32, device="cuda")
    bonus = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(jf.jf_tree_verify_workspace_size(B, N, V), dtype=torch.uint8, device="cuda")
    jf.jf_tree_verify_sampled_ragged(to_dev(w.logits), dev(draft), dev(par),
                                     dev(tree_len.astype(np.int32)), dev(u), dev(bu), T, acc,
                                     path, bonus, ws, err)
    cu = np.concatenate([[0], np.cumsum(tree_len)]).astype(np.int32)
    Tn = int(cu[-1])
    pk = lambda a: np.ascontiguousarray(np.concatenate([a[b, :n] for b, n in enumerate(tree_len)]))  # noqa: E731
    acc_p, path_p, bonus_p = torch.empty_like(acc), torch.empty_like(path), torch.empty_like(bonus)
    ws_p = torch.empty(jf.jf_tree_verify_packed_workspace_size(Tn, V), dtype=torch.uint8,
                       device="cuda")
    jf.jf_tree_verify_sampled_packed(to_dev(pk(w.logits)), dev(pk(draft)), dev(pk(par)), dev(cu),
                                     N, dev(pk(u)), dev(bu), T, acc_p, path_p, bonus_p, ws_p, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(acc, acc_p) and torch.equal(path, path_p) and torch.equal(bonus, bonus_p)
    acc, path, bonus = acc.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy()
    for b, n in enumerate(tree_len):
        r_acc, r_path, r_bonus = jf.tree_verify_sampled(
            to_dev(w.logits[b:b + 1, :n]), dev(draft[b:b + 1, :n]), dev(par[b:b + 1, :n]),
            dev(u[b:b + 1, :n]), dev(bu[b:b + 1]), T)
        assert acc[b] == r_acc.item() and bonus[b] == r_bonus.item(), b
        assert (path[b, :n] == r_path.cpu().numpy()[0]).all() and (path[b, n:] == -1).all()
