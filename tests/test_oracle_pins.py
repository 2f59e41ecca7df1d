"""Pins for the fp64 CPU oracle: each test checks the oracle against something other
than itself -- hand-worked fixtures, brute force, closed forms, or a library routine
(numpy argmax, torch scaled_dot_product_attention) in a special case the method
reduces to.  CPU only."""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
from tree_speculative_decoding_jf_gb300 import workloads as wl
from conftest import GOLDEN


# ----------------------------------------------------------------------------- helpers

def closure(parent):
    """Ancestor-or-self relation by boolean reflexive-transitive closure of the parent
    adjacency (repeated squaring) -- a different computation from walking parents."""
    N = len(parent)
    A = np.zeros((N, N), dtype=bool)
    for i in range(1, N):
        A[i, parent[i]] = True
    R = A | np.eye(N, dtype=bool)
    while True:
        R2 = (R.astype(np.int64) @ R.astype(np.int64)) > 0
        if (R2 == R).all():
            return R
        R = R2


def pack_rows(R):
    """Pack boolean rows LSB-first into little-endian uint64 words (numpy packbits)."""
    N = R.shape[1]
    W = (N + 63) // 64
    padded = np.zeros((R.shape[0], W * 64), dtype=bool)
    padded[:, :N] = R
    return np.packbits(padded, axis=1, bitorder="little").view("<u8")


def all_topological_trees(N):
    for choice in itertools.product(*[range(i) for i in range(1, N)]):
        yield np.array((-1,) + choice, dtype=np.int32)


def random_tree(rng, N):
    p = np.full(N, -1, dtype=np.int32)
    for i in range(1, N):
        p[i] = rng.integers(0, i)
    return p


def f32(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def logical_kv(w, b, g):
    """Contiguous K, V [P_b + N][D] (float64) for sequence b, kv-head g, gathered from
    the pool with numpy fancy indexing through the block table."""
    L = int(w.prefix_len[b]) + w.N
    t = np.arange(L)
    pages = w.block_table[b][t // w.page]
    slots = t % w.page
    k = f32(w.k_cache[pages, slots, g, :])
    v = f32(w.v_cache[pages, slots, g, :])
    return k, v


def sdpa(q, k, v, scale, mask=None):
    """torch fp64 scaled_dot_product_attention for one head: q [n][D], k/v [L][D]."""
    tq = torch.from_numpy(q)[None, None]
    tk = torch.from_numpy(k)[None, None]
    tv = torch.from_numpy(v)[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, scale=scale)
    return out[0, 0].numpy()


def tiny(B=1, N=8, Hq=4, Hkv=2, D=16, P=20, tree="random", seed=0, permute=False,
         parent=None, V=64):
    rng = np.random.default_rng(seed + 1000)
    if parent is None:
        if tree == "random":
            parent = np.stack([random_tree(rng, N) for _ in range(B)])
            tree_kind = "chain"
        else:
            parent, tree_kind = None, tree
    if parent is not None:
        return wl.make_workload("tiny", B, N, Hq, Hkv, D, V, P, parent=np.asarray(parent),
                                permute_pages=permute, seed=seed, logits_dtype="f32")
    return wl.make_workload("tiny", B, N, Hq, Hkv, D, V, P, tree=tree_kind,
                            permute_pages=permute, seed=seed, logits_dtype="f32")


def read_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.rstrip("\n") for ln in f if ln.strip() and not ln.startswith("#")]


# ----------------------------------------------------------------------------- mask

def test_mask_golden_hand_worked():
    lines = read_golden("mask_7node.txt")
    parent = np.array([int(x) for x in lines[0].split(":")[1].split()], dtype=np.int32)
    P = int(lines[1].split(":")[1])
    mask, depth, pos = oracle.tree_mask(parent[None], np.array([P], dtype=np.int32))
    for ln in lines[2:]:
        node, vis, dep, ps = [s.strip() for s in ln.split(":")]
        i = int(node)
        want = 0
        for j in vis.split():
            want |= 1 << int(j)
        assert int(mask[0, i, 0]) == want
        assert depth[0, i] == int(dep) and pos[0, i] == int(ps)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6])
def test_mask_exhaustive_small_trees_vs_closure(N):
    for parent in all_topological_trees(N):
        mask, depth, pos = oracle.tree_mask(parent[None], np.array([7], dtype=np.int32))
        R = closure(parent)
        assert (mask[0] == pack_rows(R)).all()
        assert (depth[0] == R.sum(1) - 1).all()
        assert (pos[0] == 7 + R.sum(1) - 1).all()


@pytest.mark.parametrize("N", [12, 64, 65, 130, 256])
def test_mask_random_trees_vs_closure_multiword(N):
    rng = np.random.default_rng(N)
    parents = np.stack([random_tree(rng, N) for _ in range(3)] + [wl.tree_chain(N)])
    P = np.array([0, 5, 16, 1000], dtype=np.int32)
    mask, depth, pos = oracle.tree_mask(parents, P)
    for b in range(len(parents)):
        R = closure(parents[b])
        assert (mask[b] == pack_rows(R)).all()   # includes zero padding past N
        assert (pos[b] == P[b] + depth[b]).all()


def test_mask_invariants_chain_star():
    N = 70
    m, d, _ = oracle.tree_mask(wl.tree_chain(N)[None], np.zeros(1, np.int32))
    bits = np.unpackbits(m[0].view(np.uint8), axis=1, bitorder="little")[:, :N].astype(bool)
    assert (bits == np.tril(np.ones((N, N), dtype=bool))).all()
    assert (d[0] == np.arange(N)).all()
    m, d, _ = oracle.tree_mask(wl.tree_star(N)[None], np.zeros(1, np.int32))
    bits = np.unpackbits(m[0].view(np.uint8), axis=1, bitorder="little")[:, :N].astype(bool)
    want = np.eye(N, dtype=bool)
    want[:, 0] = True
    assert (bits == want).all()


def test_mask_parent_recurrence_and_popcount():
    rng = np.random.default_rng(5)
    parent = random_tree(rng, 200)
    m, d, _ = oracle.tree_mask(parent[None], np.zeros(1, np.int32))
    for i in range(1, 200):
        bit = np.zeros(4, dtype=np.uint64)
        bit[i // 64] = np.uint64(1) << np.uint64(i % 64)
        assert (m[0, i] == (m[0, parent[i]] | bit)).all()
        pc = sum(bin(int(x)).count("1") for x in m[0, i])
        assert pc == d[0, i] + 1


def test_mask_rejects_non_topological_tree():
    with pytest.raises(oracle.OracleError):
        oracle.tree_mask(np.array([[-1, 2, 0]], np.int32), np.zeros(1, np.int32))
    with pytest.raises(oracle.OracleError):
        oracle.tree_mask(np.array([[0, 0]], np.int32), np.zeros(1, np.int32))


# ----------------------------------------------------------------------------- attention

@pytest.mark.parametrize("P,N", [(0, 8), (20, 8), (37, 13), (5, 40)])
def test_attention_chain_equals_causal_sdpa(P, N):
    w = tiny(N=N, P=P, tree="chain", Hq=4, Hkv=2, D=16, seed=P + N)
    out, lse = oracle.tree_attention(w)
    G = w.G
    for h in range(w.Hq):
        k, v = logical_kv(w, 0, h // G)
        q = f32(w.q[0, :, h, :])
        causal = np.tril(np.ones((N, P + N), dtype=bool), k=P)   # bottom-right causal
        ref = sdpa(q, k, v, w.scale, causal)
        np.testing.assert_allclose(out[0, :, h, :], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("P", [1, 17, 64])
def test_attention_single_node_equals_decode_sdpa(P):
    w = tiny(N=1, P=P, tree="chain", Hq=8, Hkv=2, D=32, seed=P)
    out, lse = oracle.tree_attention(w)
    for h in range(w.Hq):
        k, v = logical_kv(w, 0, h // w.G)
        q = f32(w.q[0, :, h, :])
        np.testing.assert_allclose(out[0, :, h, :], sdpa(q, k, v, w.scale), rtol=1e-12, atol=1e-13)
        s = (q @ k.T)[0] * w.scale
        np.testing.assert_allclose(lse[0, h, 0], np.logaddexp.reduce(s), rtol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_attention_root_path_brute_force(seed):
    """Each node's output equals plain attention over prefix + its root path alone
    (the branch factorisation of the draft distribution, explainer §2)."""
    rng = np.random.default_rng(seed)
    N, P = int(rng.integers(2, 14)), int(rng.integers(0, 40))
    w = tiny(B=2, N=N, P=P, Hq=4, Hkv=1, D=8, seed=seed, permute=bool(seed % 2))
    out, lse = oracle.tree_attention(w)
    for b in range(w.B):
        for i in range(N):
            path, a = [], i
            while a >= 0:
                path.append(a)
                a = int(w.parent[b, a])
            keys = list(range(P)) + [P + j for j in sorted(path)]
            for h in range(w.Hq):
                k, v = logical_kv(w, b, h // w.G)
                q = f32(w.q[b, i, h, :])[None]
                ref = sdpa(q, k[keys], v[keys], w.scale)[0]
                np.testing.assert_allclose(out[b, i, h], ref, rtol=1e-12, atol=1e-13)


def _relabel(parent, rng):
    """Random topological relabelling: returns perm with new_id = perm[old_id]."""
    N = len(parent)
    children = [[] for _ in range(N)]
    for i in range(1, N):
        children[parent[i]].append(i)
    perm = np.empty(N, dtype=np.int64)
    ready, nxt = [0], 0
    while ready:
        x = ready.pop(int(rng.integers(0, len(ready))))
        perm[x] = nxt
        nxt += 1
        ready.extend(children[x])
    return perm


def test_attention_sibling_renumbering_equivariant():
    rng = np.random.default_rng(11)
    N, P = 12, 9
    w = tiny(N=N, P=P, Hq=2, Hkv=1, D=8, seed=3)
    perm = _relabel(w.parent[0], rng)
    w2 = tiny(N=N, P=P, Hq=2, Hkv=1, D=8, seed=3)
    newp = np.full(N, -1, np.int32)
    for i in range(1, N):
        newp[perm[i]] = perm[w.parent[0, i]]
    w2.parent = newp[None].copy()
    w2.q = w.q.copy()
    w2.q[0, perm] = w.q[0]
    for c_src, c_dst in ((w.k_cache, w2.k_cache), (w.v_cache, w2.v_cache)):
        for j in range(N):
            t_old, t_new = P + j, P + perm[j]
            po, pn = w.block_table[0, t_old // 16], w2.block_table[0, t_new // 16]
            c_dst[pn, t_new % 16] = c_src[po, t_old % 16]
    o1, l1 = oracle.tree_attention(w)
    o2, l2 = oracle.tree_attention(w2)
    np.testing.assert_allclose(o2[0, perm], o1[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l2[0][:, perm], l1[0], rtol=1e-12)


def test_attention_masked_weights_exactly_zero():
    w = tiny(N=16, P=10, Hq=2, Hkv=1, D=8, seed=7)
    R = closure(w.parent[0])
    for h in range(w.Hq):
        probs = oracle.attention_probs(w, 0, h)
        assert (probs[:, :10] > 0).all()
        tree = probs[:, 10:]
        assert (tree[~R] == 0.0).all()
        assert (tree[R] > 0).all()
        np.testing.assert_allclose(probs.sum(1), 1.0, rtol=1e-13)


def test_attention_closed_form_single_root_no_prefix():
    w = tiny(N=1, P=0, Hq=4, Hkv=2, D=16, tree="chain", seed=2)
    out, lse = oracle.tree_attention(w)
    for h in range(4):
        g = h // 2
        v = f32(w.v_cache[w.block_table[0, 0], 0, g])
        k = f32(w.k_cache[w.block_table[0, 0], 0, g])
        assert (out[0, 0, h] == v).all()                       # exactly v_root
        assert lse[0, h, 0] == pytest.approx(w.scale * float(f32(w.q[0, 0, h]) @ k), rel=1e-14)


def test_attention_closed_form_equal_keys_gives_mean_of_visible_values():
    w = tiny(N=10, P=7, Hq=2, Hkv=1, D=8, seed=4)
    w.k_cache[:] = w.k_cache[0, 0]            # every key identical -> uniform weights
    out, _ = oracle.tree_attention(w)
    R = closure(w.parent[0])
    k, v = logical_kv(w, 0, 0)
    for i in range(10):
        vis = list(range(7)) + [7 + j for j in np.nonzero(R[i])[0]]
        np.testing.assert_allclose(out[0, i, 0], v[vis].mean(0), rtol=1e-12, atol=1e-14)


def test_attention_gqa_equals_mha_with_duplicated_kv_heads():
    w1 = tiny(N=6, P=11, Hq=2, Hkv=1, D=8, seed=9)
    w2 = tiny(N=6, P=11, Hq=2, Hkv=2, D=8, seed=9)
    w2.parent = w1.parent.copy()
    w2.q = w1.q.copy()
    w2.k_cache = np.repeat(w1.k_cache, 2, axis=2)
    w2.v_cache = np.repeat(w1.v_cache, 2, axis=2)
    w2.block_table = w1.block_table.copy()
    o1, l1 = oracle.tree_attention(w1)
    o2, l2 = oracle.tree_attention(w2)
    assert (o1 == o2).all() and (l1 == l2).all()


def test_attention_page_permutation_invariant():
    a = tiny(B=2, N=9, P=45, Hq=4, Hkv=2, D=8, seed=21, permute=False)
    b = tiny(B=2, N=9, P=45, Hq=4, Hkv=2, D=8, seed=21, permute=True)
    assert not (a.block_table == b.block_table).all()
    # put a's logical rows into b's pool layout
    for bb in range(2):
        L = int(a.prefix_len[bb]) + a.N
        for t in range(L):
            pa, pb = a.block_table[bb, t // 16], b.block_table[bb, t // 16]
            b.k_cache[pb, t % 16] = a.k_cache[pa, t % 16]
            b.v_cache[pb, t % 16] = a.v_cache[pa, t % 16]
    b.q, b.parent = a.q, a.parent
    oa, la = oracle.tree_attention(a)
    ob, lb = oracle.tree_attention(b)
    assert (oa == ob).all() and (la == lb).all()


def test_attention_rows_sample_matches_full():
    w = tiny(B=2, N=7, P=30, Hq=4, Hkv=2, D=8, seed=5)
    out, lse = oracle.tree_attention(w)
    rb, rh, ri = np.array([1, 0, 1]), np.array([3, 0, 2]), np.array([6, 0, 4])
    o, l = oracle.tree_attention_rows(w, rb, rh, ri)
    for n in range(3):
        assert (o[n] == out[rb[n], ri[n], rh[n]]).all()
        assert l[n] == lse[rb[n], rh[n], ri[n]]


def test_ragged_reading_node_rows_depend_only_on_earlier_nodes():
    """Ragged trees are read as each sequence's first n_b nodes.  That reading is sound
    because a node's mask row and attention row involve only itself and earlier nodes
    (ancestors have smaller ids): the fixed-size problem restricted to rows i < n equals
    the problem built from the first n nodes, bit for bit."""
    import dataclasses
    w = tiny(B=2, N=9, P=21, Hq=4, Hkv=2, D=8, seed=12)
    full_o, full_l = oracle.tree_attention(w)
    full_m, full_d, full_p = oracle.tree_mask(w.parent, w.prefix_len)
    for b in range(w.B):
        for n in (1, 4, 9):
            ws = dataclasses.replace(w, B=1, N=n, prefix_len=w.prefix_len[b:b + 1].copy(),
                                     parent=w.parent[b:b + 1, :n].copy(),
                                     q=w.q[b:b + 1, :n].copy(),
                                     block_table=w.block_table[b:b + 1].copy())
            o, l = oracle.tree_attention(ws)
            assert (o[0] == full_o[b, :n]).all() and (l[0] == full_l[b, :, :n]).all()
            m, d, p = oracle.tree_mask(ws.parent, ws.prefix_len)
            assert (m[0, :, 0] == full_m[b, :n, 0]).all()
            assert (d[0] == full_d[b, :n]).all() and (p[0] == full_p[b, :n]).all()


# ----------------------------------------------------------------------------- verify

def _golden_argmax_rows():
    rows = []
    for ln in read_golden("argmax_rows.txt"):
        idx, vals = ln.split(":")
        rows.append((int(idx), [float(x) for x in vals.split()]))
    return rows


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_argmax_golden_ties_and_signed_zero(dtype):
    for idx, vals in _golden_argmax_rows():
        x = np.array(vals, dtype=np.float32)
        if dtype == "bf16":
            x = wl.to_bf16_bits(x)
            assert (wl.bf16_bits_to_f32(x) == np.array(vals, dtype=np.float32)).all()
        assert oracle.argmax(x[None], dtype)[0] == idx


def test_argmax_matches_numpy_first_occurrence():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((64, 5000)) * 2).astype(np.float32)
    x[3, 100] = x[3, 4000] = 50.0      # tie: first occurrence
    assert (oracle.argmax(x, "f32") == np.argmax(x, axis=1)).all()
    xb = wl.to_bf16_bits(x)            # bf16 rounding creates many ties
    assert (oracle.argmax(xb, "bf16") == np.argmax(wl.bf16_bits_to_f32(xb), axis=1)).all()


def _golden_walk_cases():
    lines = read_golden("verify_walk.txt")
    cases, cur = [], None
    for ln in lines:
        key, val = ln.split(":", 1)
        key = key.strip()
        if key == "case":
            cur = {"name": val.strip()}
            cases.append(cur)
        elif key == "expect":
            a, p, bo = val.split("|")
            cur["expect"] = (int(a), [int(x) for x in p.split()], int(bo))
        else:
            cur[key] = np.array([int(x) for x in val.split()], dtype=np.int32)
    return cases


@pytest.mark.parametrize("case", _golden_walk_cases(), ids=lambda c: c["name"])
def test_tree_walk_golden(case):
    acc, path, bonus = oracle.tree_walk(case["argmax"][None], case["draft"][None],
                                        case["parent"][None])
    a, p, bo = case["expect"]
    assert acc[0] == a and list(path[0]) == p and bonus[0] == bo


def _brute_force_walk(argmax, draft, parent):
    """Enumerate every root path, keep the all-accepted ones, take the longest and
    among those the lexicographically smallest sequence of node ids."""
    N = len(parent)
    best = [0]
    for n in range(N):
        path, a = [], n
        while a >= 0:
            path.append(a)
            a = int(parent[a])
        path = path[::-1]
        ok = all(draft[c] == argmax[parent[c]] for c in path[1:])
        if ok and (len(path) > len(best) or (len(path) == len(best) and path < best)):
            best = path
    return len(best) - 1, best + [-1] * (N - len(best)), int(argmax[best[-1]])


@pytest.mark.parametrize("seed", range(40))
def test_tree_walk_brute_force(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 13))
    parent = random_tree(rng, N)
    argmax = rng.integers(0, 3, N).astype(np.int32)
    draft = rng.integers(0, 3, N).astype(np.int32)
    acc, path, bonus = oracle.tree_walk(argmax[None], draft[None], parent[None])
    a, p, bo = _brute_force_walk(argmax, draft, parent)
    assert acc[0] == a and list(path[0]) == p and bonus[0] == bo


def test_tree_walk_accept_len_invariant_under_renumbering():
    rng = np.random.default_rng(3)
    for _ in range(20):
        N = 12
        parent = random_tree(rng, N)
        argmax = rng.integers(0, 2, N).astype(np.int32)
        draft = rng.integers(0, 2, N).astype(np.int32)
        perm = _relabel(parent, rng)
        p2 = np.full(N, -1, np.int32)
        a2, d2 = np.empty(N, np.int32), np.empty(N, np.int32)
        for i in range(N):
            a2[perm[i]], d2[perm[i]] = argmax[i], draft[i]
            if i:
                p2[perm[i]] = perm[parent[i]]
        x = oracle.tree_walk(argmax[None], draft[None], parent[None])
        y = oracle.tree_walk(a2[None], d2[None], p2[None])
        assert x[0][0] == y[0][0]


def test_chain5_forcing_gives_accept_len_five():
    w = wl.make_workload("chain5", 1, 16, 4, 1, 16, 4096, 32, tree="chain",
                         forcing="chain5", seed=3)
    am, acc, path, bonus = oracle.tree_verify(w)
    assert acc[0] == 5 and list(path[0][:7]) == [0, 1, 2, 3, 4, 5, -1]
    assert bonus[0] == am[0, 5]


# ----------------------------------------------------------------------------- inputs

def test_generators_are_deterministic():
    a = wl.config("c1_tiny_random16")
    b = wl.config("c1_tiny_random16")
    for f in ("parent", "q", "k_cache", "v_cache", "block_table", "logits", "draft"):
        assert (getattr(a, f) == getattr(b, f)).all()


def test_best_first_tree_shape():
    rng = np.random.default_rng(0)
    parent, tokens = wl.tree_best_first(rng, 256, 151936)
    assert parent[0] == -1 and all(0 <= parent[i] < i for i in range(1, 256))
    depth = np.zeros(256, int)
    for i in range(1, 256):
        depth[i] = depth[parent[i]] + 1
    assert depth.max() <= 15
    for p in set(parent[1:].tolist()):
        kids = tokens[parent == p]
        assert len(set(kids.tolist())) == len(kids)      # distinct candidate tokens


def test_c1_config_shape_and_forcing():
    w = wl.config("c1_tiny_random16")
    assert w.q.shape == (1, 16, 4, 64) and w.k_cache.shape == (9, 16, 1, 64)
    _, depth, _ = oracle.tree_mask(w.parent, w.prefix_len)
    assert depth.max() <= 6
    am = oracle.argmax(w.logits, "f32")
    forced = [c for c in range(1, 16) if w.draft[0, c] == am[0, w.parent[0, c]]]
    assert len(forced) >= 3


# ---------------------------------------------------------------- accepted-path KV compaction

def _logical_rows(cache, block_table, b, L, page=16):
    """Rows of sequence b at logical positions 0..L-1, read through its block table."""
    return np.stack([cache[block_table[b, t // page], t % page] for t in range(L)])


def _compaction_by_lists(w, path, acc):
    """Independent restatement: each sequence's context is a list of rows; the new context
    keeps the prefix, then the rows of the accepted path in order, then whatever followed
    (positions past the accepted path are not touched).  The lists are written back through
    the block tables into copies of the pool."""
    k, v = w.k_cache.copy(), w.v_cache.copy()
    newp = np.empty(w.B, np.int32)
    for b in range(w.B):
        P, a = int(w.prefix_len[b]), int(acc[b])
        L = P + w.N
        ks, vs = _logical_rows(w.k_cache, w.block_table, b, L), _logical_rows(w.v_cache, w.block_table, b, L)
        order = list(range(P)) + [P + int(path[b, j]) for j in range(a + 1)] + list(range(P + a + 1, L))
        for t, src in enumerate(order):
            k[w.block_table[b, t // 16], t % 16] = ks[src]
            v[w.block_table[b, t // 16], t % 16] = vs[src]
        newp[b] = P + a + 1
    return k, v, newp


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_compaction_matches_list_restatement(seed):
    w = wl.make_workload("cmp", 3, 12, 4, 2, 64, 64, np.array([5, 17, 40], np.int32),
                         tree="random_depth_limited", permute_pages=True, seed=seed,
                         with_logits=False)
    path, acc = wl.random_accepted_paths(w.parent, seed)
    k, v, newp, ok = oracle.compact_accepted_kv(w.k_cache, w.v_cache, w.block_table,
                                                w.prefix_len, path, acc)
    ek, ev, enewp = _compaction_by_lists(w, path, acc)
    assert ok
    assert (newp == enewp).all()
    assert (k == ek).all() and (v == ev).all()


def test_compaction_overlapping_path_reads_before_writes():
    """path [0, 2, 3, 5]: the row that lands on position P+2 is also the source of P+1."""
    w = wl.make_workload("ovl", 1, 8, 2, 1, 64, 64, 19, tree="chain", seed=4, with_logits=False)
    parent = np.array([[-1, 0, 0, 2, 3, 3, 5, 6]], np.int32)
    path = np.array([[0, 2, 3, 5, -1, -1, -1, -1]], np.int32)
    acc = np.array([3], np.int32)
    k, _, newp, ok = oracle.compact_accepted_kv(w.k_cache, w.v_cache, w.block_table,
                                                w.prefix_len, path, acc)
    assert ok and newp[0] == 19 + 4
    rows_before = _logical_rows(w.k_cache, w.block_table, 0, 27)
    rows_after = _logical_rows(k, w.block_table, 0, 27)
    for j, node in enumerate([0, 2, 3, 5]):
        assert (rows_after[19 + j] == rows_before[19 + node]).all()
    assert (rows_after[:19] == rows_before[:19]).all()
    assert (rows_after[23:] == rows_before[23:]).all()
    del parent


def test_compaction_chain_and_empty_path_are_no_ops():
    w = wl.make_workload("noop", 2, 10, 4, 2, 128, 64, np.array([3, 33], np.int32),
                         tree="chain", seed=5, with_logits=False)
    chain = np.tile(np.arange(10, dtype=np.int32), (2, 1))
    for acc in (np.array([9, 4], np.int32), np.array([0, 0], np.int32)):
        path = np.where(np.arange(10)[None, :] <= acc[:, None], chain, -1).astype(np.int32)
        k, v, newp, ok = oracle.compact_accepted_kv(w.k_cache, w.v_cache, w.block_table,
                                                    w.prefix_len, path, acc)
        assert ok and (newp == w.prefix_len + acc + 1).all()
        assert (k == w.k_cache).all() and (v == w.v_cache).all()


def test_compaction_rejects_malformed_and_leaves_sequence():
    w = wl.make_workload("bad", 2, 6, 2, 1, 64, 64, np.array([4, 9], np.int32),
                         tree="chain", seed=6, with_logits=False)
    path = np.array([[0, 3, 2, -1, -1, -1], [0, 1, 2, -1, -1, -1]], np.int32)   # b=0 not increasing
    acc = np.array([2, 2], np.int32)
    k, _, newp, ok = oracle.compact_accepted_kv(w.k_cache, w.v_cache, w.block_table,
                                                w.prefix_len, path, acc)
    assert not ok
    assert newp[0] == 4 and newp[1] == 9 + 3
    assert (_logical_rows(k, w.block_table, 0, 10) == _logical_rows(w.k_cache, w.block_table, 0, 10)).all()


# ---------------------------------------------------------------- best-first draft tree

from oracle import draft_tree as odt    # noqa: E402


def test_draft_candidates_logp_matches_torch_log_softmax():
    x = wl.bf16_bits_to_f32(wl.draft_logits(1, 3, 5000, seed=1))[0]
    for d in range(3):
        tok, lp = odt.depth_candidates(x[d], 8)
        ref = torch.log_softmax(torch.from_numpy(x[d]).double(), dim=0).numpy()
        assert np.allclose(lp, ref[tok], rtol=0, atol=1e-12)
        order = np.lexsort((np.arange(x.shape[1]), -x[d].astype(np.float64)))
        assert (tok == order[:8]).all()


def test_draft_candidates_ties_take_lower_ids():
    x = np.zeros(50, np.float32)
    x[[7, 3, 40]] = 2.0
    x[[1, 9]] = 1.0
    tok, _ = odt.depth_candidates(x, 6)
    assert tok.tolist() == [3, 7, 40, 1, 9, 0]


def _lattice_brute_force(ct, lp, N, root):
    """Every node of the lattice (rank paths up to Dmax), scored in fp64 from the root,
    sorted by (score desc, depth, rank path); the first N with parents looked up by path."""
    Dmax, K = ct.shape
    nodes = [((), 0.0)]
    frontier = [((), 0.0)]
    for d in range(Dmax):
        nxt = []
        for path, s in frontier:
            for r in range(K):
                nxt.append((path + (r,), s + float(lp[d, r])))
        nodes += nxt
        frontier = nxt
    nodes.sort(key=lambda n: (-n[1], len(n[0]), n[0]))
    top = nodes[:N]
    index = {path: i for i, (path, _) in enumerate(top)}
    parent = [index.get(p[:-1], -2) if p else -1 for p, _ in top]
    draft = [root if not p else int(ct[len(p) - 1, p[-1]]) for p, _ in top]
    return (np.array(parent), np.array(draft), np.array([len(p) for p, _ in top]),
            np.array([s for _, s in top], np.float64), [p for p, _ in top])


@pytest.mark.parametrize("K,Dmax,N,seed", [(2, 4, 20, 0), (3, 3, 30, 1), (4, 3, 40, 2),
                                           (1, 6, 7, 3), (5, 1, 6, 4)])
def test_best_first_matches_lattice_brute_force(K, Dmax, N, seed):
    rng = np.random.default_rng(seed)
    ct = rng.integers(0, 1000, size=(Dmax, K))
    lp = np.sort(rng.standard_normal((Dmax, K)) * 2 - 3, axis=1)[:, ::-1].copy()
    got = odt.best_first_tree(ct, lp, N, root_token=77)
    ref = _lattice_brute_force(ct, lp, N, 77)
    for g, r in zip(got[:4], ref[:4]):
        assert (np.asarray(g) == np.asarray(r)).all()
    assert got[4] == ref[4]
    for path, s in zip(got[4], got[3]):
        assert odt.path_score(lp, path) == s


def test_best_first_scores_are_exact_sums():
    """Two depth-2 branches whose cumulative log-probs differ by 1e-12 (equal in fp32):
    the exact (fp64) sum orders them, (1, 0) before (0, 1), although a tie would put the
    smaller rank path first."""
    ct = np.array([[1, 2], [3, 4]])
    lp = np.array([[-1.0, -1.0 - 1e-12], [-3.0, -3.0 - 2e-12]])
    parent, draft, depth, score, paths = odt.best_first_tree(ct, lp, 6, root_token=0)
    assert paths == [(), (0,), (1,), (0, 0), (1, 0), (0, 1)]
    assert parent.tolist() == [-1, 0, 0, 1, 2, 1]
    assert draft.tolist() == [0, 1, 2, 3, 3, 4]
    assert np.float32(score[4]) == np.float32(score[5]) and score[4] > score[5]


def test_best_first_equal_scores_prefer_shallow_then_small_rank():
    ct = np.array([[10, 11], [20, 21]])
    lp = np.zeros((2, 2))                      # every node scores 0: pure tie-breaking
    parent, draft, depth, _, _ = odt.best_first_tree(ct, lp, 7, root_token=5)
    assert depth.tolist() == [0, 1, 1, 2, 2, 2, 2]
    assert draft.tolist() == [5, 10, 11, 20, 21, 20, 21]
    assert parent.tolist() == [-1, 0, 0, 1, 1, 2, 2]


def test_best_first_invariants_random():
    x = wl.bf16_bits_to_f32(wl.draft_logits(1, 16, 2000, seed=7))[0]
    tok, lp = odt.candidates(x[None], 8)
    parent, draft, depth, score, _ = odt.best_first_tree(tok[0], lp[0], 256, root_token=3)
    assert parent[0] == -1 and depth[0] == 0 and draft[0] == 3
    for i in range(1, 256):
        p = parent[i]
        assert 0 <= p < i and depth[i] == depth[p] + 1 and score[i] <= score[p]
        assert draft[i] in tok[0, depth[i] - 1]
    assert depth.max() <= 16


# ---------------------------------------------------------------- stochastic verification

from oracle import sampled_verify as osv    # noqa: E402


def _golden_sampled_cases():
    cases, cur = [], None
    for ln in read_golden("sampled_verify.txt"):
        key, val = ln.split(":", 1)
        key = key.strip()
        if key == "case":
            cur = {"name": val.strip(), "p": []}
            cases.append(cur)
        elif key == "expect":
            a, p, bo = val.split("|")
            cur["expect"] = (int(a), [int(x) for x in p.split()], int(bo))
        elif key.startswith("p") and key[1:].isdigit():
            cur["p"].append([float(x) for x in val.split()])
        elif key == "bonus_uniform":
            cur["bonus_uniform"] = float(val)
        else:
            cur[key] = np.array([float(x) for x in val.split()])
    return cases


@pytest.mark.parametrize("case", _golden_sampled_cases(), ids=lambda c: c["name"])
def test_sampled_verify_golden(case):
    logits = np.log(np.array(case["p"], np.float64)).astype(np.float32)[None]
    acc, path, bonus, margins = osv.tree_verify_sampled(
        logits, "f32", case["draft"].astype(np.int32)[None], case["parent"].astype(np.int32)[None],
        case["uniform"][None], np.array([case["bonus_uniform"]]), 1.0)
    a, p, bo = case["expect"]
    assert acc[0] == a and list(path[0]) == p and bonus[0] == bo
    assert min(m for _, _, m in margins[0]) > 0.01      # no decision sits on a boundary


def _chi2_ok(counts, probs, n):
    """Pearson chi-square of observed counts against n * probs; loose bound (the seeds are
    fixed, so this is deterministic) that still rejects a wrong distribution."""
    exp = probs * n
    stat = float(((counts - exp) ** 2 / np.maximum(exp, 1e-12)).sum())
    return stat < 40.0, stat


def test_sampled_verify_emits_the_target_distribution():
    """Losslessness: over many draws of the random numbers, the first emitted token follows
    p(root) and, given that child 1 (resp. 2) was accepted, the second follows p(1) (resp.
    p(2)) -- whatever the drafted tokens are."""
    rng = np.random.default_rng(0)
    V, T = 6, 0.8
    parent = np.array([-1, 0, 0, 0, 1, 1, 2], np.int32)
    draft = np.array([0, 2, 0, 5, 1, 3, 4], np.int32)
    N = len(parent)
    rows = rng.standard_normal((N, V)).astype(np.float32)
    n = 40000
    logits = np.broadcast_to(rows, (n, N, V))
    par = np.broadcast_to(parent, (n, N))
    dr = np.broadcast_to(draft, (n, N))
    acc, path, bonus, _ = osv.tree_verify_sampled(logits, "f32", dr, par, rng.random((n, N)),
                                                  rng.random(n), T)
    first = np.where(acc >= 1, draft[np.maximum(path[:, 1], 0)], bonus)
    ok, stat = _chi2_ok(np.bincount(first, minlength=V), osv.target_probs(rows[0].astype(np.float64), T), n)
    assert ok, stat
    for c in (1, 2):
        sel = (acc >= 1) & (path[:, 1] == c)
        second = np.where(acc[sel] >= 2, draft[np.maximum(path[sel, 2], 0)], bonus[sel])
        ok, stat = _chi2_ok(np.bincount(second, minlength=V),
                            osv.target_probs(rows[c].astype(np.float64), T), int(sel.sum()))
        assert ok, (c, stat)


def test_sampled_verify_wrong_residual_is_detected():
    """The distribution test has teeth: renormalising without removing rejected tokens
    (a plausible slip) changes the first token's distribution enough to fail it."""
    rng = np.random.default_rng(1)
    V, T = 6, 0.8
    rows = rng.standard_normal((4, V)).astype(np.float64)
    p = osv.target_probs(rows[0], T)
    drafts = [2, 0, 5]
    n = 40000
    counts = np.zeros(V)
    for _ in range(n):                      # the slip: r never loses the rejected tokens
        y = None
        for x in drafts:
            if rng.random() < p[x]:
                y = x
                break
        if y is None:
            y = int(np.searchsorted(np.cumsum(p), rng.random(), side="right"))
        counts[y] += 1
    assert not _chi2_ok(counts, p, n)[0]


def test_sampled_verify_at_low_temperature_is_greedy():
    """T -> 0 makes p one-hot at the argmax: a child is accepted iff its token is the
    parent's argmax, and the bonus is the argmax at the last node -- the greedy walk (with
    distinct sibling tokens, at most one child per node can match)."""
    rng = np.random.default_rng(2)
    B, N, V = 6, 24, 50
    parent = np.stack([np.array([-1] + [rng.integers(max(0, i - 4), i) for i in range(1, N)])
                       for _ in range(B)]).astype(np.int32)
    logits = (rng.standard_normal((B, N, V)) * 2).astype(np.float32)
    am = logits.argmax(-1)
    srt = np.sort(logits, -1)
    assert (srt[..., -1] - srt[..., -2]).min() > 1e-3
    draft = np.zeros((B, N), np.int32)
    for b in range(B):
        for p_ in range(N):
            kids = np.flatnonzero(parent[b] == p_)
            toks = rng.permutation(V)[:len(kids)]
            if len(kids) and rng.random() < 0.7:
                toks[rng.integers(len(kids))] = am[b, p_] if am[b, p_] not in toks else toks[0]
            draft[b, kids] = toks
    acc, path, bonus, _ = osv.tree_verify_sampled(logits, "f32", draft, parent,
                                                  rng.uniform(0.01, 0.99, (B, N)),
                                                  rng.uniform(0.01, 0.99, B), 1e-5)
    racc, rpath, rbonus = oracle.tree_walk(am.astype(np.int32), draft, parent)
    assert (acc == racc).all() and (path == rpath).all() and (bonus == rbonus).all()
    assert racc.max() >= 2
