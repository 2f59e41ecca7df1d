"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the same
seeded inputs.  Masks, argmax, accepted lengths, paths and bonus tokens must match
bit-exactly; attention outputs within |gpu - ref| <= 2e-3 + 1e-2 * |ref| (bf16 inputs,
fp32 accumulation, bf16 output)."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
LSE_ATOL = 2e-3


@pytest.fixture(scope="module")
def jf():
    from tree_speculative_decoding_jf_gb300 import build
    build.build()
    from tree_speculative_decoding_jf_gb300 import jf as mod
    return mod


_CACHE = {}


def cfg(name, forcing=None):
    key = (name, forcing)
    if key not in _CACHE:
        _CACHE.clear() if len(_CACHE) > 3 else None
        _CACHE[key] = wl.config(name, forcing=forcing)
    return _CACHE[key]


def dev_err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ----------------------------------------------------------------------------- mask

def gpu_mask(jf, w):
    t = wl.device_tensors(w, with_logits=False)
    err = dev_err()
    mask, depth, pos = jf.build_tree_mask(t["parent"], t["prefix_len"], dev_err=err)
    torch.cuda.synchronize()
    return (mask.cpu().numpy().view(np.uint64), depth.cpu().numpy(), pos.cpu().numpy(),
            int(err.item()))


@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_mask_configs_bit_exact(jf, name):
    w = cfg(name)
    m, d, p, err = gpu_mask(jf, w)
    rm, rd, rp = oracle.tree_mask(w.parent, w.prefix_len)
    assert err == 0
    assert (m == rm).all() and (d == rd).all() and (p == rp).all()


@pytest.mark.parametrize("N,tree", [(1, "chain"), (64, "random"), (65, "random"),
                                    (300, "random"), (4096, "chain"), (4096, "star")])
def test_mask_edge_sizes(jf, N, tree):
    rng = np.random.default_rng(N)
    B = 3
    if tree == "random":
        parent = np.stack([np.array([-1] + [rng.integers(0, i) for i in range(1, N)], np.int32)
                           for _ in range(B)])
    elif tree == "chain":
        parent = np.stack([wl.tree_chain(N)] * B)
    else:
        parent = np.stack([wl.tree_star(N)] * B)
    prefix = np.array([0, 17, 5000], np.int32)
    tp = torch.from_numpy(parent).cuda()
    tl = torch.from_numpy(prefix).cuda()
    err = dev_err()
    mask, depth, pos = jf.build_tree_mask(tp, tl, dev_err=err)
    rm, rd, rpos = oracle.tree_mask(parent, prefix)
    assert err.item() == 0
    assert (mask.cpu().numpy().view(np.uint64) == rm).all()
    assert (depth.cpu().numpy() == rd).all() and (pos.cpu().numpy() == rpos).all()


def test_mask_reports_malformed_tree(jf):
    parent = torch.tensor([[-1, 0, 2, 1], [-1, 0, 1, 2]], dtype=torch.int32, device="cuda")
    err = dev_err()
    jf.build_tree_mask(parent, torch.zeros(2, dtype=torch.int32, device="cuda"), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & jf.DEVERR_BAD_PARENT


# ----------------------------------------------------------------------------- verify

def gpu_verify(jf, w, logits=None):
    t = wl.device_tensors(w, with_logits=logits is None)
    lg = t["logits"] if logits is None else logits
    err = dev_err()
    am, acc, path, bonus = jf.tree_verify(lg, t["draft"], t["parent"], dev_err=err)
    torch.cuda.synchronize()
    return am.cpu().numpy(), acc.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy(), int(err.item())


def assert_verify_matches(jf, w):
    am, acc, path, bonus, err = gpu_verify(jf, w)
    ram, racc, rpath, rbonus = oracle.tree_verify(w)
    assert err == 0
    assert (am == ram).all(), "argmax differs"
    assert (acc == racc).all() and (path == rpath).all() and (bonus == rbonus).all()
    return racc


@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_verify_configs_bit_exact(jf, name):
    acc = assert_verify_matches(jf, cfg(name))
    if name.startswith("c2"):
        assert (acc == 5).all()


@pytest.mark.parametrize("name", ["c3_qwen3_8b_tree256", "c4_qwen3_8b_b32_tree64_paged"])
def test_verify_forced_variants_bit_exact(jf, name):
    acc = assert_verify_matches(jf, cfg(name, forcing="half"))
    assert acc.max() >= 1


def test_verify_golden_walk_cases(jf):
    from test_oracle_pins import _golden_walk_cases
    rng = np.random.default_rng(0)
    for case in _golden_walk_cases():
        N = len(case["parent"])
        V = 64
        logits = rng.uniform(-1, 1, size=(1, N, V)).astype(np.float32)
        logits[0, np.arange(N), case["argmax"]] = 5.0
        lg = torch.from_numpy(logits).cuda()
        am, acc, path, bonus = jf.tree_verify(lg, torch.from_numpy(case["draft"][None]).cuda(),
                                              torch.from_numpy(case["parent"][None]).cuda())
        a, p, bo = case["expect"]
        assert (am.cpu().numpy()[0] == case["argmax"]).all()
        assert acc.item() == a and list(path.cpu().numpy()[0]) == p and bonus.item() == bo


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_verify_argmax_golden_rows(jf, dtype):
    from test_oracle_pins import _golden_argmax_rows
    for idx, vals in _golden_argmax_rows():
        x = np.array(vals, dtype=np.float32)[None, None]
        if dtype == "bf16":
            t = torch.from_numpy(x).to(torch.bfloat16).cuda()
        else:
            t = torch.from_numpy(x).cuda()
        z = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
        par = torch.full((1, 1), -1, dtype=torch.int32, device="cuda")
        am, _, _, bonus = jf.tree_verify(t, z, par)
        assert am.item() == idx and bonus.item() == idx


@pytest.mark.parametrize("V,offset", [(1001, 0), (1001, 1), (151937, 3), (7, 1), (8192 * 3 + 5, 2)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_verify_ties_and_unaligned_rows(jf, V, offset, dtype):
    """Odd vocab sizes and row starts off the 16-byte grid; planted ties at the max in the
    scalar head, the vector body and the tail of the rows."""
    rng = np.random.default_rng(V + offset)
    B, N = 2, 24
    x = rng.standard_normal((B * N * V + offset,)).astype(np.float32) * 2
    rows = x[offset:].reshape(B, N, V)
    for r in range(B * N):
        b, i = divmod(r, N)
        pos = sorted(set(rng.integers(0, V, size=3).tolist() + [0, V - 1][r % 2:r % 2 + 1]))
        rows[b, i, pos] = 40.0
        if r % 3 == 0:
            rows[b, i, :] = -rows[b, i, :] ** 2 - 1.0
            rows[b, i, pos] = -0.0 if r % 2 else 0.0
    if dtype == "bf16":
        full = torch.from_numpy(x).to(torch.bfloat16)
        ref_rows = full[offset:].view(B, N, V).view(torch.int16).numpy().view(np.uint16)
    else:
        full = torch.from_numpy(x)
        ref_rows = rows
    lg = full.cuda()[offset:].view(B, N, V)
    parent = np.stack([np.array([-1] + [rng.integers(0, i) for i in range(1, N)], np.int32)
                       for _ in range(B)])
    ram = oracle.argmax(ref_rows, dtype)
    draft = np.where(rng.random((B, N)) < 0.6, ram[np.arange(B)[:, None], np.maximum(parent, 0)],
                     rng.integers(0, V, (B, N))).astype(np.int32)
    am, acc, path, bonus = jf.tree_verify(lg, torch.from_numpy(draft).cuda(),
                                          torch.from_numpy(parent).cuda())
    racc, rpath, rbonus = oracle.tree_walk(ram, draft, parent)
    assert (am.cpu().numpy() == ram).all()
    assert (acc.cpu().numpy() == racc).all() and (path.cpu().numpy() == rpath).all()
    assert (bonus.cpu().numpy() == rbonus).all()


@pytest.mark.parametrize("N", [1024, 4096])
def test_verify_long_accepted_chain(jf, N):
    V = 64
    rng = np.random.default_rng(N)
    logits = rng.uniform(-1, 1, size=(1, N, V)).astype(np.float32)
    tok = rng.integers(0, V, N)
    logits[0, np.arange(N), tok] = 3.0
    draft = np.concatenate([[0], tok[:-1]]).astype(np.int32)[None]
    parent = wl.tree_chain(N)[None]
    am, acc, path, bonus = jf.tree_verify(torch.from_numpy(logits).cuda(),
                                          torch.from_numpy(draft).cuda(),
                                          torch.from_numpy(parent).cuda())
    assert acc.item() == N - 1 and (path.cpu().numpy()[0] == np.arange(N)).all()
    assert bonus.item() == tok[-1]
    if N <= 1024:
        racc, rpath, rbonus = oracle.tree_walk(am.cpu().numpy(), draft, parent)
        assert racc[0] == N - 1 and rbonus[0] == bonus.item()


def test_verify_reports_bad_tokens_and_parents(jf):
    lg = torch.randn(1, 4, 50, device="cuda")
    par = torch.tensor([[-1, 0, 0, 1]], dtype=torch.int32, device="cuda")
    err = dev_err()
    jf.tree_verify(lg, torch.tensor([[0, 3, 99, 1]], dtype=torch.int32, device="cuda"), par,
                   dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == jf.DEVERR_BAD_TOKEN
    err = dev_err()
    jf.tree_verify(lg, torch.zeros(1, 4, dtype=torch.int32, device="cuda"),
                   torch.tensor([[-1, 0, 3, 1]], dtype=torch.int32, device="cuda"), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == jf.DEVERR_BAD_PARENT


# ----------------------------------------------------------------------------- attention

def gpu_attention(jf, w, t=None):
    t = t or wl.device_tensors(w, with_logits=False)
    mask, _, _ = jf.build_tree_mask(t["parent"], t["prefix_len"])
    err = dev_err()
    out, lse = jf.tree_attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                 t["prefix_len"], mask, scale=w.scale, with_lse=True, dev_err=err)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(err.item())


def sample_rows(w, n, seed=0):
    """Rows spread over sequences, heads and nodes, always including the root, the last
    node and the deepest node of each sequence."""
    rng = np.random.default_rng(seed)
    rb = list(rng.integers(0, w.B, n))
    ri = list(rng.integers(0, w.N, n))
    rh = list(rng.integers(0, w.Hq, n))
    for b in range(w.B):
        depth = np.zeros(w.N, int)
        for i in range(1, w.N):
            depth[i] = depth[w.parent[b, i]] + 1
        for i in (0, w.N - 1, int(depth.argmax())):
            for h in (0, w.Hq - 1):
                rb.append(b); ri.append(i); rh.append(h)
    return np.array(rb), np.array(rh), np.array(ri)


def assert_attention_close(w, out, lse, rows):
    rb, rh, ri = rows
    ref_o, ref_l = oracle.tree_attention_rows(w, rb, rh, ri)
    got = out[rb, ri, rh]
    err = np.abs(got - ref_o)
    bad = err > ATOL + RTOL * np.abs(ref_o)
    assert not bad.any(), (f"{bad.sum()} elements out of tolerance; max abs err {err.max():.3e}; "
                           f"first bad row {np.argwhere(bad)[0]}")
    lerr = np.abs(lse[rb, rh, ri] - ref_l)
    assert lerr.max() <= LSE_ATOL, f"lse max abs err {lerr.max():.3e}"


@pytest.mark.parametrize("name,nrows", [("c1_tiny_random16", None), ("c2_qwen3_8b_chain16", None),
                                        ("c3_qwen3_8b_tree256", 1024),
                                        ("c4_qwen3_8b_b32_tree64_paged", 768),
                                        ("c5_qwen3_30b_b8_tree256_32k", 256)])
def test_attention_configs(jf, name, nrows):
    w = cfg(name)
    out, lse, err = gpu_attention(jf, w)
    assert err == 0
    assert np.isfinite(out).all()
    rows = oracle.all_rows(w) if nrows is None else sample_rows(w, nrows)
    assert_attention_close(w, out, lse, rows)


@pytest.mark.parametrize("name", ["c3_qwen3_8b_tree256", "c4_qwen3_8b_b32_tree64_paged",
                                  "c5_qwen3_30b_b8_tree256_32k"])
def test_attention_every_row_of_the_large_workloads(jf, name):
    """Every output row of the budget-256 and 32-sequence workloads against the fp64 oracle
    (workload 5: 65536 rows over 32768-token prefixes, about 1.1 TFLOP of fp64 on the host),
    so no dispatch boundary, split range or stream-K piece escapes the check."""
    w = cfg(name)
    out, lse, err = gpu_attention(jf, w)
    assert err == 0
    assert_attention_close(w, out, lse, oracle.all_rows(w))


def first_stream_k_cut_pair(w, sms):
    """(b, kv-head) of the first pair that a stream-K range boundary cuts inside, for the
    range partition the attention call uses on `sms` SMs: the key tiles of all pairs laid
    end to end head-major (pair (b, g) at g*S + pre[b], S = tiles of one head over all
    sequences) and cut into nvirt = sms // n_groups ranges of q or q + 1 tiles."""
    G = w.Hq // w.Hkv
    n_groups = -(-(-(-w.N * G // 128)) // 2)
    tiles = [-(-(int(w.prefix_len[b]) + w.N) // 128) for b in range(w.B)]
    pre = np.concatenate([[0], np.cumsum(tiles)])
    S = int(pre[-1])
    nvirt = sms // n_groups
    q, rem = divmod(w.Hkv * S, nvirt)
    for v in range(1, nvirt):
        x = v * q + min(v, rem)
        g, off = divmod(x, S)
        b = int(np.searchsorted(pre, off, side="right") - 1)
        if off > pre[b]:
            return b, g
    return None


def test_attention_c5_every_row_of_a_stream_k_cut_pair(jf):
    """Rows of a (sequence, kv-head) pair split between two stream-K ranges are merged by
    the boundary combine: check every row of the first such pair against the oracle."""
    w = cfg("c5_qwen3_30b_b8_tree256_32k")
    cut = first_stream_k_cut_pair(w, torch.cuda.get_device_properties(0).multi_processor_count)
    if cut is None:
        pytest.skip("every range boundary falls between pairs on this SM count")
    b, g = cut
    G = w.Hq // w.Hkv
    i, h = np.meshgrid(np.arange(w.N), np.arange(g * G, (g + 1) * G), indexing="ij")
    rows = (np.full(i.size, b), h.ravel(), i.ravel())
    out, lse, err = gpu_attention(jf, w)
    assert err == 0
    assert_attention_close(w, out, lse, rows)


SHAPES = [  # B, N, Hq, Hkv, D, P, tree
    (1, 1, 4, 1, 64, 0, "chain"),
    (1, 1, 8, 2, 128, 1, "chain"),
    (2, 5, 2, 2, 64, 15, "random"),
    (1, 16, 32, 8, 128, 16, "chain"),
    (3, 33, 4, 1, 128, 17, "random"),
    (1, 100, 8, 1, 64, 127, "random"),
    (2, 40, 8, 8, 128, 129, "random"),
    (1, 75, 4, 2, 128, 300, "random"),       # 150 rows -> a padded second row tile
    (1, 256, 16, 2, 128, 1000, "random"),    # G = 8, 16 row tiles
    (1, 130, 1, 1, 64, 70, "random"),        # G = 1, ragged multiword mask
    (1, 1024, 4, 1, 128, 64, "random"),      # many nodes, W = 16
    (2, 7, 128, 1, 64, 33, "random"),        # G = 128: one node per row tile
    (1, 2048, 2, 2, 64, 100, "random"),      # G = 1, W = 32: deep tree over many key tiles
    (1, 1, 4, 1, 64, 20000, "chain"),        # one unit, long prefix: > 16 splits to combine
    (1, 4, 8, 1, 128, 1500, "random"),       # one unit, 12 key tiles: 9..16 splits
    (1, 8, 8, 1, 128, 900, "random"),        # 5..8 splits
    (2, 8, 8, 2, 64, 800, "random"),         # 5..8 splits, D = 64
    (20, 128, 32, 4, 64, 300, "random"),     # 4 row-tile groups, 320 units: stream-K, D = 64
    (24, 64, 32, 4, 128, 90, "random"),      # 2 row-tile groups, 192 units: stream-K, D = 128
    (20, 40, 32, 4, 128, 3, "random"),       # stream-K over 1..6-tile pairs: many per range
    (20, 40, 32, 4, 128, 0, "random"),       # the same with sequence 0 unprefixed: 1..7-key rows
    (1, 12, 4, 1, 128, 0, "random"),         # no prefix, G = 4: rows of 1..7 keys (depth <= 6)
    (2, 24, 8, 1, 128, 0, "random"),         # no prefix in sequence 0, G = 8
    (3, 9, 8, 2, 64, 0, "chain"),            # no prefix, chain: row i sees i + 1 keys, D = 64
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%d_N%d_Hq%d_Hkv%d_D%d_P%d_%s" % s)
def test_attention_shapes_full_oracle(jf, shape):
    B, N, Hq, Hkv, D, P, tree = shape
    rng = np.random.default_rng(N * 7 + P)
    parent = None
    if tree == "random":
        parent = np.stack([np.array([-1] + [rng.integers(max(0, i - 6), i) for i in range(1, N)],
                                    np.int32) for _ in range(B)])
    prefix = np.array([P + 37 * b for b in range(B)], np.int32)
    w = wl.make_workload("shape", B, N, Hq, Hkv, D, 64, prefix, tree="chain", parent=parent,
                         permute_pages=True, seed=N + P, with_logits=False)
    out, lse, err = gpu_attention(jf, w)
    assert err == 0
    nrows = B * N * Hq
    rows = oracle.all_rows(w) if nrows <= 8192 else sample_rows(w, 2048)
    assert_attention_close(w, out, lse, rows)


@pytest.mark.parametrize("dispatch", ["stream_k", "splits"])
def test_attention_tiny_prefixes_full_oracle(jf, dispatch):
    """Prefixes of 0, 1 and 2 keys: rows see only a handful of keys, so the rounding of the
    probabilities does not average out.  Every row against the fp64 oracle.  20 sequences of
    40 nodes at G = 8 take the stream-K dispatch, 2 sequences the key-split one."""
    B = 20 if dispatch == "stream_k" else 2
    rng = np.random.default_rng(B)
    parent = np.stack([np.array([-1] + [rng.integers(max(0, i - 3), i) for i in range(1, 40)],
                                np.int32) for _ in range(B)])
    prefix = np.array([b % 3 for b in range(B)], np.int32)
    w = wl.make_workload("tiny", B, 40, 32, 4, 128, 64, prefix, tree="chain", parent=parent,
                         permute_pages=True, seed=77 + B, with_logits=False)
    out, lse, err = gpu_attention(jf, w)
    assert err == 0
    assert_attention_close(w, out, lse, oracle.all_rows(w) if B <= 2 else sample_rows(w, 6000))


def test_attention_single_root_without_prefix_is_v_root(jf):
    w = wl.make_workload("root", 2, 1, 8, 2, 128, 64, 0, tree="chain", seed=5, with_logits=False)
    out, _, err = gpu_attention(jf, w)
    for b in range(2):
        for h in range(8):
            v = wl.bf16_bits_to_f32(w.v_cache[w.block_table[b, 0], 0, h // 4])
            assert (out[b, 0, h] == v).all()


def test_attention_nan_in_unused_page_slots(jf):
    """Slots past P_b + N in the last page hold NaN; they must not leak into the output."""
    w = wl.make_workload("nan", 2, 19, 8, 2, 128, 64, np.array([46, 130], np.int32),
                         tree="random_depth_limited", seed=9, with_logits=False)
    for b in range(2):
        L = int(w.prefix_len[b]) + w.N
        for t in range(L, ((L + 15) // 16) * 16):
            pg = w.block_table[b, t // 16]
            w.k_cache[pg, t % 16] = wl.BF16_NAN
            w.v_cache[pg, t % 16] = wl.BF16_NAN
    out, lse, err = gpu_attention(jf, w)
    assert np.isfinite(out).all()
    assert_attention_close(w, out, lse, oracle.all_rows(w))


def test_attention_page_permutation_bit_identical(jf):
    a = wl.make_workload("pa", 2, 24, 8, 2, 128, 64, np.array([300, 77], np.int32),
                         tree="random_depth_limited", seed=3, with_logits=False)
    b = wl.make_workload("pb", 2, 24, 8, 2, 128, 64, np.array([300, 77], np.int32),
                         tree="random_depth_limited", seed=3, permute_pages=True, with_logits=False)
    for s in range(2):
        L = int(a.prefix_len[s]) + a.N
        for t in range(L):
            pa, pb = a.block_table[s, t // 16], b.block_table[s, t // 16]
            b.k_cache[pb, t % 16] = a.k_cache[pa, t % 16]
            b.v_cache[pb, t % 16] = a.v_cache[pa, t % 16]
    oa, la, _ = gpu_attention(jf, a)
    ob, lb, _ = gpu_attention(jf, b)
    assert (oa == ob).all() and (la == lb).all()


def test_attention_non_ancestor_kv_does_not_matter(jf):
    """Randomising K/V of every tree node outside node i's root path leaves row i
    bit-identical (masked weights are exactly zero)."""
    w = wl.make_workload("anc", 1, 48, 8, 2, 128, 64, 200, tree="random_depth_limited",
                         seed=12, with_logits=False)
    base, _, _ = gpu_attention(jf, w)
    rng = np.random.default_rng(1)
    for i in (0, 7, 47):
        anc = set()
        a = i
        while a >= 0:
            anc.add(a)
            a = int(w.parent[0, a])
        w2 = wl.make_workload("anc", 1, 48, 8, 2, 128, 64, 200, tree="random_depth_limited",
                              seed=12, with_logits=False)
        for j in range(48):
            if j not in anc:
                t = 200 + j
                pg = w2.block_table[0, t // 16]
                w2.k_cache[pg, t % 16] = wl.to_bf16_bits(rng.standard_normal((2, 128)).astype(np.float32) * 3)
                w2.v_cache[pg, t % 16] = wl.to_bf16_bits(rng.standard_normal((2, 128)).astype(np.float32) * 3)
        out, _, _ = gpu_attention(jf, w2)
        assert (out[0, i] == base[0, i]).all()


def test_attention_reports_bad_page_and_prefix(jf):
    w = wl.make_workload("bad", 2, 8, 4, 1, 64, 64, np.array([40, 40], np.int32), seed=1,
                         with_logits=False)
    t = wl.device_tensors(w, with_logits=False)
    t["block_table"][1, 1] = w.num_pages + 5
    mask, _, _ = jf.build_tree_mask(t["parent"], t["prefix_len"])
    err = dev_err()
    jf.tree_attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"], mask,
                      dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == jf.DEVERR_BAD_PAGE
    t = wl.device_tensors(w, with_logits=False)
    t["prefix_len"][0] = -3
    err = dev_err()
    jf.tree_attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"], mask,
                      dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == jf.DEVERR_BAD_PREFIX


def test_attention_back_to_back_calls_same_result(jf):
    w = cfg("c2_qwen3_8b_chain16")
    t = wl.device_tensors(w, with_logits=False)
    a, la, _ = gpu_attention(jf, w, t)
    b, lb, _ = gpu_attention(jf, w, t)
    assert (a == b).all() and (la == lb).all()
