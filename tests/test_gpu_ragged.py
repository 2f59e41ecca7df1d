"""GPU parity for ragged trees (per-sequence tree sizes, the `_ragged` calls).

A ragged batch is defined by slicing: sequence b with n_b = tree_len[b] nodes must give
exactly what the fixed-size computation gives on the one-sequence problem made of its
first n_b nodes.  So the oracle runs on those slices (B = 1, N = n_b) and the GPU rows
i < n_b are compared with it: masks, accepted lengths and paths bit-exactly, attention
within |gpu - ref| <= 2e-3 + 1e-2 |ref|.  Padding is made hostile: parents and drafts of
padding nodes are out of range, their K/V slots hold NaN and block-table entries past each
sequence's last needed page are -1, so any read of them shows up as a device error or a
NaN.  With every tree_len equal to N the ragged calls must reproduce the fixed-size calls
bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
LSE_ATOL = 2e-3
BF16_NAN = np.uint16(0x7FC0)


@pytest.fixture(scope="module")
def jf():
    from tree_speculative_decoding_jf_gb300 import build
    build.build()
    from tree_speculative_decoding_jf_gb300 import jf as mod
    return mod


def dev_err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def slice_seq(w, b, n):
    """The one-sequence workload of sequence b's first n nodes."""
    return dataclasses.replace(
        w, B=1, N=n, prefix_len=w.prefix_len[b:b + 1].copy(),
        parent=w.parent[b:b + 1, :n].copy(), q=w.q[b:b + 1, :n].copy(),
        block_table=w.block_table[b:b + 1].copy(),
        logits=w.logits[b:b + 1, :n].copy() if w.logits.size else w.logits,
        draft=w.draft[b:b + 1, :n].copy())


def poison_padding(w, tree_len):
    """Out-of-range parents/drafts for padding nodes, NaN K/V in the padding slots and -1
    block-table entries past the pages a ragged sequence needs."""
    parent, draft = w.parent.copy(), w.draft.copy()
    kc, vc, bt = w.k_cache.copy(), w.v_cache.copy(), w.block_table.copy()
    for b, n in enumerate(tree_len):
        parent[b, n:] = 10 ** 6
        draft[b, n:] = -5
        P = int(w.prefix_len[b])
        for pos in range(P + n, P + w.N):
            page = bt[b, pos // w.page]
            if page >= 0:
                kc[page, pos % w.page] = BF16_NAN
                vc[page, pos % w.page] = BF16_NAN
        need = (P + n + w.page - 1) // w.page
        bt[b, need:] = -1
    return dataclasses.replace(w, parent=parent, draft=draft, k_cache=kc, v_cache=vc,
                               block_table=bt)


def ragged_attention(jf, w, tree_len):
    t = wl.device_tensors(w, with_logits=False)
    tl = torch.tensor(tree_len, dtype=torch.int32, device="cuda")
    err = dev_err()
    mask, _, _ = jf.build_tree_mask(t["parent"], t["prefix_len"], dev_err=err, tree_len=tl)
    out, lse = jf.tree_attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                 t["prefix_len"], mask, scale=w.scale, with_lse=True,
                                 dev_err=err, tree_len=tl)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(err.item())


def check_rows(w, tree_len, out, lse, rows_per_seq, seed=0):
    rng = np.random.default_rng(seed)
    for b, n in enumerate(tree_len):
        ws = slice_seq(w, b, n)
        k = min(rows_per_seq, n * w.Hq)
        ri = np.concatenate([[0, n - 1], rng.integers(0, n, k)]).astype(np.int32)
        rh = np.concatenate([[0, w.Hq - 1], rng.integers(0, w.Hq, k)]).astype(np.int32)
        rb = np.zeros_like(ri)
        ref_o, ref_l = oracle.tree_attention_rows(ws, rb, rh, ri)
        got = out[b, ri, rh]
        err = np.abs(got - ref_o)
        bad = err > ATOL + RTOL * np.abs(ref_o)
        assert not bad.any(), (f"sequence {b} (n={n}): {bad.sum()} elements out of tolerance, "
                               f"max abs err {err.max():.3e}")
        assert np.abs(lse[b, rh, ri] - ref_l).max() <= LSE_ATOL
    for b, n in enumerate(tree_len):     # padding rows carry no meaning (may be unwritten)
        assert np.isfinite(out[b, :n]).all()


def make(B, N, Hq, Hkv, D, prefix, seed, permute=True):
    rng = np.random.default_rng(seed)
    parent = np.stack([np.array([-1] + [rng.integers(max(0, i - 6), i) for i in range(1, N)],
                                np.int32) for _ in range(B)])
    return wl.make_workload("ragged", B, N, Hq, Hkv, D, 64, np.asarray(prefix, np.int32),
                            tree="chain", parent=parent, permute_pages=permute, seed=seed,
                            with_logits=False)


# (B, N, Hq, Hkv, D, prefixes, tree_len): plain dispatch with key splits, stream-K,
# longest-first dispatch and D = 64 / G = 1 with a one-node tree.
RAGGED = [
    (3, 64, 8, 2, 128, [0, 300, 1000], [1, 37, 64]),
    (8, 256, 32, 4, 128, [600, 1500, 977, 2000, 64, 1234, 15, 800],
     [256, 1, 100, 17, 255, 128, 200, 64]),
    (40, 16, 32, 8, 128, None, None),
    (2, 130, 2, 2, 64, [70, 5], [129, 1]),
]


@pytest.mark.parametrize("case", range(len(RAGGED)))
def test_ragged_attention_matches_slices(jf, case):
    B, N, Hq, Hkv, D, prefix, tree_len = RAGGED[case]
    rng = np.random.default_rng(100 + case)
    if prefix is None:
        prefix = rng.integers(100, 2000, B)
        tree_len = rng.integers(1, N + 1, B)
    tree_len = [int(x) for x in tree_len]
    w = poison_padding(make(B, N, Hq, Hkv, D, prefix, seed=7 + case), tree_len)
    out, lse, err = ragged_attention(jf, w, tree_len)
    assert err == 0
    check_rows(w, tree_len, out, lse, rows_per_seq=48 if B > 8 else 160, seed=case)


@pytest.mark.parametrize("shape", ["per_unit", "stream_k_sized"])
def test_ragged_full_length_matches_fixed_size(jf, shape):
    """Every tree at full size: the ragged call computes what the fixed-size call computes.
    Bit for bit when both take the same dispatch; the fixed-size call of the 8 x 256-node
    shape takes stream-K (ragged calls never do: stream-K ranges cannot skip padding row
    groups), so there the two agree within the attention tolerance."""
    if shape == "per_unit":
        w = make(3, 64, 8, 2, 128, [0, 300, 1000], seed=3)
    else:
        w = make(8, 256, 32, 4, 128, [600, 1500, 977, 2000, 64, 1234, 15, 800], seed=3)
    t = wl.device_tensors(w, with_logits=False)
    mask, depth, pos = jf.build_tree_mask(t["parent"], t["prefix_len"])
    ref = jf.tree_attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                            t["prefix_len"], mask, scale=w.scale, with_lse=True)
    tl = torch.full((w.B,), w.N, dtype=torch.int32, device="cuda")
    mask2, depth2, pos2 = jf.build_tree_mask(t["parent"], t["prefix_len"], tree_len=tl)
    got = jf.tree_attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                            t["prefix_len"], mask2, scale=w.scale, with_lse=True, tree_len=tl)
    torch.cuda.synchronize()
    assert torch.equal(mask, mask2) and torch.equal(depth, depth2) and torch.equal(pos, pos2)
    if shape == "per_unit":
        assert torch.equal(ref[0].view(torch.int16), got[0].view(torch.int16))
        assert torch.equal(ref[1], got[1])
    else:
        a, b = ref[0].float(), got[0].float()
        assert ((a - b).abs() <= ATOL + RTOL * a.abs()).all()
        assert (ref[1] - got[1]).abs().max().item() <= LSE_ATOL


def test_ragged_small_trees_skip_padding_groups(jf):
    """8 sequences of budget 256 at G = 8 (eight 256-row groups each) with trees of 1..63
    nodes: only the first group of each sequence holds real nodes.  Its rows must match the
    oracle; the call must leave the other groups' rows alone (they carry no meaning), which
    the poisoned output shows."""
    tree_len = [1, 5, 31, 32, 33, 63, 17, 2]
    w = poison_padding(make(8, 256, 32, 4, 128, [300, 1500, 64, 2000, 700, 15, 900, 5], seed=11),
                       tree_len)
    t = wl.device_tensors(w, with_logits=False)
    tl = torch.tensor(tree_len, dtype=torch.int32, device="cuda")
    mask, _, _ = jf.build_tree_mask(t["parent"], t["prefix_len"], tree_len=tl)
    out = torch.full_like(t["q"], float("nan"))
    lse = torch.full((w.B, w.Hq, w.N), float("nan"), device="cuda")
    nws = jf.jf_tree_attention_workspace_size(w.B, w.N, w.Hq, w.Hkv, w.D, w.max_pages, w.page)
    ws = torch.empty(max(16, nws), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    jf.jf_tree_attention_ragged(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                t["prefix_len"], tl, mask, w.scale, out, lse, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    o = out.float().cpu().numpy()
    check_rows(w, tree_len, o, lse.cpu().numpy(), rows_per_seq=64)
    G = w.Hq // w.Hkv
    per_group = 256 // G                 # nodes per 256-row group
    for b, n in enumerate(tree_len):     # rows of the padding-only groups stay untouched
        first_skipped = (n + per_group - 1) // per_group * per_group
        assert np.isnan(o[b, first_skipped:]).all()


def test_ragged_mask_matches_slices(jf):
    B, N = 6, 150
    rng = np.random.default_rng(11)
    parent = np.stack([np.array([-1] + [rng.integers(0, i) for i in range(1, N)], np.int32)
                       for _ in range(B)])
    prefix = rng.integers(0, 500, B).astype(np.int32)
    tree_len = [1, 2, 64, 65, 149, 150]
    par = parent.copy()
    for b, n in enumerate(tree_len):
        par[b, n:] = -99                       # malformed, but padding: never read
    err = dev_err()
    tl = torch.tensor(tree_len, dtype=torch.int32, device="cuda")
    mask, depth, pos = jf.build_tree_mask(torch.from_numpy(par).cuda(),
                                          torch.from_numpy(prefix).cuda(), dev_err=err,
                                          tree_len=tl)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    m = mask.cpu().numpy().view(np.uint64)
    d, p = depth.cpu().numpy(), pos.cpu().numpy()
    W = (N + 63) // 64
    for b, n in enumerate(tree_len):
        rm, rd, rp = oracle.tree_mask(parent[b:b + 1, :n], prefix[b:b + 1])
        Wn = rm.shape[-1]
        assert (m[b, :n, :Wn] == rm[0]).all() and (m[b, :n, Wn:] == 0).all()
        assert (d[b, :n] == rd[0]).all() and (p[b, :n] == rp[0]).all()
        assert (m[b, n:] == 0).all() and (d[b, n:] == -1).all() and (p[b, n:] == -1).all()
    assert m.shape == (B, N, W)


def test_ragged_verify_matches_slices_and_ignores_padding(jf):
    B, N, V = 5, 40, 1024
    w = wl.make_workload("rv", B, N, 4, 1, 64, V, 128, tree="random_depth_limited",
                         logits_dtype="f32", forcing="half", seed=21)
    tree_len = [1, 2, 17, 39, 40]
    am = oracle.argmax(w.logits, "f32").reshape(B, N)
    parent, draft = w.parent.copy(), w.draft.copy()
    for b, n in enumerate(tree_len):
        # padding children of the root carrying the root's argmax: accepted if not excluded
        parent[b, n:] = 0
        draft[b, n:] = am[b, 0]
    logits = torch.from_numpy(w.logits).cuda()
    tl = torch.tensor(tree_len, dtype=torch.int32, device="cuda")
    err = dev_err()
    g_am, acc, path, bonus = jf.tree_verify(logits, torch.from_numpy(draft).cuda(),
                                            torch.from_numpy(parent).cuda(), dev_err=err,
                                            tree_len=tl)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    acc, path, bonus = acc.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy()
    assert (g_am.cpu().numpy() == am).all()
    for b, n in enumerate(tree_len):
        r_acc, r_path, r_bonus = oracle.tree_walk(am[b:b + 1, :n], draft[b:b + 1, :n],
                                                  parent[b:b + 1, :n])
        assert acc[b] == r_acc[0] and bonus[b] == r_bonus[0]
        assert (path[b, :n] == r_path[0]).all() and (path[b, n:] == -1).all()


def test_ragged_tree_len_out_of_range_is_reported(jf):
    w = make(2, 16, 4, 1, 64, [40, 40], seed=5)
    t = wl.device_tensors(w, with_logits=False)
    tl = torch.tensor([0, 17], dtype=torch.int32, device="cuda")
    err = dev_err()
    mask, _, _ = jf.build_tree_mask(t["parent"], t["prefix_len"], dev_err=err, tree_len=tl)
    jf.tree_attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"],
                      mask, scale=w.scale, dev_err=err, tree_len=tl)
    torch.cuda.synchronize()
    assert int(err.item()) & jf.DEVERR_BAD_TREE_LEN
