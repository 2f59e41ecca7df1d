"""GPU parity for the packed (cu_seqlens) layout of ragged trees, the `_packed` calls.

Sequence b's n_b nodes sit at rows cu[b] .. cu[b + 1] - 1 of every per-node array, with
no padding rows.  A packed call must give, row for row, what the `_ragged` call gives on
the same trees in padded [B][N] arrays (same kernels and plan: bit for bit), and therefore
what the fp64 oracle gives on each sequence's slice (masks, argmax, accepted lengths,
paths, bonus tokens exactly; attention within |gpu - ref| <= 2e-3 + 1e-2 |ref|).  Output
buffers start as NaN: every packed row must be written, and a 128-row tile that reaches
into the next sequence must not overwrite that sequence's rows."""
import numpy as np
import pytest
import torch

import oracle
from test_gpu_ragged import RAGGED, check_rows, make, poison_padding
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jf():
    from tree_speculative_decoding_jf_gb300 import build
    build.build()
    from tree_speculative_decoding_jf_gb300 import jf as mod
    return mod


def cu_of(tree_len):
    return np.concatenate([[0], np.cumsum(tree_len)]).astype(np.int32)


def pack(a, tree_len):
    """[B][N][...] -> [T][...]: each sequence's first n_b rows, sequence after sequence."""
    return np.ascontiguousarray(np.concatenate([a[b, :n] for b, n in enumerate(tree_len)]))


def ragged_vs_packed_attention(jf, w, tree_len):
    B, N, Hq = w.B, w.N, w.Hq
    t = wl.device_tensors(w, with_logits=False)
    tl = torch.tensor(tree_len, dtype=torch.int32, device="cuda")
    cu_np = cu_of(tree_len)
    T = int(cu_np[-1])
    cu = torch.from_numpy(cu_np).cuda()
    nws = jf.jf_tree_attention_workspace_size(B, N, Hq, w.Hkv, w.D, w.max_pages, w.page)
    ws = torch.empty(max(16, nws), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # ragged reference (padded arrays)
    W = (N + 63) // 64
    mask_r = torch.empty((B, N, W), dtype=torch.int64, device="cuda")
    depth_r = torch.empty((B, N), dtype=torch.int32, device="cuda")
    pos_r = torch.empty((B, N), dtype=torch.int32, device="cuda")
    jf.jf_build_tree_mask_ragged(t["parent"], t["prefix_len"], tl, mask_r, depth_r, pos_r, err)
    out_r = torch.empty_like(t["q"])
    lse_r = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    jf.jf_tree_attention_ragged(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                t["prefix_len"], tl, mask_r, w.scale, out_r, lse_r, ws, err)
    # packed
    par_p = torch.from_numpy(pack(w.parent, tree_len)).cuda()
    q_p = torch.from_numpy(pack(w.q, tree_len).view(np.int16)).view(torch.bfloat16).cuda()
    mask_p = torch.full((T, W), -1, dtype=torch.int64, device="cuda")
    depth_p = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    pos_p = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    jf.jf_build_tree_mask_packed(par_p, t["prefix_len"], cu, N, mask_p, depth_p, pos_p, err)
    out_p = torch.full((T, Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse_p = torch.full((Hq, T), float("nan"), dtype=torch.float32, device="cuda")
    jf.jf_tree_attention_packed(q_p, t["k_cache"], t["v_cache"], t["block_table"],
                                t["prefix_len"], cu, N, mask_p, w.scale, out_p, lse_p, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    mr, mp = mask_r.cpu().numpy(), mask_p.cpu().numpy()
    assert (pack(mr, tree_len) == mp).all()
    assert (pack(depth_r.cpu().numpy(), tree_len) == depth_p.cpu().numpy()).all()
    assert (pack(pos_r.cpu().numpy(), tree_len) == pos_p.cpu().numpy()).all()
    o_r = out_r.view(torch.int16).cpu().numpy()
    o_p = out_p.view(torch.int16).cpu().numpy()
    assert (pack(o_r, tree_len) == o_p).all(), "packed rows differ from the ragged call's"
    l_r, l_p = lse_r.cpu().numpy(), lse_p.cpu().numpy()
    assert (pack(l_r.transpose(0, 2, 1), tree_len) == l_p.T).all()
    # back to the padded view for the oracle comparison (padding rows stay NaN)
    o = np.full((B, N, Hq, w.D), np.nan, np.float32)
    lse = np.full((B, Hq, N), np.nan, np.float32)
    of, lf = out_p.float().cpu().numpy(), l_p
    for b, n in enumerate(tree_len):
        o[b, :n] = of[cu_np[b]:cu_np[b + 1]]
        lse[b, :, :n] = lf[:, cu_np[b]:cu_np[b + 1]]
    return o, lse


@pytest.mark.parametrize("case", range(len(RAGGED)))
def test_packed_attention_equals_ragged_and_oracle(jf, case):
    B, N, Hq, Hkv, D, prefix, tree_len = RAGGED[case]
    rng = np.random.default_rng(300 + case)
    if prefix is None:
        prefix = rng.integers(100, 2000, B)
        tree_len = rng.integers(1, N + 1, B)
    tree_len = [int(x) for x in tree_len]
    w = poison_padding(make(B, N, Hq, Hkv, D, prefix, seed=17 + case), tree_len)
    o, lse = ragged_vs_packed_attention(jf, w, tree_len)
    check_rows(w, tree_len, o, lse, rows_per_seq=48 if B > 8 else 128, seed=case)


def test_packed_tiles_cross_sequence_boundaries(jf):
    """G = 8: a 128-row tile holds 16 nodes, and with these sizes nearly every sequence ends
    inside a tile whose remaining rows are the next sequence's first nodes."""
    tree_len = [5, 16, 17, 1, 31, 40, 9, 33]
    w = poison_padding(make(8, 48, 32, 4, 128, [300, 1500, 64, 2000, 700, 15, 900, 5], seed=23),
                       tree_len)
    o, lse = ragged_vs_packed_attention(jf, w, tree_len)
    check_rows(w, tree_len, o, lse, rows_per_seq=96, seed=5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [3001, 151936])      # one chunk per row, or several
def test_packed_verify_equals_ragged_and_oracle(jf, dtype, V):
    B, N = 6, 40
    w = wl.make_workload("pv", B, N, 4, 1, 64, V, 128, tree="random_depth_limited",
                         logits_dtype=dtype, forcing="half", seed=31 + V % 7)
    tree_len = [1, 2, 17, 39, 40, 23]
    lg = w.logits.reshape(B, N, V)
    am = oracle.argmax(lg, dtype).reshape(B, N)
    parent, draft = w.parent.copy(), w.draft.copy()
    for b, n in enumerate(tree_len):
        parent[b, n:] = 0                     # padding (never read by either call)
        draft[b, n:] = am[b, 0]
    to_dev = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()) \
        if dtype == "bf16" else (lambda a: torch.from_numpy(a).cuda())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tl = torch.tensor(tree_len, dtype=torch.int32, device="cuda")
    r_am, r_acc, r_path, r_bonus = jf.tree_verify(to_dev(np.ascontiguousarray(lg)),
                                                  torch.from_numpy(draft).cuda(),
                                                  torch.from_numpy(parent).cuda(), dev_err=err,
                                                  tree_len=tl)
    cu_np = cu_of(tree_len)
    T = int(cu_np[-1])
    lg_p = to_dev(pack(lg, tree_len))
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    bonus = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    am_p = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(jf.jf_tree_verify_packed_workspace_size(T, V), dtype=torch.uint8,
                     device="cuda")
    jf.jf_tree_verify_packed(lg_p, torch.from_numpy(pack(draft, tree_len)).cuda(),
                             torch.from_numpy(pack(parent, tree_len)).cuda(),
                             torch.from_numpy(cu_np).cuda(), N, acc, path, bonus, am_p, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert (am_p.cpu().numpy() == pack(am, tree_len)).all()
    assert (pack(r_am.cpu().numpy(), tree_len) == am_p.cpu().numpy()).all()
    assert torch.equal(acc, r_acc) and torch.equal(path, r_path) and torch.equal(bonus, r_bonus)
    acc, path, bonus = acc.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy()
    for b, n in enumerate(tree_len):
        o_acc, o_path, o_bonus = oracle.tree_walk(am[b:b + 1, :n], draft[b:b + 1, :n],
                                                  parent[b:b + 1, :n])
        assert acc[b] == o_acc[0] and bonus[b] == o_bonus[0]
        assert (path[b, :n] == o_path[0]).all() and (path[b, n:] == -1).all()
    assert acc.max() >= 2


def test_packed_bad_spans_are_reported_and_skipped(jf):
    """An empty span and one longer than N_max: both reported, neither sequence's rows
    touched, the valid sequence computed as usual."""
    B, N = 3, 16
    w = make(B, N, 4, 1, 64, [40, 40, 40], seed=5)
    t = wl.device_tensors(w, with_logits=False)
    cu_np = np.array([0, 0, 17, 20], np.int32)        # spans of 0, 17 (> N) and 3 nodes
    T = 20
    cu = torch.from_numpy(cu_np).cuda()
    par_p = torch.from_numpy(np.concatenate([w.parent[0], [0], w.parent[2, :3]])
                             .astype(np.int32)).cuda()
    q_p = torch.from_numpy(np.concatenate([w.q[0, :16], w.q[0, :1], w.q[2, :3]])
                           .view(np.int16)).view(torch.bfloat16).cuda()
    W = 1
    mask_p = torch.full((T, W), -1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    jf.jf_build_tree_mask_packed(par_p, t["prefix_len"], cu, N, mask_p, None, None, err)
    nws = jf.jf_tree_attention_workspace_size(B, N, w.Hq, w.Hkv, w.D, w.max_pages, w.page)
    ws = torch.empty(max(16, nws), dtype=torch.uint8, device="cuda")
    out_p = torch.full((T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    jf.jf_tree_attention_packed(q_p, t["k_cache"], t["v_cache"], t["block_table"],
                                t["prefix_len"], cu, N, mask_p, w.scale, out_p, None, ws, err)
    torch.cuda.synchronize()
    assert err.item() & jf.DEVERR_BAD_TREE_LEN
    m = mask_p.cpu().numpy()
    assert (m[:17] == -1).all()                       # the bad spans' rows untouched
    o = out_p.float().cpu().numpy()
    assert np.isnan(o[:17]).all() and np.isfinite(o[17:]).all()
    rm, _, _ = oracle.tree_mask(w.parent[2:3, :3], w.prefix_len[2:3])
    assert (m[17:, :1].view(np.uint64) == rm[0]).all()
