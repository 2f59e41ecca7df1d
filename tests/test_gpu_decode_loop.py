"""A speculative-decoding loop through the whole path, several steps in a row, against the
fp64 oracle doing the same steps on CPU.

Each step: ragged draft trees (a seeded tree and budget per sequence), their queries and
keys/values written at positions P_b .. P_b + N - 1 of the paged pool (the target
forward pass's stand-in, the same values on both sides), then mask, attention and greedy
verification on the GPU, and the accepted path's K/V compacted next to the prefix; the
next step starts from the compacted pool and the new prefix lengths, which on the GPU side
stay on the device (the compaction's output is the next mask and attention calls' input,
with no host round trip between the steps).  The oracle runs mask,
attention rows, argmax, walk and compaction on its own copy of the state: masks, accepted
lengths, paths, bonus tokens, new prefix lengths and the whole pool must agree bit for bit
after every step, attention rows within 2e-3 + 1e-2 |ref|.  Nothing the GPU computes feeds
the oracle: the only shared inputs are the seeded trees, tokens, logits, queries and K/V."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from test_gpu_ragged import check_rows
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jf():
    from tree_speculative_decoding_jf_gb300 import build
    build.build()
    from tree_speculative_decoding_jf_gb300 import jf as mod
    return mod


def bf16_bits(rng, shape):
    return wl.to_bf16_bits(rng.standard_normal(shape).astype(np.float32))


@pytest.mark.parametrize("G,D", [(4, 128), (8, 64)])
def test_decode_loop_matches_oracle(jf, G, D):
    B, N, Hkv, V, steps = 4, 48, 2, 512, 4
    Hq = G * Hkv
    P0 = np.array([100, 37, 0, 513], np.int32)
    # pages for the prefix plus every step's tree: each step adds at most N positions
    base = wl.make_workload("loop", B, N, Hq, Hkv, D, V, P0 + steps * N, tree="chain",
                            permute_pages=True, seed=G * 10 + D, with_logits=False)
    rng = np.random.default_rng(G * 1000 + D)
    k_np, v_np, bt = base.k_cache.copy(), base.v_cache.copy(), base.block_table
    k_gpu = torch.from_numpy(k_np.view(np.int16)).view(torch.bfloat16).cuda()
    v_gpu = torch.from_numpy(v_np.view(np.int16)).view(torch.bfloat16).cuda()
    bt_gpu = torch.from_numpy(bt).cuda()
    P = P0.copy()
    P_dev = torch.from_numpy(P0).cuda()        # the GPU side keeps its prefix lengths on device
    total_accepted = 0
    for step in range(steps):
        tree_len = rng.integers(1, N + 1, B)
        tree_len[step % B] = N
        parent = np.full((B, N), -1, np.int32)
        for b in range(B):
            n = int(tree_len[b])
            parent[b, :n] = [-1] + [int(rng.integers(max(0, i - 5), i)) for i in range(1, n)]
        draft = rng.integers(0, V, (B, N)).astype(np.int32)
        q = bf16_bits(rng, (B, N, Hq, D))
        k_new, v_new = bf16_bits(rng, (B, N, Hkv, D)), bf16_bits(rng, (B, N, Hkv, D))
        # the forward pass's K/V of the tree nodes at positions P_b + i, on both sides
        slots = np.array([[bt[b, (P[b] + i) // 16] * 16 + (P[b] + i) % 16 for i in range(N)]
                          for b in range(B)], np.int64)
        k_np.reshape(-1, Hkv, D)[slots.reshape(-1)] = k_new.reshape(-1, Hkv, D)
        v_np.reshape(-1, Hkv, D)[slots.reshape(-1)] = v_new.reshape(-1, Hkv, D)
        idx = torch.from_numpy(slots.reshape(-1)).cuda()
        k_gpu.view(-1, Hkv, D)[idx] = torch.from_numpy(k_new.reshape(-1, Hkv, D).view(np.int16)) \
            .view(torch.bfloat16).cuda()
        v_gpu.view(-1, Hkv, D)[idx] = torch.from_numpy(v_new.reshape(-1, Hkv, D).view(np.int16)) \
            .view(torch.bfloat16).cuda()
        # target logits: about 60% of the nodes carry their parent's maximum
        logits = rng.standard_normal((B, N, V)).astype(np.float32)
        for b in range(B):
            for c in range(1, int(tree_len[b])):
                if rng.random() < 0.6:
                    logits[b, parent[b, c], draft[b, c]] = 10.0 + rng.random()
        w = dataclasses.replace(base, prefix_len=P.copy(), parent=parent, q=q, k_cache=k_np,
                                v_cache=v_np, logits=logits, logits_dtype="f32", draft=draft)

        # ---- GPU
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        tl = torch.from_numpy(tree_len.astype(np.int32)).cuda()
        t_par, t_P = torch.from_numpy(parent).cuda(), P_dev
        mask, depth, pos = jf.build_tree_mask(t_par, t_P, dev_err=err, tree_len=tl)
        out, lse = jf.tree_attention(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda(),
                                     k_gpu, v_gpu, bt_gpu, t_P, mask, scale=w.scale, with_lse=True,
                                     dev_err=err, tree_len=tl)
        am, acc, path, bonus = jf.tree_verify(torch.from_numpy(logits).cuda(),
                                              torch.from_numpy(draft).cuda(), t_par, dev_err=err,
                                              tree_len=tl)
        newp = jf.compact_accepted_kv(k_gpu, v_gpu, bt_gpu, t_P, path, acc, dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0, step

        # ---- oracle, sequence by sequence on each tree's slice
        m = mask.cpu().numpy().view(np.uint64)
        acc_g, path_g, bonus_g = acc.cpu().numpy(), path.cpu().numpy(), bonus.cpu().numpy()
        r_am = oracle.argmax(logits, "f32")
        r_path = np.full((B, N), -1, np.int32)
        r_acc = np.zeros(B, np.int32)
        for b in range(B):
            n = int(tree_len[b])
            rm, rd, rp = oracle.tree_mask(parent[b:b + 1, :n], P[b:b + 1])
            assert (m[b, :n, :rm.shape[-1]] == rm[0]).all(), (step, b)
            assert (depth.cpu().numpy()[b, :n] == rd[0]).all() and (pos.cpu().numpy()[b, :n] == rp[0]).all()
            a, pth, bn = oracle.tree_walk(r_am[b:b + 1, :n], draft[b:b + 1, :n], parent[b:b + 1, :n])
            r_acc[b], r_path[b, :n] = a[0], pth[0]
            assert acc_g[b] == a[0] and bonus_g[b] == bn[0], (step, b)
            assert (path_g[b] == r_path[b]).all(), (step, b)
        check_rows(w, [int(x) for x in tree_len], out.float().cpu().numpy(), lse.cpu().numpy(),
                   rows_per_seq=64, seed=step)
        rk, rv, rnewp, ok = oracle.compact_accepted_kv(k_np, v_np, bt, P, r_path, r_acc)
        assert ok and (newp.cpu().numpy() == rnewp).all(), step
        assert (k_gpu.view(torch.int16).cpu().numpy().view(np.uint16) == rk).all(), step
        assert (v_gpu.view(torch.int16).cpu().numpy().view(np.uint16) == rv).all(), step
        k_np, v_np, P = rk, rv, rnewp.astype(np.int32)
        P_dev = newp                            # compaction -> next step, no host round trip
        total_accepted += int(r_acc.sum())
    assert total_accepted >= steps * B          # the loop really moved the prefixes
    assert (P > P0).all()
