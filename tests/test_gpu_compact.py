"""GPU parity for accepted-path KV compaction (jf_compact_accepted_kv through the C ABI)
against the CPU oracle: the whole K/V pool and the new prefix lengths must match
bit-exactly."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jf():
    from tree_speculative_decoding_jf_gb300 import build
    build.build()
    from tree_speculative_decoding_jf_gb300 import jf as mod
    return mod


def run_both(jf, w, path, acc):
    t = wl.device_tensors(w, with_logits=False)
    tp = torch.from_numpy(np.ascontiguousarray(path, np.int32)).cuda()
    ta = torch.from_numpy(np.ascontiguousarray(acc, np.int32)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    newp = jf.compact_accepted_kv(t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"],
                                  tp, ta, dev_err=err)
    torch.cuda.synchronize()
    k = t["k_cache"].view(torch.int16).cpu().numpy().view(np.uint16)
    v = t["v_cache"].view(torch.int16).cpu().numpy().view(np.uint16)
    rk, rv, rnewp, ok = oracle.compact_accepted_kv(w.k_cache, w.v_cache, w.block_table,
                                                   w.prefix_len, path, acc)
    return (k, v, newp.cpu().numpy(), int(err.item())), (rk, rv, rnewp, ok)


@pytest.mark.parametrize("seed,D", [(0, 64), (1, 128), (2, 128), (3, 64)])
def test_compaction_random_paths_bit_exact(jf, seed, D):
    w = wl.make_workload("cmp", 4, 40, 8, 2, D, 64, np.array([0, 15, 130, 1000], np.int32),
                         tree="random_depth_limited", permute_pages=True, seed=seed,
                         with_logits=False)
    path, acc = wl.random_accepted_paths(w.parent, seed)
    (k, v, newp, err), (rk, rv, rnewp, ok) = run_both(jf, w, path, acc)
    assert ok and err == 0
    assert (newp == rnewp).all()
    assert (k == rk).all() and (v == rv).all()


def test_compaction_long_path_spans_chunks(jf):
    """parent[i] = i - 2: the path to node 78 is 0, 2, .., 78 (39 accepted nodes, more than
    one 32-node chunk), and every destination after the first is an earlier source."""
    N = 80
    parent = np.array([[-1] + [max(0, i - 2) for i in range(1, N)]] * 2, np.int32)
    w = wl.make_workload("long", 2, N, 4, 1, 128, 64, np.array([7, 200], np.int32),
                         tree="chain", parent=parent, permute_pages=True, seed=11,
                         with_logits=False)
    path = np.full((2, N), -1, np.int32)
    path[:, :40] = np.arange(0, 80, 2, dtype=np.int32)
    acc = np.array([39, 39], np.int32)
    (k, v, newp, err), (rk, rv, rnewp, ok) = run_both(jf, w, path, acc)
    assert ok and err == 0 and (newp == rnewp).all()
    assert (k == rk).all() and (v == rv).all()


def test_compaction_after_gpu_verify(jf):
    """The path and length the GPU verify writes feed the compaction directly."""
    w = wl.config("c1_tiny_random16")
    t = wl.device_tensors(w)
    am, acc, path, bonus = jf.tree_verify(t["logits"], t["draft"], t["parent"])
    torch.cuda.synchronize()
    p_np, a_np = path.cpu().numpy(), acc.cpu().numpy()
    (k, v, newp, err), (rk, rv, rnewp, ok) = run_both(jf, w, p_np, a_np)
    assert ok and err == 0 and (newp == rnewp).all()
    assert (k == rk).all() and (v == rv).all()


def test_compaction_malformed_path_leaves_sequence(jf):
    w = wl.make_workload("bad", 2, 6, 2, 1, 64, 64, np.array([4, 9], np.int32),
                         tree="chain", seed=6, with_logits=False)
    path = np.array([[0, 3, 2, -1, -1, -1], [0, 1, 2, -1, -1, -1]], np.int32)
    acc = np.array([2, 2], np.int32)
    (k, v, newp, err), (rk, rv, rnewp, ok) = run_both(jf, w, path, acc)
    assert not ok and (err & jf.DEVERR_BAD_PATH)
    assert (newp == rnewp).all() and newp[0] == 4
    assert (k == rk).all() and (v == rv).all()
