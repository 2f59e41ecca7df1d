"""Splitting one batch's sequences across ranks (the N > 1 layout of a serving job): two
gloo ranks on CPU each run the oracle on their shard of a 5-sequence batch, and the
gathered union must equal the single-rank result bit for bit (masks, attention outputs and
LSEs, argmax, accepted lengths, paths, bonus tokens).  The per-sequence independence that
this checks is what lets the GPU path shard by sequence with no data exchange."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _workload():
    sys.path.insert(0, ROOT)
    from tree_speculative_decoding_jf_gb300 import workloads as wl
    return wl.make_workload("shard5", B=5, N=16, Hq=4, Hkv=1, D=64, V=512,
                            prefix_len=[128, 37, 0, 300, 1], tree="random_depth_limited",
                            logits_dtype="f32", permute_pages=True, seed=11)


def _run(w):
    import oracle
    mask, depth, pos = oracle.tree_mask(w.parent, w.prefix_len)
    out, lse = oracle.tree_attention(w)
    am, acc, path, bonus = oracle.tree_verify(w)
    return {"mask": mask, "depth": depth, "pos": pos, "out": out, "lse": lse, "argmax": am, "acc": acc, "path": path,
            "bonus": bonus}


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from tree_speculative_decoding_jf_gb300 import workloads as wl
    w = _workload()
    seqs = wl.shard_sequences(w.B, rank, world)
    part = _run(wl.sub_workload(w, seqs))
    got = [None] * world
    dist.all_gather_object(got, (seqs.tolist(), part))
    if rank == 0:
        q.put(got)
    dist.barrier()
    dist.destroy_process_group()


def test_shard_sequences_cover_the_batch_once():
    sys.path.insert(0, ROOT)
    from tree_speculative_decoding_jf_gb300 import workloads as wl
    for B in (1, 2, 5, 8):
        for world in (1, 2, 3, 4):
            parts = [wl.shard_sequences(B, r, world) for r in range(world)]
            assert sorted(np.concatenate(parts).tolist()) == list(range(B))
    with pytest.raises(ValueError):
        wl.shard_sequences(4, 2, 2)


def test_sharded_oracle_equals_single_rank_gloo_world2():
    w = _workload()
    full = _run(w)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    seen = []
    for seqs, part in got:
        for k, b in enumerate(seqs):
            seen.append(b)
            for key in ("mask", "depth", "pos"):
                np.testing.assert_array_equal(part[key][k], full[key][b])
            np.testing.assert_array_equal(part["out"][k], full["out"][b])
            np.testing.assert_array_equal(part["lse"][k], full["lse"][b])
            np.testing.assert_array_equal(part["argmax"][k], full["argmax"][b])
            assert part["acc"][k] == full["acc"][b] and part["bonus"][k] == full["bonus"][b]
            np.testing.assert_array_equal(part["path"][k], full["path"][b])
    assert sorted(seen) == list(range(w.B))
