"""Vocabulary-sharded greedy verification across ranks (the layout of a vocabulary-parallel
output layer): gloo ranks on CPU each hold one token range of every node's logits, encode
their per-chunk maxima as the 8-byte keys the library exchanges (order-preserving value
bits, then 0xFFFFFFFF minus the global token id), all-gather them, take the unsigned
maximum per node and run the oracle's walk on the decoded ids.  Every rank must reach the
unsharded oracle's argmax, accepted lengths, paths and bonus tokens bit for bit, with the
maxima tied across ranges going to the lowest id and -0 equal to +0.  The keys are built
here from the oracle's argmax of each slice, so this checks the exchange protocol; the
GPU kernels that produce and merge the keys are checked against it in
test_gpu_shard_verify.py."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from conftest import ROOT

B, N, V, CHUNKS = 3, 20, 997, 4


def _logits(dtype: str):
    """Seeded logits [B][N][V] with maxima tied across the ranges of a 2- and 3-way split;
    float32 values, or bf16 bit patterns (uint16) for "bf16"."""
    sys.path.insert(0, ROOT)
    from tree_speculative_decoding_jf_gb300 import workloads as wl
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((B, N, V)) * 2).astype(np.float32)
    for r in range(0, B * N, 2):
        b, i = divmod(r, N)
        pos = [int(rng.integers(0, 300)), int(rng.integers(340, 660)), int(rng.integers(700, V))]
        if r % 3 == 0:
            x[b, i] = -x[b, i] ** 2 - 1.0
            x[b, i, pos] = [-0.0, 0.0, -0.0]
        else:
            x[b, i, pos] = 40.0
    return wl.to_bf16_bits(x) if dtype == "bf16" else x


def _tree():
    rng = np.random.default_rng(9)
    return np.stack([np.array([-1] + [rng.integers(0, i) for i in range(1, N)], np.int32)
                     for _ in range(B)])


def _values_f32(rows, dtype):
    if dtype == "bf16":
        return (rows.astype(np.uint32) << 16).view(np.float32)
    return rows.astype(np.float32)


def _ordered(v32):
    u = np.ascontiguousarray(v32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = np.where(u == 0x80000000, 0, u)
    return np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)


def range_keys(rows, dtype, offset, chunks):
    """Keys [B][N][chunks] of one token range (rows [B][N][V_range]) as int64 bit patterns:
    each slice's first maximum from the oracle's argmax, global id = offset + local id;
    slices past the range's end get key 0."""
    import oracle
    Vr = rows.shape[-1]
    clen = (-(-Vr // chunks) + 7) // 8 * 8
    keys = np.zeros(rows.shape[:-1] + (chunks,), dtype=np.uint64)
    for c in range(chunks):
        s, e = c * clen, min(Vr, (c + 1) * clen)
        if s >= Vr:
            continue
        seg = np.ascontiguousarray(rows[..., s:e])
        am = oracle.argmax(seg, dtype)
        val = _values_f32(np.take_along_axis(seg, am[..., None], -1)[..., 0], dtype)
        ids = (am.astype(np.uint64) + np.uint64(s + offset))
        keys[..., c] = (_ordered(val) << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - ids)
    return keys.view(np.int64)


def merge_keys(gathered):
    """gathered int64 [S][B][N][chunks] -> argmax int32 [B][N]: unsigned max, decoded id."""
    k = gathered.view(np.uint64).max(axis=(0, 3))
    return (np.uint64(0xFFFFFFFF) - (k & np.uint64(0xFFFFFFFF))).astype(np.int32)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, dtype, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    logits, parent = _logits(dtype), _tree()
    ref_am = oracle.argmax(logits, dtype)
    draft = ref_am[np.arange(B)[:, None], np.maximum(parent, 0)].astype(np.int32)
    draft[:, 1::5] = (draft[:, 1::5] + 1) % V               # some nodes rejected
    lo, hi = V * rank // world, V * (rank + 1) // world
    mine = torch.from_numpy(range_keys(np.ascontiguousarray(logits[..., lo:hi]), dtype, lo,
                                       CHUNKS))
    got = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(got, mine)
    am = merge_keys(torch.stack(got).numpy())
    acc, path, bonus = oracle.tree_walk(am, draft, parent)
    racc, rpath, rbonus = oracle.tree_walk(ref_am, draft, parent)
    ok = bool((am == ref_am).all() and (acc == racc).all() and (path == rpath).all()
              and (bonus == rbonus).all() and racc.max() >= 2)
    res = [None] * world
    dist.all_gather_object(res, ok)
    if rank == 0:
        q.put(res)
    dist.barrier()
    dist.destroy_process_group()


def test_range_keys_match_the_unsharded_argmax_single_process():
    """Without ranks: any split of the vocabulary, keys merged, gives the oracle's argmax."""
    sys.path.insert(0, ROOT)
    import oracle
    for dtype in ("f32", "bf16"):
        logits = _logits(dtype)
        ref = oracle.argmax(logits, dtype)
        for cuts in ([0, V], [0, 3, V], [0, 333, 664, V], [0, 1, 2, 500, V]):
            keys = [range_keys(np.ascontiguousarray(logits[..., a:b]), dtype, a, CHUNKS)
                    for a, b in zip(cuts[:-1], cuts[1:])]
            np.testing.assert_array_equal(merge_keys(np.stack(keys[::-1])), ref)


def test_signed_reduction_would_break_the_key_order():
    """The keys are unsigned: a positive maximum sets the top bit, so a signed MAX of the
    int64 storage picks the wrong range.  The exchange gathers and merges unsigned."""
    a = range_keys(np.array([[[1.0]]], np.float32), "f32", 0, 1)
    b = range_keys(np.array([[[-1.0]]], np.float32), "f32", 1, 1)
    assert a.view(np.uint64)[0, 0, 0] > b.view(np.uint64)[0, 0, 0]
    assert a[0, 0, 0] < b[0, 0, 0]


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_vocab_sharded_verify_gloo(world, dtype):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, dtype, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert res == [True] * world
