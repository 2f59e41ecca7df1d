"""GPU parity of vocabulary-sharded greedy verification: the logits of each node are cut
into token ranges (as a vocabulary-parallel output layer leaves them, one range per GPU),
each range's argmax keys come from jf_tree_verify_shard_keys, and jf_tree_verify_from_keys
walks the tree on all of them.  Here the ranges run one after another on one GPU and the
"all-gather" is a stack of their key tensors.  Argmax, accepted lengths, paths and bonus
tokens must equal both the unsharded jf_tree_verify and the fp64 oracle bit for bit,
including maxima tied across ranges (the lowest token id wins) and -0 against +0."""
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


def cuts(V, S, rng, ragged=True):
    """S token ranges covering [0, V): equal ranges, or random cut points off the 8-token
    grid with one range of at most three tokens."""
    if not ragged:
        b = [V * s // S for s in range(S + 1)]
    else:
        inner = sorted(rng.choice(np.arange(1, V), size=S - 1, replace=False).tolist())
        b = [0] + inner + [V]
        if V > 16 and S > 1:
            b[1] = int(rng.integers(1, 4))                  # a tiny first range
            b = sorted(set(b))
    return list(zip(b[:-1], b[1:]))


def ordered_bits(x32: np.ndarray) -> np.ndarray:
    """The documented key order of a float32 value: larger value, larger integer; -0 -> +0."""
    u = x32.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = np.where(u == 0x80000000, 0, u)
    return np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)


def sharded(jf, lg, ranges, order, chunks=None):
    B, N, V = lg.shape
    if chunks is None:
        chunks = max(jf.jf_tree_verify_shard_chunks(B, N, hi - lo) for lo, hi in ranges)
    keys = [None] * len(ranges)
    for s in order:
        lo, hi = ranges[s]
        keys[s] = jf.tree_verify_shard_keys(lg[:, :, lo:hi].contiguous(), lo, chunks)
    return torch.stack([keys[s] for s in order]), chunks


def plant(rng, x, ranges, tie_rows):
    """Each row in tie_rows gets its maximum at two or three tokens in different ranges;
    every third of them is all-negative with the maxima at -0 / +0."""
    B, N, V = x.shape
    for r in tie_rows:
        b, i = divmod(int(r), N)
        picks = rng.choice(len(ranges), size=min(3, len(ranges)), replace=False)
        pos = [int(rng.integers(*ranges[s])) for s in picks]
        if r % 3 == 0:
            x[b, i, :] = -x[b, i, :] ** 2 - 1.0
            for k, p in enumerate(pos):
                x[b, i, p] = -0.0 if k % 2 else 0.0
        else:
            x[b, i, pos] = 50.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,N,V,S,ragged", [
    (2, 16, 1001, 2, True),
    (3, 64, 32000, 4, True),
    (2, 256, 151936, 8, False),
    (4, 24, 151937, 3, True),
    (1, 1, 50, 2, True),
])
def test_sharded_verify_matches_unsharded_and_oracle(jf, dtype, B, N, V, S, ragged):
    rng = np.random.default_rng(B * 1000 + N + V + S)
    x = (rng.standard_normal((B, N, V)) * 2).astype(np.float32)
    ranges = cuts(V, S, rng, ragged)
    plant(rng, x, ranges, rng.choice(B * N, size=max(1, B * N // 2), replace=False))
    if dtype == "bf16":
        lg = torch.from_numpy(x).to(torch.bfloat16).cuda()
        ref_rows = lg.cpu().view(torch.int16).numpy().view(np.uint16)
    else:
        lg = torch.from_numpy(x).cuda()
        ref_rows = x
    parent = np.stack([np.array([-1] + [rng.integers(0, i) for i in range(1, N)], np.int32)
                       for _ in range(B)])
    ram = oracle.argmax(ref_rows, dtype)
    draft = np.where(rng.random((B, N)) < 0.7, ram[np.arange(B)[:, None], np.maximum(parent, 0)],
                     rng.integers(0, V, (B, N))).astype(np.int32)
    d, p = torch.from_numpy(draft).cuda(), torch.from_numpy(parent).cuda()
    order = rng.permutation(len(ranges)).tolist()
    keys, _ = sharded(jf, lg, ranges, order)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    am, acc, path, bonus = jf.tree_verify_from_keys(keys, V, d, p, dev_err=err)
    uam, uacc, upath, ubonus = jf.tree_verify(lg, d, p)
    racc, rpath, rbonus = oracle.tree_walk(ram, draft, parent)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert (am.cpu().numpy() == ram).all() and (am == uam).all()
    assert (acc.cpu().numpy() == racc).all() and (acc == uacc).all()
    assert (path.cpu().numpy() == rpath).all() and (path == upath).all()
    assert (bonus.cpu().numpy() == rbonus).all() and (bonus == ubonus).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_shard_keys_follow_the_documented_encoding(jf, dtype):
    """Every chunk key equals (ordered value bits) << 32 | (0xFFFFFFFF - global id of the
    chunk's first maximum); chunks past the range's end are 0."""
    rng = np.random.default_rng(7)
    B, N, Vs, off = 2, 5, 3001, 123457
    x = (rng.standard_normal((B, N, Vs)) * 3).astype(np.float32)
    x[0, 1, [10, 20, 2000]] = 30.0                   # ties inside one slice and across slices
    x[1, 2, :] = -np.abs(x[1, 2, :]) - 1
    x[1, 2, [5, 2999]] = [0.0, -0.0]
    if dtype == "bf16":
        t = torch.from_numpy(x).to(torch.bfloat16)
        vals = t.float().numpy()
    else:
        t = torch.from_numpy(x)
        vals = x
    chunks = 100                                     # slices of 32 tokens; the last six empty
    keys = jf.tree_verify_shard_keys(t.cuda(), off, chunks).cpu().numpy().view(np.uint64)
    clen = (-(-Vs // chunks) + 7) // 8 * 8
    for b in range(B):
        for i in range(N):
            for c in range(chunks):
                s, e = c * clen, min(Vs, (c + 1) * clen)
                if s >= Vs:
                    assert keys[b, i, c] == 0
                    continue
                seg = vals[b, i, s:e]
                m = seg.max()
                j = int(np.flatnonzero(seg == m)[0]) + s + off
                want = (int(ordered_bits(np.array([m]))[0]) << 32) | (0xFFFFFFFF - j)
                assert int(keys[b, i, c]) == want, (b, i, c)


def test_more_chunks_than_tokens_and_single_range(jf):
    """A range shorter than one slice per chunk, and S = 1 (the unsharded case)."""
    rng = np.random.default_rng(3)
    B, N, V = 2, 8, 40
    x = rng.standard_normal((B, N, V)).astype(np.float32)
    lg = torch.from_numpy(x).cuda()
    parent = np.stack([wl.tree_chain(N), wl.tree_star(N)]).astype(np.int32)
    ram = oracle.argmax(x, "f32")
    draft = ram[np.arange(B)[:, None], np.maximum(parent, 0)].astype(np.int32)
    d, p = torch.from_numpy(draft).cuda(), torch.from_numpy(parent).cuda()
    racc, rpath, rbonus = oracle.tree_walk(ram, draft, parent)
    for ranges, chunks in (([(0, 3), (3, 40)], 9), ([(0, 40)], 1), ([(0, 40)], 6)):
        keys, _ = sharded(jf, lg, ranges, list(range(len(ranges))), chunks)
        am, acc, path, bonus = jf.tree_verify_from_keys(keys, V, d, p)
        assert (am.cpu().numpy() == ram).all()
        assert (acc.cpu().numpy() == racc).all() and (path.cpu().numpy() == rpath).all()
        assert (bonus.cpu().numpy() == rbonus).all()
    assert racc[0] == N - 1                          # the chain is accepted to its end


def test_from_keys_reports_bad_tokens_and_parents(jf):
    lg = torch.randn(1, 4, 50, device="cuda")
    keys, _ = sharded(jf, lg, [(0, 20), (20, 50)], [1, 0])
    par = torch.tensor([[-1, 0, 0, 1]], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    jf.tree_verify_from_keys(keys, 50, torch.tensor([[0, 3, 99, 1]], dtype=torch.int32,
                                                    device="cuda"), par, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == jf.DEVERR_BAD_TOKEN
    err.zero_()
    jf.tree_verify_from_keys(keys, 50, torch.zeros(1, 4, dtype=torch.int32, device="cuda"),
                             torch.tensor([[-1, 0, 3, 1]], dtype=torch.int32, device="cuda"),
                             dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == jf.DEVERR_BAD_PARENT
