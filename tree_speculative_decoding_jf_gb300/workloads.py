"""Seeded synthetic inputs for tree-causal paged attention and greedy tree verify.

This module only draws random numbers and lays them out; it computes none of the
hot path (no ancestor sets, no attention, no argmax, no tree walk).  Both the CUDA
path and the CPU oracle read the arrays it returns.

Recipes (JetFlow explainer §4 names the workloads: Qwen3-8B / Qwen3-30B-A3B, draft
budgets 16 and 256; the pages print no tensors, so every tensor here is synthetic):

* Q/K/V: bf16 rounded (round-to-nearest-even) from fp32 N(0, 1) draws.
* Verify logits: N(0, 2) (second parameter = standard deviation), bf16 or fp32.
* Paged KV pool: ``k_cache``/``v_cache`` are ``[num_pages][page][Hkv][D]``; sequence b
  owns logical positions ``[0, P_b + N)``: the prefix, then the N tree nodes appended
  after it (node j at logical position ``P_b + j``).  Logical position t lives in
  ``page = block_table[b][t // page]``, slot ``t % page``.
* Trees: ``parent[b][0] = -1`` and ``0 <= parent[b][i] < i`` (topological order).
  - ``random_depth_limited``: ``parent[i]`` uniform over earlier nodes of depth < 6.
  - ``chain``: ``parent[i] = i - 1``.
  - ``best_first``: JetFlow explainer §2 (tree construction) ranks nodes by cumulative
    draft log-probability and expands best-first up to a budget.  Each node gets 8
    candidate children with log-probs ``log_softmax(N(0, 3) logits)`` and 8 distinct
    tokens drawn uniformly from the vocabulary; a max-heap on cumulative log-prob
    (ties: smaller parent id, then smaller candidate rank) pops the next node, which
    takes the next node id; candidates deeper than 16 levels are not pushed.
* Forced drafts ("children forced to equal their parent's argmax") are realised by
  planting a unique maximum (value 64.0, far above any N(0, 2) draw) at a random token
  of the parent's logits row and giving the forced child that token, so the generator
  never has to compute an argmax.

All random draws come from numpy PCG64 streams spawned from the config seed, so the
arrays are the same on every machine.
"""
from __future__ import annotations

import dataclasses
import heapq
import math
from typing import Optional

import numpy as np

PAGE = 16
PLANT = 64.0
BF16_NAN = 0x7FC0

# Component order of the spawned PCG64 streams (fixed; changing it changes every input).
_STREAMS = ("tree", "prefix", "q", "k", "v", "logits", "draft", "pages")


def _streams(seed: int) -> dict:
    ss = np.random.SeedSequence(seed)
    return {name: np.random.Generator(np.random.PCG64(s))
            for name, s in zip(_STREAMS, ss.spawn(len(_STREAMS)))}


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round-to-nearest-even (no NaNs expected)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0, chunk: int = 1 << 25):
    """bf16 bits of N(0, std) draws, generated in chunks to bound peak memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[s:e] = to_bf16_bits(x)
    return out.reshape(shape)


# ----------------------------------------------------------------------------- trees

def tree_chain(N: int) -> np.ndarray:
    return np.arange(-1, N - 1, dtype=np.int32)


def tree_star(N: int) -> np.ndarray:
    p = np.zeros(N, dtype=np.int32)
    p[0] = -1
    return p


def tree_random_depth_limited(rng, N: int, max_parent_depth: int = 5) -> np.ndarray:
    """parent[i] uniform over earlier nodes whose depth is < max_parent_depth + 1."""
    parent = np.full(N, -1, dtype=np.int32)
    depth = np.zeros(N, dtype=np.int64)
    for i in range(1, N):
        cand = np.nonzero(depth[:i] <= max_parent_depth)[0]
        p = int(cand[rng.integers(0, len(cand))])
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def tree_best_first(rng, N: int, V: int, n_cand: int = 8, sigma: float = 3.0,
                    max_levels: int = 16):
    """Best-first draft tree (input recipe).  Returns (parent, tokens)."""
    parent = [-1]
    depth = [0]
    score = [0.0]
    tokens = [int(rng.integers(0, V))]          # root token: the last accepted token
    heap = []

    def push_children(node):
        if depth[node] + 1 > max_levels - 1:
            return
        z = rng.standard_normal(n_cand) * sigma
        zmax = z.max()
        lp = z - zmax - math.log(np.exp(z - zmax).sum())
        toks = rng.choice(V, size=n_cand, replace=False)
        for r in range(n_cand):
            heapq.heappush(heap, (-(score[node] + float(lp[r])), node, r, int(toks[r])))

    push_children(0)
    while len(parent) < N:
        negs, p, _r, tok = heapq.heappop(heap)
        parent.append(p)
        depth.append(depth[p] + 1)
        score.append(-negs)
        tokens.append(tok)
        push_children(len(parent) - 1)
    return np.asarray(parent, dtype=np.int32), np.asarray(tokens, dtype=np.int32)


# ----------------------------------------------------------------------------- workload

@dataclasses.dataclass
class Workload:
    name: str
    B: int
    N: int
    Hq: int
    Hkv: int
    D: int
    V: int
    page: int
    scale: float
    prefix_len: np.ndarray      # int32 [B]
    parent: np.ndarray          # int32 [B][N]
    q: np.ndarray               # uint16 bf16 bits [B][N][Hq][D]
    k_cache: np.ndarray         # uint16 bf16 bits [num_pages][page][Hkv][D]
    v_cache: np.ndarray         # uint16 bf16 bits [num_pages][page][Hkv][D]
    block_table: np.ndarray     # int32 [B][max_pages], -1 past each sequence's pages
    logits: np.ndarray          # float32 or uint16 bf16 bits [B][N][V]
    logits_dtype: str           # "f32" | "bf16"
    draft: np.ndarray           # int32 [B][N] (draft[b][0] is the root token, not verified)
    seed: int

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def kv_len(self) -> np.ndarray:
        return self.prefix_len.astype(np.int64) + self.N


def make_workload(name: str, B: int, N: int, Hq: int, Hkv: int, D: int, V: int,
                  prefix_len, tree: str = "chain", logits_dtype: str = "bf16",
                  permute_pages: bool = False, forcing: str = "none", seed: int = 0,
                  page: int = PAGE, scale: Optional[float] = None,
                  parent: Optional[np.ndarray] = None,
                  with_logits: bool = True) -> Workload:
    rs = _streams(seed)
    prefix_len = np.broadcast_to(np.asarray(prefix_len, dtype=np.int32), (B,)).copy()

    # --- trees and their draft tokens
    parents = np.empty((B, N), dtype=np.int32)
    draft = np.empty((B, N), dtype=np.int32)
    for b in range(B):
        if parent is not None:
            parents[b] = parent[b] if parent.ndim == 2 else parent
            draft[b] = rs["draft"].integers(0, V, size=N)
        elif tree == "chain":
            parents[b] = tree_chain(N)
            draft[b] = rs["draft"].integers(0, V, size=N)
        elif tree == "star":
            parents[b] = tree_star(N)
            draft[b] = rs["draft"].integers(0, V, size=N)
        elif tree == "random_depth_limited":
            parents[b] = tree_random_depth_limited(rs["tree"], N)
            draft[b] = rs["draft"].integers(0, V, size=N)
        elif tree == "best_first":
            parents[b], draft[b] = tree_best_first(rs["tree"], N, V)
        else:
            raise ValueError(f"unknown tree kind {tree!r}")

    # --- paged KV pool
    pages_per_seq = (prefix_len.astype(np.int64) + N + page - 1) // page
    num_pages = int(pages_per_seq.sum())
    max_pages = int(pages_per_seq.max())
    order = np.arange(num_pages, dtype=np.int32)
    if permute_pages:
        order = rs["pages"].permutation(num_pages).astype(np.int32)
    block_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(pages_per_seq[b])
        block_table[b, :n] = order[off:off + n]
        off += n

    q = _normal_bf16(rs["q"], (B, N, Hq, D))
    k_cache = _normal_bf16(rs["k"], (num_pages, page, Hkv, D))
    v_cache = _normal_bf16(rs["v"], (num_pages, page, Hkv, D))

    # --- verify logits (N(0, 2)) and forced drafts (planted maxima)
    if with_logits:
        if logits_dtype == "f32":
            logits = (rs["logits"].standard_normal((B, N, V), dtype=np.float32) * np.float32(2.0))
            plant_val = np.float32(PLANT)
        else:
            logits = _normal_bf16(rs["logits"], (B, N, V), std=2.0)
            plant_val = to_bf16_bits(np.array([PLANT], dtype=np.float32))[0]
    else:
        logits = np.zeros((B, N, 0), dtype=np.float32 if logits_dtype == "f32" else np.uint16)
        plant_val = None
    rd = rs["draft"]
    if forcing != "none":
        if not with_logits:
            raise ValueError("forcing needs logits")
        for b in range(B):
            planted = {}

            def plant(row):
                if row not in planted:
                    t = int(rd.integers(0, V))
                    logits[b, row, t] = plant_val
                    planted[row] = t
                return planted[row]

            if forcing == "half":             # each non-root child forced w.p. 1/2
                coins = rd.random(N)
                for c in range(1, N):
                    if coins[c] < 0.5:
                        draft[b, c] = plant(int(parents[b, c]))
            elif forcing == "chain5":        # accepted path of exactly 5 draft nodes
                assert (parents[b] == tree_chain(N)).all() and N >= 7
                for c in range(1, 6):
                    draft[b, c] = plant(c - 1)
                t5 = plant(5)
                x = int(rd.integers(0, V - 1))
                draft[b, 6] = x if x < t5 else x + 1
            else:
                raise ValueError(f"unknown forcing {forcing!r}")

    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return Workload(name=name, B=B, N=N, Hq=Hq, Hkv=Hkv, D=D, V=V, page=page, scale=scale,
                    prefix_len=prefix_len, parent=parents, q=q, k_cache=k_cache,
                    v_cache=v_cache, block_table=block_table, logits=logits,
                    logits_dtype=logits_dtype, draft=draft, seed=seed)


# The five configurations (Qwen3-8B: Hq=32, Hkv=8, D=128; Qwen3-30B-A3B: Hq=32, Hkv=4,
# D=128; vocabulary 151936).  Seeds: 0 for the first, then the 0-based index.
CONFIGS = {
    "c1_tiny_random16": dict(B=1, N=16, Hq=4, Hkv=1, D=64, V=1024, prefix_len=128,
                             tree="random_depth_limited", logits_dtype="f32",
                             forcing="half", seed=0),
    "c2_qwen3_8b_chain16": dict(B=1, N=16, Hq=32, Hkv=8, D=128, V=151936, prefix_len=2048,
                                tree="chain", logits_dtype="bf16", forcing="chain5", seed=1),
    "c3_qwen3_8b_tree256": dict(B=1, N=256, Hq=32, Hkv=8, D=128, V=151936, prefix_len=4096,
                                tree="best_first", logits_dtype="bf16", seed=2),
    "c4_qwen3_8b_b32_tree64_paged": dict(B=32, N=64, Hq=32, Hkv=8, D=128, V=151936,
                                         prefix_len=None, tree="best_first",
                                         logits_dtype="bf16", permute_pages=True, seed=3),
    "c5_qwen3_30b_b8_tree256_32k": dict(B=8, N=256, Hq=32, Hkv=4, D=128, V=151936,
                                        prefix_len=32768, tree="best_first",
                                        logits_dtype="bf16", seed=4),
}
CONFIG_NAMES = list(CONFIGS)


def config(name: str, forcing: Optional[str] = None, with_logits: bool = True) -> Workload:
    """Build one of the five named workloads (optionally with a forced-draft variant)."""
    kw = dict(CONFIGS[name])
    if kw["prefix_len"] is None:    # per-sequence prefix uniform in [512, 8192]
        kw["prefix_len"] = _streams(kw["seed"])["prefix"].integers(512, 8193, size=kw["B"])
    if forcing is not None:
        kw["forcing"] = forcing
    if not with_logits:               # forced drafts only concern the verify logits
        kw["forcing"] = "none"
    return make_workload(name, with_logits=with_logits, **kw)


def device_tensors(w: Workload, device="cuda", with_logits: bool = True) -> dict:
    """Copy a workload's arrays into torch tensors on ``device`` (bf16 bit patterns are
    reinterpreted, not converted)."""
    import torch

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

    d = dict(q=bf16(w.q), k_cache=bf16(w.k_cache), v_cache=bf16(w.v_cache),
             block_table=i32(w.block_table), prefix_len=i32(w.prefix_len), parent=i32(w.parent),
             draft=i32(w.draft))
    if with_logits and w.logits.size:
        if w.logits_dtype == "f32":
            d["logits"] = torch.from_numpy(np.ascontiguousarray(w.logits)).to(device)
        else:
            d["logits"] = bf16(w.logits)
    return d

def random_accepted_paths(parent: np.ndarray, seed: int = 0):
    """Seeded synthetic verify outputs for the KV-compaction row: per sequence, a node
    drawn uniformly and its root path (node ids from the root, -1 padded) with the path's
    length in accepted draft nodes (the root excluded).  Returns (path, accept_len)."""
    parent = np.asarray(parent, dtype=np.int32)
    B, N = parent.shape
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x9A7E]))
    path = np.full((B, N), -1, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        node = int(rng.integers(0, N))
        chain = []
        while node >= 0:
            chain.append(node)
            node = int(parent[b, node])
        chain.reverse()
        path[b, :len(chain)] = chain
        acc[b] = len(chain) - 1
    return path, acc

def draft_logits(B: int, Dmax: int, V: int, sigma: float = 3.0, dtype: str = "bf16",
                 seed: int = 0) -> np.ndarray:
    """Seeded synthetic per-depth draft logits ~ N(0, sigma) (sigma a standard deviation),
    [B][Dmax][V]: bf16 bit patterns (uint16, round to nearest even) or float32."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0xD7AF]))
    x = (rng.standard_normal((B, Dmax, V), dtype=np.float32) * np.float32(sigma)).astype(np.float32)
    return to_bf16_bits(x) if dtype == "bf16" else x



def sampling_uniforms(B: int, N: int, seed: int = 0):
    """Seeded random numbers of stochastic verification: (uniform float32 [B][N],
    bonus_uniform float32 [B]), all in [0, 1)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x5A3F]))
    u = rng.random((B, N), dtype=np.float32)
    bu = rng.random(B, dtype=np.float32)
    return u, bu


# ----------------------------------------------------------------------------- sharding

def shard_sequences(B: int, rank: int, world: int) -> np.ndarray:
    """Sequences of one batch that rank `rank` of `world` owns when the batch is split
    across GPUs: b = rank, rank + world, ...  Sequences are independent through the whole
    path (mask, attention, verify), so the split needs no exchange."""
    if not (0 <= rank < world):
        raise ValueError(f"rank {rank} outside a world of {world}")
    return np.arange(rank, B, world, dtype=np.int64)


def sub_workload(w: Workload, seqs) -> Workload:
    """The workload of sequences `seqs` of `w`: every per-sequence array is taken in that
    order; the paged K/V pool is shared as is (the block-table rows keep their page ids)."""
    seqs = np.asarray(seqs, dtype=np.int64)
    if seqs.size == 0:
        raise ValueError("a shard needs at least one sequence")
    return dataclasses.replace(
        w, name=f"{w.name}[{','.join(str(int(b)) for b in seqs)}]", B=int(seqs.size),
        prefix_len=w.prefix_len[seqs].copy(), parent=w.parent[seqs].copy(), q=w.q[seqs].copy(),
        block_table=w.block_table[seqs].copy(), logits=w.logits[seqs].copy(),
        draft=w.draft[seqs].copy())
