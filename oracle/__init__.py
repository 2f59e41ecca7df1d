"""fp64 CPU oracle for tree-causal paged attention and greedy tree verification.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU
baseline use it; the product path (the CUDA library and its binding) never imports it.
It is a thin ctypes layer over ``jf_oracle.c`` (plain C, fp64, OpenMP across rows), which
shares no code with the CUDA kernels.  See ``jf_oracle.c`` for the definitions followed.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jf_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile jf_oracle.c into liboracle.so with gcc (-O2 -fopenmp, no SIMD intrinsics)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.jfo_tree_mask.argtypes = [P, P, i32, i32, P, P, P]
        lib.jfo_tree_attention_rows.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                                i32, i32, f64, i64, P, P, P, P, P]
        lib.jfo_attention_probs.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                            i32, f64, i32, i32, P]
        lib.jfo_argmax_f32.argtypes = [P, i64, i64, P]
        lib.jfo_argmax_bf16.argtypes = [P, i64, i64, P]
        lib.jfo_tree_walk.argtypes = [P, P, P, i32, i32, P, P, P]
        lib.jfo_compact_accepted_kv.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                                i32, P]
        for f in ("jfo_tree_mask", "jfo_tree_attention_rows", "jfo_attention_probs",
                  "jfo_argmax_f32", "jfo_argmax_bf16", "jfo_tree_walk",
                  "jfo_compact_accepted_kv"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what}: oracle status {rc} ({'invalid tree' if rc == 2 else 'bad argument'})")


def tree_mask(parent, prefix_len):
    """parent int32 [B][N], prefix_len int32 [B] -> (mask uint64 [B][N][W], depth, pos)."""
    parent = _c(parent, np.int32)
    prefix_len = _c(prefix_len, np.int32)
    B, N = parent.shape
    W = (N + 63) // 64
    mask = np.zeros((B, N, W), dtype=np.uint64)
    depth = np.zeros((B, N), dtype=np.int32)
    pos = np.zeros((B, N), dtype=np.int32)
    _check(_load().jfo_tree_mask(_p(parent), _p(prefix_len), B, N, _p(mask), _p(depth), _p(pos)),
           "tree_mask")
    return mask, depth, pos


def tree_attention_rows(w, rows_b, rows_h, rows_i):
    """fp64 attention for the listed (b, h, i) rows of workload ``w``.
    Returns (out float64 [nrows][D], lse float64 [nrows])."""
    rb, rh, ri = (_c(r, np.int32) for r in (rows_b, rows_h, rows_i))
    n = len(rb)
    out = np.zeros((n, w.D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    q, kc, vc = _c(w.q, np.uint16), _c(w.k_cache, np.uint16), _c(w.v_cache, np.uint16)
    bt, pl, par = _c(w.block_table, np.int32), _c(w.prefix_len, np.int32), _c(w.parent, np.int32)
    _check(_load().jfo_tree_attention_rows(
        _p(q), _p(kc), _p(vc), _p(bt), _p(pl), _p(par), w.B, w.N, w.Hq, w.Hkv, w.D, w.page,
        w.max_pages, float(w.scale), n, _p(rb), _p(rh), _p(ri), _p(out), _p(lse)),
        "tree_attention_rows")
    return out, lse


def all_rows(w):
    """Every (b, h, i) row in [B][N][Hq] order (the layout of the output tensor)."""
    b, i, h = np.meshgrid(np.arange(w.B), np.arange(w.N), np.arange(w.Hq), indexing="ij")
    return b.ravel(), h.ravel(), i.ravel()


def tree_attention(w):
    """Full fp64 attention: (out float64 [B][N][Hq][D], lse float64 [B][Hq][N])."""
    rb, rh, ri = all_rows(w)
    out, lse = tree_attention_rows(w, rb, rh, ri)
    out = out.reshape(w.B, w.N, w.Hq, w.D)
    lse = lse.reshape(w.B, w.N, w.Hq).transpose(0, 2, 1).copy()
    return out, lse


def attention_probs(w, b, h):
    """Probability matrix [N][P_b + N] of one (b, h), zeros where masked."""
    L = int(w.prefix_len[b]) + w.N
    probs = np.zeros((w.N, L), dtype=np.float64)
    q, kc, vc = _c(w.q, np.uint16), _c(w.k_cache, np.uint16), _c(w.v_cache, np.uint16)
    bt, pl, par = _c(w.block_table, np.int32), _c(w.prefix_len, np.int32), _c(w.parent, np.int32)
    _check(_load().jfo_attention_probs(
        _p(q), _p(kc), _p(vc), _p(bt), _p(pl), _p(par), w.B, w.N, w.Hq, w.Hkv, w.D, w.page,
        w.max_pages, float(w.scale), int(b), int(h), _p(probs)), "attention_probs")
    return probs


def argmax(logits, dtype: str):
    """Row argmax, lowest index on ties, -0 == +0.  logits [..., V] as float32 ("f32")
    or bf16 bit patterns uint16 ("bf16")."""
    shape = logits.shape
    V = shape[-1]
    rows = int(np.prod(shape[:-1]))
    out = np.zeros(rows, dtype=np.int32)
    if dtype == "f32":
        x = _c(logits, np.float32)
        rc = _load().jfo_argmax_f32(_p(x), rows, V, _p(out))
    elif dtype == "bf16":
        x = _c(logits, np.uint16)
        rc = _load().jfo_argmax_bf16(_p(x), rows, V, _p(out))
    else:
        raise ValueError(dtype)
    _check(rc, "argmax")
    return out.reshape(shape[:-1])


def tree_walk(argmax_, draft, parent):
    """-> (accept_len int32 [B], path int32 [B][N] (-1 padded), bonus int32 [B])."""
    am, dr, par = _c(argmax_, np.int32), _c(draft, np.int32), _c(parent, np.int32)
    B, N = par.shape
    acc = np.zeros(B, dtype=np.int32)
    path = np.zeros((B, N), dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int32)
    _check(_load().jfo_tree_walk(_p(am), _p(dr), _p(par), B, N, _p(acc), _p(path), _p(bonus)),
           "tree_walk")
    return acc, path, bonus


def tree_verify(w):
    """Greedy verification of workload ``w``: (argmax, accept_len, path, bonus)."""
    am = argmax(w.logits, w.logits_dtype)
    acc, path, bonus = tree_walk(am, w.draft, w.parent)
    return am, acc, path, bonus


def compact_accepted_kv(k_cache: np.ndarray, v_cache: np.ndarray, block_table: np.ndarray,
                        prefix_len: np.ndarray, path: np.ndarray, accept_len: np.ndarray,
                        page: int = 16):
    """Accepted-path KV compaction on copies of the caches (see jfo_compact_accepted_kv).
    Returns (k_cache, v_cache, new_prefix_len, ok) where ok is False if any sequence was
    malformed (and left unchanged)."""
    k = np.ascontiguousarray(k_cache, dtype=np.uint16).copy()
    v = np.ascontiguousarray(v_cache, dtype=np.uint16).copy()
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    pl = np.ascontiguousarray(prefix_len, dtype=np.int32)
    pth = np.ascontiguousarray(path, dtype=np.int32)
    al = np.ascontiguousarray(accept_len, dtype=np.int32)
    B, N = pth.shape
    num_pages, pg, Hkv, D = k.shape
    assert pg == page
    newp = np.empty(B, np.int32)
    rc = _load().jfo_compact_accepted_kv(_p(k), _p(v), _p(bt), _p(pl), _p(pth), _p(al), B, N, Hkv,
                                         D, page, bt.shape[1], num_pages, _p(newp))
    return k, v, newp, rc == 0

