"""Thin ctypes binding over libjf.so (declared in include/jf.h).

The functions named ``jf_*`` mirror the C entry points one to one: they take torch tensors
that already live on the GPU, check dtype/shape/contiguity, and pass raw pointers and the
current CUDA stream.  All computation happens in the library's kernels; there is no
fallback of any kind -- if libjf.so is missing or fails to load, importing this module
raises.  ``build_tree_mask``, ``tree_attention`` and ``tree_verify`` are conveniences that
also allocate the outputs (with torch) before calling the same entry points.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libjf.so")

JF_OK = 0
STATUS_NAMES = {0: "JF_OK", 1: "JF_ERR_INVALID_ARGUMENT", 2: "JF_ERR_INVALID_TREE",
                3: "JF_ERR_UNSUPPORTED", 4: "JF_ERR_WORKSPACE_TOO_SMALL", 5: "JF_ERR_CUDA",
                6: "JF_ERR_TIMEOUT", 7: "JF_ERR_MISALIGNED", 8: "JF_ERR_SCRATCH_CAPACITY"}
JF_DTYPE_BF16, JF_DTYPE_F32 = 0, 1
DEVERR_BAD_PARENT, DEVERR_BAD_PAGE, DEVERR_BAD_PREFIX = 0x1, 0x2, 0x4
DEVERR_BAD_TOKEN, DEVERR_TIMEOUT, DEVERR_BAD_PATH = 0x8, 0x10, 0x20
DEVERR_BAD_TREE_LEN = 0x40
MAX_NODES = 4096
PAGE_SIZE = 16


class JFError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m tree_speculative_decoding_jf_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    lib.jf_status_string.argtypes = [ctypes.c_int]
    lib.jf_status_string.restype = ctypes.c_char_p
    lib.jf_version.restype = ctypes.c_int
    lib.jf_build_tree_mask.argtypes = [P, P, i32, i32, P, P, P, P, P]
    lib.jf_build_tree_mask.restype = ctypes.c_int
    lib.jf_tree_attention_workspace_size.argtypes = [i32] * 7
    lib.jf_tree_attention_workspace_size.restype = sz
    lib.jf_tree_attention.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                      f32, P, P, P, sz, P, P]
    lib.jf_tree_attention.restype = ctypes.c_int
    lib.jf_tree_verify_workspace_size.argtypes = [i32, i32, i32]
    lib.jf_tree_verify_workspace_size.restype = sz
    lib.jf_tree_verify.argtypes = [P, i32, P, P, i32, i32, i32, P, P, P, P, P, sz, P, P]
    lib.jf_tree_verify.restype = ctypes.c_int
    lib.jf_tree_verify_static.argtypes = [P, i32, P, P, i32, i32, i32, P, P, P, P, P, P]
    lib.jf_tree_verify_static.restype = ctypes.c_int
    lib.jf_compact_accepted_kv.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                           P, P, P]
    lib.jf_compact_accepted_kv.restype = ctypes.c_int
    lib.jf_build_draft_tree.argtypes = [P, i32, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
    lib.jf_build_draft_tree_ragged.argtypes = [P, i32, P, P, i32, i32, i32, i32, i32, P, P, P, P,
                                               P, P, P, P]
    lib.jf_build_draft_tree_ragged.restype = ctypes.c_int
    lib.jf_build_draft_tree.restype = ctypes.c_int
    lib.jf_build_tree_mask_ragged.argtypes = [P, P, P, i32, i32, P, P, P, P, P]
    lib.jf_build_tree_mask_ragged.restype = ctypes.c_int
    lib.jf_tree_attention_ragged.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                             i32, i32, f32, P, P, P, sz, P, P]
    lib.jf_tree_attention_ragged.restype = ctypes.c_int
    lib.jf_tree_verify_ragged.argtypes = [P, i32, P, P, P, i32, i32, i32, P, P, P, P, P, sz, P, P]
    lib.jf_tree_verify_ragged.restype = ctypes.c_int
    lib.jf_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64, ctypes.c_int32]
    lib.jf_tree_verify_sampled.argtypes = [P, i32, P, P, P, P, f32, i32, i32, i32, P, P, P, P, sz,
                                           P, P]
    lib.jf_tree_verify_sampled.restype = ctypes.c_int
    lib.jf_debug_set_wait_limit_ns.restype = ctypes.c_int
    lib.jf_tree_verify_shard_chunks.argtypes = [i32, i32, i32]
    lib.jf_tree_verify_shard_chunks.restype = ctypes.c_int32
    lib.jf_tree_verify_shard_keys.argtypes = [P, i32, i32, i32, i32, i32, i32, P, P]
    lib.jf_tree_verify_shard_keys.restype = ctypes.c_int
    lib.jf_tree_verify_from_keys.argtypes = [P, i32, i32, P, P, i32, i32, i32, P, P, P, P, P, sz,
                                             P, P]
    lib.jf_tree_verify_from_keys.restype = ctypes.c_int
    lib.jf_build_tree_mask_packed.argtypes = [P, P, P, i32, i32, i32, P, P, P, P, P]
    lib.jf_build_tree_mask_packed.restype = ctypes.c_int
    lib.jf_tree_attention_packed.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                             i32, i32, i32, f32, P, P, P, sz, P, P]
    lib.jf_tree_attention_packed.restype = ctypes.c_int
    lib.jf_tree_verify_packed_workspace_size.argtypes = [i32, i32]
    lib.jf_tree_verify_packed_workspace_size.restype = sz
    lib.jf_tree_verify_packed.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, P, P, P, P, P, sz,
                                          P, P]
    lib.jf_tree_verify_packed.restype = ctypes.c_int
    lib.jf_tree_verify_sampled_ragged.argtypes = [P, i32, P, P, P, P, P, f32, i32, i32, i32, P, P,
                                                  P, P, sz, P, P]
    lib.jf_tree_verify_sampled_ragged.restype = ctypes.c_int
    lib.jf_tree_verify_sampled_packed.argtypes = [P, i32, P, P, P, P, P, f32, i32, i32, i32, i32,
                                                  P, P, P, P, sz, P, P]
    lib.jf_tree_verify_sampled_packed.restype = ctypes.c_int
    return lib


_lib = _load()
SIZE_MAX = ctypes.c_size_t(-1).value


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _check(fn: str, status: int):
    if status != JF_OK:
        raise JFError(fn, status)


def jf_status_string(status: int) -> str:
    return _lib.jf_status_string(status).decode()


def jf_version() -> int:
    return _lib.jf_version()


def jf_debug_set_wait_limit_ns(limit_ns: int, withhold_arrivals: bool = False) -> None:
    """Test hook: time limit of the attention kernels' pipeline waits on the current device,
    optionally with the data-arrival signals withheld so a wait can never complete
    ((0, False) restores normal operation).  See include/jf.h."""
    _check("jf_debug_set_wait_limit_ns",
           _lib.jf_debug_set_wait_limit_ns(int(limit_ns), 1 if withhold_arrivals else 0))


def jf_build_tree_mask(parent, prefix_len, mask, depth=None, pos=None, dev_err=None,
                       stream=None) -> None:
    _mask_call(parent, prefix_len, None, mask, depth, pos, dev_err, stream)


def jf_build_tree_mask_ragged(parent, prefix_len, tree_len, mask, depth=None, pos=None,
                              dev_err=None, stream=None) -> None:
    """Per-sequence tree sizes: nodes i >= tree_len[b] are padding (see include/jf.h)."""
    _need(tree_len, "tree_len", torch.int32, (parent.shape[0],))
    _mask_call(parent, prefix_len, tree_len, mask, depth, pos, dev_err, stream)


def _mask_call(parent, prefix_len, tree_len, mask, depth, pos, dev_err, stream) -> None:
    B, N = parent.shape
    W = (N + 63) // 64
    _need(parent, "parent", torch.int32)
    _need(prefix_len, "prefix_len", torch.int32, (B,))
    _need(mask, "mask", torch.int64, (B, N, W))
    for name, t in (("depth", depth), ("pos", pos)):
        if t is not None:
            _need(t, name, torch.int32, (B, N))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    if tree_len is None:
        _check("jf_build_tree_mask", _lib.jf_build_tree_mask(
            _ptr(parent), _ptr(prefix_len), B, N, _ptr(mask), _ptr(depth), _ptr(pos),
            _ptr(dev_err), _stream(stream)))
    else:
        _check("jf_build_tree_mask_ragged", _lib.jf_build_tree_mask_ragged(
            _ptr(parent), _ptr(prefix_len), _ptr(tree_len), B, N, _ptr(mask), _ptr(depth),
            _ptr(pos), _ptr(dev_err), _stream(stream)))


def jf_tree_attention_workspace_size(B, N, Hq, Hkv, D, max_pages, page_size=PAGE_SIZE) -> int:
    n = _lib.jf_tree_attention_workspace_size(B, N, Hq, Hkv, D, max_pages, page_size)
    if n == SIZE_MAX:
        raise JFError("jf_tree_attention_workspace_size", 3)
    return int(n)


def jf_tree_attention(q, k_cache, v_cache, block_table, prefix_len, mask, scale, out, lse=None,
                      workspace=None, dev_err=None, stream=None) -> None:
    _attention_call(q, k_cache, v_cache, block_table, prefix_len, None, mask, scale, out, lse,
                    workspace, dev_err, stream)


def jf_tree_attention_ragged(q, k_cache, v_cache, block_table, prefix_len, tree_len, mask,
                             scale, out, lse=None, workspace=None, dev_err=None,
                             stream=None) -> None:
    """Per-sequence tree sizes: sequence b's tree keys are P_b .. P_b + tree_len[b] - 1."""
    _need(tree_len, "tree_len", torch.int32, (q.shape[0],))
    _attention_call(q, k_cache, v_cache, block_table, prefix_len, tree_len, mask, scale, out,
                    lse, workspace, dev_err, stream)


def _attention_call(q, k_cache, v_cache, block_table, prefix_len, tree_len, mask, scale, out,
                    lse, workspace, dev_err, stream) -> None:
    B, N, Hq, D = q.shape
    num_pages, page, Hkv, D2 = k_cache.shape
    max_pages = block_table.shape[1]
    W = (N + 63) // 64
    _need(q, "q", torch.bfloat16)
    _need(k_cache, "k_cache", torch.bfloat16)
    _need(v_cache, "v_cache", torch.bfloat16, k_cache.shape)
    _need(block_table, "block_table", torch.int32, (B, max_pages))
    _need(prefix_len, "prefix_len", torch.int32, (B,))
    _need(mask, "mask", torch.int64, (B, N, W))
    _need(out, "out", torch.bfloat16, (B, N, Hq, D))
    if D2 != D:
        raise ValueError("q and k_cache head dims differ")
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, Hq, N))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    ws_bytes = 0
    if workspace is not None:
        if workspace.device.type != "cuda" or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    if tree_len is None:
        _check("jf_tree_attention", _lib.jf_tree_attention(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(prefix_len),
            _ptr(mask), B, N, Hq, Hkv, D, page, max_pages, num_pages, float(scale), _ptr(out),
            _ptr(lse), _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream)))
    else:
        _check("jf_tree_attention_ragged", _lib.jf_tree_attention_ragged(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(prefix_len),
            _ptr(tree_len), _ptr(mask), B, N, Hq, Hkv, D, page, max_pages, num_pages,
            float(scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(dev_err),
            _stream(stream)))


def jf_tree_verify_workspace_size(B, N, V) -> int:
    n = _lib.jf_tree_verify_workspace_size(B, N, V)
    if n == SIZE_MAX:
        raise JFError("jf_tree_verify_workspace_size", 3)
    return int(n)


def jf_tree_verify(logits, draft, parent, accept_len, path, bonus, argmax=None, workspace=None,
                   dev_err=None, stream=None) -> None:
    _verify_call(logits, draft, parent, None, accept_len, path, bonus, argmax, workspace,
                 dev_err, stream)


def jf_tree_verify_ragged(logits, draft, parent, tree_len, accept_len, path, bonus, argmax=None,
                          workspace=None, dev_err=None, stream=None) -> None:
    """Per-sequence tree sizes: nodes i >= tree_len[b] are never accepted."""
    _need(tree_len, "tree_len", torch.int32, (logits.shape[0],))
    _verify_call(logits, draft, parent, tree_len, accept_len, path, bonus, argmax, workspace,
                 dev_err, stream)


def jf_tree_verify_sampled(logits, draft, parent, uniform, bonus_uniform, temperature,
                           accept_len, path, bonus, workspace, dev_err=None, stream=None) -> None:
    """Lossless (stochastic) verification; uniform float32 [B][N] and bonus_uniform float32
    [B] are the random numbers in [0, 1) (see include/jf.h).  The workspace is sized by
    jf_tree_verify_workspace_size."""
    B, N, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = JF_DTYPE_BF16
    elif logits.dtype == torch.float32:
        dt = JF_DTYPE_F32
    else:
        raise TypeError("logits must be bfloat16 or float32")
    _need(logits, "logits", logits.dtype)
    _need(draft, "draft", torch.int32, (B, N))
    _need(parent, "parent", torch.int32, (B, N))
    _need(uniform, "uniform", torch.float32, (B, N))
    _need(bonus_uniform, "bonus_uniform", torch.float32, (B,))
    _need(accept_len, "accept_len", torch.int32, (B,))
    _need(path, "path", torch.int32, (B, N))
    _need(bonus, "bonus", torch.int32, (B,))
    _need(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    _check("jf_tree_verify_sampled", _lib.jf_tree_verify_sampled(
        _ptr(logits), dt, _ptr(draft), _ptr(parent), _ptr(uniform), _ptr(bonus_uniform),
        float(temperature), B, N, V, _ptr(accept_len), _ptr(path), _ptr(bonus), _ptr(workspace),
        workspace.numel(), _ptr(dev_err), _stream(stream)))


def _verify_call(logits, draft, parent, tree_len, accept_len, path, bonus, argmax, workspace,
                 dev_err, stream) -> None:
    B, N, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = JF_DTYPE_BF16
    elif logits.dtype == torch.float32:
        dt = JF_DTYPE_F32
    else:
        raise TypeError("logits must be bfloat16 or float32")
    _need(logits, "logits", logits.dtype)
    _need(draft, "draft", torch.int32, (B, N))
    _need(parent, "parent", torch.int32, (B, N))
    _need(accept_len, "accept_len", torch.int32, (B,))
    _need(path, "path", torch.int32, (B, N))
    _need(bonus, "bonus", torch.int32, (B,))
    if argmax is not None:
        _need(argmax, "argmax", torch.int32, (B, N))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    ws_bytes = 0
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
    if tree_len is None:
        _check("jf_tree_verify", _lib.jf_tree_verify(
            _ptr(logits), dt, _ptr(draft), _ptr(parent), B, N, V, _ptr(argmax),
            _ptr(accept_len), _ptr(path), _ptr(bonus), _ptr(workspace), ws_bytes, _ptr(dev_err),
            _stream(stream)))
    else:
        _check("jf_tree_verify_ragged", _lib.jf_tree_verify_ragged(
            _ptr(logits), dt, _ptr(draft), _ptr(parent), _ptr(tree_len), B, N, V, _ptr(argmax),
            _ptr(accept_len), _ptr(path), _ptr(bonus), _ptr(workspace), ws_bytes, _ptr(dev_err),
            _stream(stream)))


def jf_tree_verify_static(logits, draft, parent, accept_len, path, bonus, argmax=None,
                          dev_err=None, stream=None) -> None:
    """jf_tree_verify without a workspace: the library's fixed scratch array is used
    (see include/jf.h for its capacity and the rules for concurrent calls)."""
    B, N, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = JF_DTYPE_BF16
    elif logits.dtype == torch.float32:
        dt = JF_DTYPE_F32
    else:
        raise TypeError("logits must be bfloat16 or float32")
    _need(logits, "logits", logits.dtype)
    for name, t, shape in (("draft", draft, (B, N)), ("parent", parent, (B, N)),
                           ("accept_len", accept_len, (B,)), ("path", path, (B, N)),
                           ("bonus", bonus, (B,))):
        _need(t, name, torch.int32, shape)
    if argmax is not None:
        _need(argmax, "argmax", torch.int32, (B, N))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    _check("jf_tree_verify_static", _lib.jf_tree_verify_static(
        _ptr(logits), dt, _ptr(draft), _ptr(parent), B, N, V, _ptr(argmax), _ptr(accept_len),
        _ptr(path), _ptr(bonus), _ptr(dev_err), _stream(stream)))


def jf_tree_verify_shard_chunks(B, N, V_shard) -> int:
    n = _lib.jf_tree_verify_shard_chunks(B, N, V_shard)
    if n < 0:
        raise JFError("jf_tree_verify_shard_chunks", 3)
    return int(n)


def jf_tree_verify_shard_keys(logits_shard, vocab_offset, keys, stream=None) -> None:
    """Argmax keys of one vocabulary range: logits_shard [B][N][V_shard] (bf16 or f32) holds
    the tokens vocab_offset .. vocab_offset + V_shard - 1; keys is int64 [B][N][chunks]
    (the uint64 keys' bits).  See include/jf.h."""
    B, N, Vs = logits_shard.shape
    if logits_shard.dtype == torch.bfloat16:
        dt = JF_DTYPE_BF16
    elif logits_shard.dtype == torch.float32:
        dt = JF_DTYPE_F32
    else:
        raise TypeError("logits_shard must be bfloat16 or float32")
    _need(logits_shard, "logits_shard", logits_shard.dtype)
    _need(keys, "keys", torch.int64)
    if keys.dim() != 3 or tuple(keys.shape[:2]) != (B, N):
        raise ValueError(f"keys has shape {tuple(keys.shape)}, expected ({B}, {N}, chunks)")
    _check("jf_tree_verify_shard_keys", _lib.jf_tree_verify_shard_keys(
        _ptr(logits_shard), dt, B, N, Vs, int(vocab_offset), keys.shape[2], _ptr(keys),
        _stream(stream)))


def jf_tree_verify_from_keys(keys, V, draft, parent, accept_len, path, bonus, workspace,
                             argmax=None, dev_err=None, stream=None) -> None:
    """The greedy walk on every range's keys, int64 [S][B][N][chunks] (an all-gather of
    jf_tree_verify_shard_keys' outputs); workspace uint8 of at least 8*B*N bytes."""
    S, B, N, chunks = keys.shape
    _need(keys, "keys", torch.int64)
    for name, t, shape in (("draft", draft, (B, N)), ("parent", parent, (B, N)),
                           ("accept_len", accept_len, (B,)), ("path", path, (B, N)),
                           ("bonus", bonus, (B,))):
        _need(t, name, torch.int32, shape)
    _need(workspace, "workspace", torch.uint8)
    if argmax is not None:
        _need(argmax, "argmax", torch.int32, (B, N))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    _check("jf_tree_verify_from_keys", _lib.jf_tree_verify_from_keys(
        _ptr(keys), S, chunks, _ptr(draft), _ptr(parent), B, N, int(V), _ptr(argmax),
        _ptr(accept_len), _ptr(path), _ptr(bonus), _ptr(workspace), workspace.numel(),
        _ptr(dev_err), _stream(stream)))


def jf_build_tree_mask_packed(parent, prefix_len, cu_seqlens, N_max, mask, depth=None, pos=None,
                              dev_err=None, stream=None) -> None:
    """Packed trees: parent int32 [T] (ids within each sequence), cu_seqlens int32 [B + 1],
    mask int64 [T][ceil(N_max / 64)] (see include/jf.h)."""
    (T,) = parent.shape
    B = cu_seqlens.shape[0] - 1
    W = (N_max + 63) // 64
    _need(parent, "parent", torch.int32)
    _need(prefix_len, "prefix_len", torch.int32, (B,))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (B + 1,))
    _need(mask, "mask", torch.int64, (T, W))
    for name, t in (("depth", depth), ("pos", pos)):
        if t is not None:
            _need(t, name, torch.int32, (T,))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    _check("jf_build_tree_mask_packed", _lib.jf_build_tree_mask_packed(
        _ptr(parent), _ptr(prefix_len), _ptr(cu_seqlens), B, N_max, T, _ptr(mask), _ptr(depth),
        _ptr(pos), _ptr(dev_err), _stream(stream)))


def jf_tree_attention_packed(q, k_cache, v_cache, block_table, prefix_len, cu_seqlens, N_max,
                             mask, scale, out, lse=None, workspace=None, dev_err=None,
                             stream=None) -> None:
    """Packed trees: q and out bf16 [T][Hq][D], mask int64 [T][W], lse float32 [Hq][T];
    the workspace is sized by jf_tree_attention_workspace_size with N = N_max."""
    T, Hq, D = q.shape
    num_pages, page, Hkv, D2 = k_cache.shape
    B = cu_seqlens.shape[0] - 1
    max_pages = block_table.shape[1]
    W = (N_max + 63) // 64
    _need(q, "q", torch.bfloat16)
    _need(k_cache, "k_cache", torch.bfloat16)
    _need(v_cache, "v_cache", torch.bfloat16, k_cache.shape)
    _need(block_table, "block_table", torch.int32, (B, max_pages))
    _need(prefix_len, "prefix_len", torch.int32, (B,))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (B + 1,))
    _need(mask, "mask", torch.int64, (T, W))
    _need(out, "out", torch.bfloat16, (T, Hq, D))
    if D2 != D:
        raise ValueError("q and k_cache head dims differ")
    if lse is not None:
        _need(lse, "lse", torch.float32, (Hq, T))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    ws_bytes = 0
    if workspace is not None:
        if workspace.device.type != "cuda" or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("jf_tree_attention_packed", _lib.jf_tree_attention_packed(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(prefix_len),
        _ptr(cu_seqlens), _ptr(mask), B, N_max, T, Hq, Hkv, D, page, max_pages, num_pages,
        float(scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(dev_err),
        _stream(stream)))


def jf_tree_verify_packed_workspace_size(T, V) -> int:
    n = _lib.jf_tree_verify_packed_workspace_size(T, V)
    if n == SIZE_MAX:
        raise JFError("jf_tree_verify_packed_workspace_size", 3)
    return int(n)


def jf_tree_verify_packed(logits, draft, parent, cu_seqlens, N_max, accept_len, path, bonus,
                          argmax=None, workspace=None, dev_err=None, stream=None) -> None:
    """Packed trees: logits [T][V] (bf16 or f32), draft/parent/argmax int32 [T], path int32
    [B][N_max]; the workspace is sized by jf_tree_verify_packed_workspace_size(T, V)."""
    T, V = logits.shape
    B = cu_seqlens.shape[0] - 1
    if logits.dtype == torch.bfloat16:
        dt = JF_DTYPE_BF16
    elif logits.dtype == torch.float32:
        dt = JF_DTYPE_F32
    else:
        raise TypeError("logits must be bfloat16 or float32")
    _need(logits, "logits", logits.dtype)
    for name, t, shape in (("draft", draft, (T,)), ("parent", parent, (T,)),
                           ("cu_seqlens", cu_seqlens, (B + 1,)), ("accept_len", accept_len, (B,)),
                           ("path", path, (B, N_max)), ("bonus", bonus, (B,))):
        _need(t, name, torch.int32, shape)
    if argmax is not None:
        _need(argmax, "argmax", torch.int32, (T,))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("jf_tree_verify_packed", _lib.jf_tree_verify_packed(
        _ptr(logits), dt, _ptr(draft), _ptr(parent), _ptr(cu_seqlens), B, N_max, T, V,
        _ptr(argmax), _ptr(accept_len), _ptr(path), _ptr(bonus), _ptr(workspace), ws_bytes,
        _ptr(dev_err), _stream(stream)))


def jf_tree_verify_sampled_ragged(logits, draft, parent, tree_len, uniform, bonus_uniform,
                                  temperature, accept_len, path, bonus, workspace, dev_err=None,
                                  stream=None) -> None:
    """Lossless verification with per-sequence tree sizes (padded [B][N] arrays, tree_len
    int32 [B]); the workspace is sized by jf_tree_verify_workspace_size."""
    B, N, V = logits.shape
    dt = _logit_dtype(logits)
    _need(logits, "logits", logits.dtype)
    for name, t, shape in (("draft", draft, (B, N)), ("parent", parent, (B, N)),
                           ("tree_len", tree_len, (B,)), ("accept_len", accept_len, (B,)),
                           ("path", path, (B, N)), ("bonus", bonus, (B,))):
        _need(t, name, torch.int32, shape)
    _need(uniform, "uniform", torch.float32, (B, N))
    _need(bonus_uniform, "bonus_uniform", torch.float32, (B,))
    _need(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    _check("jf_tree_verify_sampled_ragged", _lib.jf_tree_verify_sampled_ragged(
        _ptr(logits), dt, _ptr(draft), _ptr(parent), _ptr(tree_len), _ptr(uniform),
        _ptr(bonus_uniform), float(temperature), B, N, V, _ptr(accept_len), _ptr(path),
        _ptr(bonus), _ptr(workspace), workspace.numel(), _ptr(dev_err), _stream(stream)))


def jf_tree_verify_sampled_packed(logits, draft, parent, cu_seqlens, N_max, uniform,
                                  bonus_uniform, temperature, accept_len, path, bonus, workspace,
                                  dev_err=None, stream=None) -> None:
    """Lossless verification of packed trees: logits [T][V], draft/parent int32 [T], uniform
    float32 [T], path int32 [B][N_max]; the workspace is sized by
    jf_tree_verify_packed_workspace_size(T, V)."""
    T, V = logits.shape
    B = cu_seqlens.shape[0] - 1
    dt = _logit_dtype(logits)
    _need(logits, "logits", logits.dtype)
    for name, t, shape in (("draft", draft, (T,)), ("parent", parent, (T,)),
                           ("cu_seqlens", cu_seqlens, (B + 1,)), ("accept_len", accept_len, (B,)),
                           ("path", path, (B, N_max)), ("bonus", bonus, (B,))):
        _need(t, name, torch.int32, shape)
    _need(uniform, "uniform", torch.float32, (T,))
    _need(bonus_uniform, "bonus_uniform", torch.float32, (B,))
    _need(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    _check("jf_tree_verify_sampled_packed", _lib.jf_tree_verify_sampled_packed(
        _ptr(logits), dt, _ptr(draft), _ptr(parent), _ptr(cu_seqlens), _ptr(uniform),
        _ptr(bonus_uniform), float(temperature), B, N_max, T, V, _ptr(accept_len), _ptr(path),
        _ptr(bonus), _ptr(workspace), workspace.numel(), _ptr(dev_err), _stream(stream)))


def _logit_dtype(logits) -> int:
    if logits.dtype == torch.bfloat16:
        return JF_DTYPE_BF16
    if logits.dtype == torch.float32:
        return JF_DTYPE_F32
    raise TypeError("logits must be bfloat16 or float32")


def jf_compact_accepted_kv(k_cache, v_cache, block_table, prefix_len, path, accept_len,
                           new_prefix_len, dev_err=None, stream=None) -> None:
    """Moves the accepted path's K/V next to the prefix, in place (see include/jf.h)."""
    num_pages, page, Hkv, D = k_cache.shape
    B, N = path.shape
    _need(k_cache, "k_cache", torch.bfloat16)
    _need(v_cache, "v_cache", torch.bfloat16, tuple(k_cache.shape))
    _need(block_table, "block_table", torch.int32)
    for name, t, shape in (("prefix_len", prefix_len, (B,)), ("accept_len", accept_len, (B,)),
                           ("new_prefix_len", new_prefix_len, (B,))):
        _need(t, name, torch.int32, shape)
    _need(path, "path", torch.int32, (B, N))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    _check("jf_compact_accepted_kv", _lib.jf_compact_accepted_kv(
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(prefix_len), _ptr(path),
        _ptr(accept_len), B, N, Hkv, D, page, block_table.shape[1], num_pages,
        _ptr(new_prefix_len), _ptr(dev_err), _stream(stream)))


def jf_build_draft_tree(draft_logits, K, N, cand_token, cand_logp, parent, draft, depth,
                        root_token=None, score=None, stream=None) -> None:
    """Best-first draft tree from per-depth draft logits (see include/jf.h)."""
    B, Dmax, V = draft_logits.shape
    if draft_logits.dtype == torch.bfloat16:
        dt = JF_DTYPE_BF16
    elif draft_logits.dtype == torch.float32:
        dt = JF_DTYPE_F32
    else:
        raise TypeError("draft_logits must be bfloat16 or float32")
    _need(draft_logits, "draft_logits", draft_logits.dtype)
    _need(cand_token, "cand_token", torch.int32, (B, Dmax, K))
    _need(cand_logp, "cand_logp", torch.float32, (B, Dmax, K))
    for name, t in (("parent", parent), ("draft", draft), ("depth", depth)):
        _need(t, name, torch.int32, (B, N))
    if score is not None:
        _need(score, "score", torch.float32, (B, N))
    if root_token is not None:
        _need(root_token, "root_token", torch.int32, (B,))
    _check("jf_build_draft_tree", _lib.jf_build_draft_tree(
        _ptr(draft_logits), dt, _ptr(root_token), B, Dmax, V, K, N, _ptr(cand_token),
        _ptr(cand_logp), _ptr(parent), _ptr(draft), _ptr(depth), _ptr(score), _stream(stream)))


def jf_build_draft_tree_ragged(draft_logits, K, N, budget, cand_token, cand_logp, parent, draft,
                               depth, root_token=None, score=None, dev_err=None,
                               stream=None) -> None:
    """Best-first draft trees with a budget per sequence (budget int32 [B], clamped to
    [1, N]); entries past a sequence's budget are padding (see include/jf.h)."""
    B, Dmax, V = draft_logits.shape
    dt = _logit_dtype(draft_logits)
    _need(draft_logits, "draft_logits", draft_logits.dtype)
    _need(budget, "budget", torch.int32, (B,))
    _need(cand_token, "cand_token", torch.int32, (B, Dmax, K))
    _need(cand_logp, "cand_logp", torch.float32, (B, Dmax, K))
    for name, t in (("parent", parent), ("draft", draft), ("depth", depth)):
        _need(t, name, torch.int32, (B, N))
    if score is not None:
        _need(score, "score", torch.float32, (B, N))
    if root_token is not None:
        _need(root_token, "root_token", torch.int32, (B,))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32, (1,))
    _check("jf_build_draft_tree_ragged", _lib.jf_build_draft_tree_ragged(
        _ptr(draft_logits), dt, _ptr(root_token), _ptr(budget), B, Dmax, V, K, N,
        _ptr(cand_token), _ptr(cand_logp), _ptr(parent), _ptr(draft), _ptr(depth), _ptr(score),
        _ptr(dev_err), _stream(stream)))


# ----------------------------------------------------------------------------- conveniences

def _workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    return torch.empty((nbytes + 15) // 16 * 16, dtype=torch.uint8, device=device)


def build_tree_mask(parent: torch.Tensor, prefix_len: torch.Tensor, dev_err=None, stream=None,
                    tree_len=None):
    B, N = parent.shape
    W = (N + 63) // 64
    mask = torch.empty((B, N, W), dtype=torch.int64, device=parent.device)
    depth = torch.empty((B, N), dtype=torch.int32, device=parent.device)
    pos = torch.empty((B, N), dtype=torch.int32, device=parent.device)
    if tree_len is None:
        jf_build_tree_mask(parent, prefix_len, mask, depth, pos, dev_err, stream)
    else:
        jf_build_tree_mask_ragged(parent, prefix_len, tree_len, mask, depth, pos, dev_err, stream)
    return mask, depth, pos


def tree_attention(q, k_cache, v_cache, block_table, prefix_len, mask, scale=None,
                   with_lse=False, dev_err=None, stream=None, tree_len=None):
    B, N, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    if scale is None:
        scale = D ** -0.5
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if with_lse else None
    ws = _workspace(jf_tree_attention_workspace_size(B, N, Hq, Hkv, D, block_table.shape[1],
                                                     k_cache.shape[1]), q.device)
    if tree_len is None:
        jf_tree_attention(q, k_cache, v_cache, block_table, prefix_len, mask, scale, out, lse, ws,
                          dev_err, stream)
    else:
        jf_tree_attention_ragged(q, k_cache, v_cache, block_table, prefix_len, tree_len, mask,
                                 scale, out, lse, ws, dev_err, stream)
    return (out, lse) if with_lse else out


def tree_verify(logits, draft, parent, dev_err=None, stream=None, tree_len=None):
    B, N, V = logits.shape
    dev = logits.device
    argmax = torch.empty((B, N), dtype=torch.int32, device=dev)
    accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    path = torch.empty((B, N), dtype=torch.int32, device=dev)
    bonus = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = _workspace(jf_tree_verify_workspace_size(B, N, V), dev)
    if tree_len is None:
        jf_tree_verify(logits, draft, parent, accept_len, path, bonus, argmax, ws, dev_err, stream)
    else:
        jf_tree_verify_ragged(logits, draft, parent, tree_len, accept_len, path, bonus, argmax, ws,
                              dev_err, stream)
    return argmax, accept_len, path, bonus


def tree_verify_sampled(logits, draft, parent, uniform, bonus_uniform, temperature=1.0,
                        dev_err=None, stream=None):
    """Allocating wrapper of jf_tree_verify_sampled: (accept_len, path, bonus)."""
    B, N, V = logits.shape
    dev = logits.device
    accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    path = torch.empty((B, N), dtype=torch.int32, device=dev)
    bonus = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = _workspace(jf_tree_verify_workspace_size(B, N, V), dev)
    jf_tree_verify_sampled(logits, draft, parent, uniform, bonus_uniform, temperature, accept_len,
                           path, bonus, ws, dev_err, stream)
    return accept_len, path, bonus


def tree_verify_shard_keys(logits_shard, vocab_offset, chunks=None, stream=None):
    """Allocating wrapper of jf_tree_verify_shard_keys: int64 keys [B][N][chunks].  Every
    range must use the same chunks (by default the planned count for this range's size:
    pass the largest range's count when the ranges differ in size)."""
    B, N, Vs = logits_shard.shape
    if chunks is None:
        chunks = jf_tree_verify_shard_chunks(B, N, Vs)
    keys = torch.empty((B, N, chunks), dtype=torch.int64, device=logits_shard.device)
    jf_tree_verify_shard_keys(logits_shard, vocab_offset, keys, stream)
    return keys


def tree_verify_from_keys(keys, V, draft, parent, dev_err=None, stream=None):
    """Allocating wrapper of jf_tree_verify_from_keys on gathered keys [S][B][N][chunks]:
    (argmax, accept_len, path, bonus) as tree_verify returns them."""
    S, B, N, _ = keys.shape
    dev = keys.device
    argmax = torch.empty((B, N), dtype=torch.int32, device=dev)
    accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    path = torch.empty((B, N), dtype=torch.int32, device=dev)
    bonus = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = torch.empty((8 * B * N,), dtype=torch.uint8, device=dev)
    jf_tree_verify_from_keys(keys, V, draft, parent, accept_len, path, bonus, ws, argmax,
                             dev_err, stream)
    return argmax, accept_len, path, bonus


def compact_accepted_kv(k_cache, v_cache, block_table, prefix_len, path, accept_len,
                        dev_err=None, stream=None):
    """In-place KV compaction after verification; returns the new prefix lengths."""
    new_prefix_len = torch.empty_like(prefix_len)
    jf_compact_accepted_kv(k_cache, v_cache, block_table, prefix_len, path, accept_len,
                           new_prefix_len, dev_err, stream)
    return new_prefix_len


def build_draft_tree(draft_logits, K, N, root_token=None, stream=None):
    """Returns (parent, draft, depth, score, cand_token, cand_logp)."""
    B, Dmax, V = draft_logits.shape
    dev = draft_logits.device
    cand_token = torch.empty((B, Dmax, K), dtype=torch.int32, device=dev)
    cand_logp = torch.empty((B, Dmax, K), dtype=torch.float32, device=dev)
    parent = torch.empty((B, N), dtype=torch.int32, device=dev)
    draft = torch.empty((B, N), dtype=torch.int32, device=dev)
    depth = torch.empty((B, N), dtype=torch.int32, device=dev)
    score = torch.empty((B, N), dtype=torch.float32, device=dev)
    jf_build_draft_tree(draft_logits, K, N, cand_token, cand_logp, parent, draft, depth,
                        root_token, score, stream)
    return parent, draft, depth, score, cand_token, cand_logp

