"""The C-ABI library loads, exports every function include/jf.h declares, and rejects bad
host arguments before touching the GPU.  CPU only (no kernel is launched)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from tree_speculative_decoding_jf_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(jf_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("jf_build_tree_mask", "jf_tree_attention", "jf_tree_verify",
              "jf_tree_attention_workspace_size", "jf_tree_verify_workspace_size",
              "jf_status_string", "jf_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"libjf.so does not export {n}"


def test_status_strings(lib):
    lib.jf_status_string.restype = ctypes.c_char_p
    assert lib.jf_status_string(0) == b"JF_OK"
    assert lib.jf_status_string(4) == b"JF_ERR_WORKSPACE_TOO_SMALL"
    assert lib.jf_status_string(99) == b"JF_ERR_UNKNOWN"


def test_host_argument_validation_needs_no_gpu(lib):
    P = ctypes.c_void_p
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails early
    lib.jf_build_tree_mask.argtypes = [P, P, ctypes.c_int32, ctypes.c_int32, P, P, P, P, P]
    assert lib.jf_build_tree_mask(None, fake, 1, 4, fake, None, None, None, None) == 1
    assert lib.jf_build_tree_mask(fake, fake, 0, 4, fake, None, None, None, None) == 1
    assert lib.jf_build_tree_mask(fake, fake, 1, 5000, fake, None, None, None, None) == 3
    assert lib.jf_build_tree_mask(fake, fake, 1, 4, ctypes.c_void_p(0x10004), None, None,
                                  None, None) == 7
    i32 = ctypes.c_int32
    lib.jf_tree_attention.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                      ctypes.c_float, P, P, P, ctypes.c_size_t, P, P]
    args = [fake] * 6 + [1, 16, 32, 8, 128, 16, 10, 10, 0.088, fake, None, None, 0, None, None]
    bad_d = list(args); bad_d[10] = 96
    assert lib.jf_tree_attention(*bad_d) == 3          # D not in {64, 128}
    bad_g = list(args); bad_g[9] = 5
    assert lib.jf_tree_attention(*bad_g) == 3          # Hq % Hkv != 0
    bad_page = list(args); bad_page[11] = 32
    assert lib.jf_tree_attention(*bad_page) == 3       # page size must be 16
    nul = list(args); nul[0] = None
    assert lib.jf_tree_attention(*nul) == 1
    mis = list(args); mis[0] = ctypes.c_void_p(0x10008)
    assert lib.jf_tree_attention(*mis) == 7
    lib.jf_tree_verify.argtypes = [P, i32, P, P, i32, i32, i32, P, P, P, P, P, ctypes.c_size_t,
                                   P, P]
    assert lib.jf_tree_verify(fake, 7, fake, fake, 1, 4, 10, None, fake, fake, fake, fake,
                              1 << 20, None, None) == 1      # bad dtype
    assert lib.jf_tree_verify(fake, 0, fake, fake, 1, 4, 10, None, fake, fake, fake, None,
                              1 << 20, None, None) == 1      # missing workspace


def test_ragged_calls_validate_host_arguments_without_gpu(lib):
    """The ragged entry points need tree_len and share the fixed-size checks."""
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails early
    lib.jf_build_tree_mask_ragged.argtypes = [P, P, P, i32, i32, P, P, P, P, P]
    assert lib.jf_build_tree_mask_ragged(fake, fake, None, 1, 4, fake, None, None, None, None) == 1
    assert lib.jf_build_tree_mask_ragged(fake, fake, fake, 1, 5000, fake, None, None, None,
                                         None) == 3
    lib.jf_tree_attention_ragged.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                             i32, i32, ctypes.c_float, P, P, P, ctypes.c_size_t,
                                             P, P]
    args = [fake] * 7 + [1, 16, 32, 8, 128, 16, 10, 10, 0.088, fake, None, None, 0, None, None]
    no_len = list(args); no_len[5] = None
    assert lib.jf_tree_attention_ragged(*no_len) == 1
    bad_d = list(args); bad_d[11] = 96
    assert lib.jf_tree_attention_ragged(*bad_d) == 3
    mis = list(args); mis[0] = ctypes.c_void_p(0x10008)
    assert lib.jf_tree_attention_ragged(*mis) == 7
    lib.jf_tree_verify_ragged.argtypes = [P, i32, P, P, P, i32, i32, i32, P, P, P, P, P,
                                          ctypes.c_size_t, P, P]
    assert lib.jf_tree_verify_ragged(fake, 0, fake, fake, None, 1, 4, 10, None, fake, fake, fake,
                                     fake, 1 << 20, None, None) == 1     # no tree_len
    assert lib.jf_tree_verify_ragged(fake, 7, fake, fake, fake, 1, 4, 10, None, fake, fake, fake,
                                     fake, 1 << 20, None, None) == 1     # bad dtype


def test_shard_verify_calls_validate_host_arguments_without_gpu(lib):
    """The vocabulary-sharded verify calls reject bad sizes, offsets and pointers before any
    launch."""
    P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails early
    lib.jf_tree_verify_shard_chunks.argtypes = [i32, i32, i32]
    lib.jf_tree_verify_shard_chunks.restype = i32
    assert lib.jf_tree_verify_shard_chunks(1, 0, 100) == -1
    assert lib.jf_tree_verify_shard_chunks(1, 5000, 100) == -1
    lib.jf_tree_verify_shard_keys.argtypes = [P, i32, i32, i32, i32, i32, i32, P, P]
    assert lib.jf_tree_verify_shard_keys(None, 0, 1, 4, 100, 0, 1, fake, None) == 1
    assert lib.jf_tree_verify_shard_keys(fake, 7, 1, 4, 100, 0, 1, fake, None) == 1
    assert lib.jf_tree_verify_shard_keys(fake, 0, 1, 4, 100, -1, 1, fake, None) == 1
    assert lib.jf_tree_verify_shard_keys(fake, 0, 1, 4, 100, 0, 0, fake, None) == 1
    assert lib.jf_tree_verify_shard_keys(fake, 0, 1, 5000, 100, 0, 1, fake, None) == 3
    assert lib.jf_tree_verify_shard_keys(fake, 0, 1, 4, 100, 0x7FFFFFF0, 1, fake, None) == 3
    assert lib.jf_tree_verify_shard_keys(fake, 0, 1, 4, 100, 0, 1,
                                         ctypes.c_void_p(0x10004), None) == 7
    lib.jf_tree_verify_from_keys.argtypes = [P, i32, i32, P, P, i32, i32, i32, P, P, P, P, P, sz,
                                             P, P]
    args = [fake, 2, 3, fake, fake, 2, 4, 100, None, fake, fake, fake, fake, 64, None, None]
    no_ws = list(args); no_ws[12] = None
    assert lib.jf_tree_verify_from_keys(*no_ws) == 1
    no_s = list(args); no_s[1] = 0
    assert lib.jf_tree_verify_from_keys(*no_s) == 1
    small = list(args); small[13] = 63            # 8 * B * N = 64 bytes needed
    assert lib.jf_tree_verify_from_keys(*small) == 4
    mis = list(args); mis[12] = ctypes.c_void_p(0x10004)
    assert lib.jf_tree_verify_from_keys(*mis) == 7


def test_packed_calls_validate_host_arguments_without_gpu(lib):
    """The packed (cu_seqlens) entry points need cu_seqlens and a positive T."""
    P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails early
    lib.jf_build_tree_mask_packed.argtypes = [P, P, P, i32, i32, i32, P, P, P, P, P]
    assert lib.jf_build_tree_mask_packed(fake, fake, None, 2, 16, 20, fake, None, None, None,
                                         None) == 1
    assert lib.jf_build_tree_mask_packed(fake, fake, fake, 2, 16, 0, fake, None, None, None,
                                         None) == 1
    assert lib.jf_build_tree_mask_packed(fake, fake, fake, 2, 5000, 20, fake, None, None, None,
                                         None) == 3
    lib.jf_tree_attention_packed.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                             i32, i32, i32, ctypes.c_float, P, P, P, sz, P, P]
    args = [fake] * 7 + [2, 16, 20, 32, 8, 128, 16, 10, 10, 0.088, fake, None, None, 0, None,
                         None]
    no_cu = list(args); no_cu[5] = None
    assert lib.jf_tree_attention_packed(*no_cu) == 1
    no_t = list(args); no_t[9] = 0
    assert lib.jf_tree_attention_packed(*no_t) == 1
    huge_t = list(args); huge_t[9] = 0x7FFFFFF8
    assert lib.jf_tree_attention_packed(*huge_t) == 3
    lib.jf_tree_verify_packed_workspace_size.argtypes = [i32, i32]
    lib.jf_tree_verify_packed_workspace_size.restype = sz
    assert lib.jf_tree_verify_packed_workspace_size(0, 100) == ctypes.c_size_t(-1).value
    lib.jf_tree_verify_packed.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, P, P, P, P, P, sz,
                                          P, P]
    assert lib.jf_tree_verify_packed(fake, 0, fake, fake, None, 2, 16, 20, 100, None, fake, fake,
                                     fake, fake, 1 << 20, None, None) == 1     # no cu_seqlens
    assert lib.jf_tree_verify_packed(fake, 0, fake, fake, fake, 2, 16, 0, 100, None, fake, fake,
                                     fake, fake, 1 << 20, None, None) == 1     # T = 0


def test_sampled_ragged_and_packed_calls_validate_host_arguments_without_gpu(lib):
    P, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails early
    lib.jf_tree_verify_sampled_ragged.argtypes = [P, i32, P, P, P, P, P, f32, i32, i32, i32, P, P,
                                                  P, P, sz, P, P]
    assert lib.jf_tree_verify_sampled_ragged(fake, 0, fake, fake, None, fake, fake, 1.0, 2, 8, 100,
                                             fake, fake, fake, fake, 1 << 20, None, None) == 1
    lib.jf_tree_verify_sampled_packed.argtypes = [P, i32, P, P, P, P, P, f32, i32, i32, i32, i32,
                                                  P, P, P, P, sz, P, P]
    assert lib.jf_tree_verify_sampled_packed(fake, 0, fake, fake, None, fake, fake, 1.0, 2, 8, 10,
                                             100, fake, fake, fake, fake, 1 << 20, None, None) == 1
    assert lib.jf_tree_verify_sampled_packed(fake, 0, fake, fake, fake, fake, fake, 1.0, 2, 8, 0,
                                             100, fake, fake, fake, fake, 1 << 20, None, None) == 1
    assert lib.jf_tree_verify_sampled_packed(fake, 0, fake, fake, fake, fake, fake, 0.0, 2, 8, 10,
                                             100, fake, fake, fake, fake, 1 << 20, None, None) == 1


def test_ragged_draft_tree_needs_budgets(lib):
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: the call fails early
    lib.jf_build_draft_tree_ragged.argtypes = [P, i32, P, P, i32, i32, i32, i32, i32, P, P, P, P,
                                               P, P, P, P]
    assert lib.jf_build_draft_tree_ragged(fake, 0, None, None, 2, 4, 100, 4, 16, fake, fake, fake,
                                          fake, fake, None, None, None) == 1
    assert lib.jf_build_draft_tree_ragged(fake, 0, None, fake, 2, 2, 100, 2, 16, fake, fake, fake,
                                          fake, fake, None, None, None) == 3   # lattice 7 < 16
