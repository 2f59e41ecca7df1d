"""jf_tree_verify_static -- the allocation-free verify entry point for callers that cannot
allocate device memory on their call path -- must give the same argmax, accepted length,
path and bonus as jf_tree_verify and as the fp64 oracle (integer outputs: bit-exact), on
two calls in a row with different inputs (the shared scratch keeps the previous call's
contents, which must not leak).  The call goes straight through the C ABI with raw
device pointers."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _outputs(B, N):
    z = lambda *s: torch.full(s, -7, dtype=torch.int32, device="cuda")   # noqa: E731
    return z(B, N), z(B), z(B, N), z(B), torch.zeros(1, dtype=torch.int32, device="cuda")


def _inputs(seed, B, N, V, dtype):
    w = wl.make_workload("noalloc", B, N, 4, 1, 64, V, 32, tree="random_depth_limited",
                         logits_dtype=dtype, forcing="half", seed=seed)
    t = wl.device_tensors(w)
    return t["logits"], t["draft"], t["parent"], w


def test_static_verify_matches_workspace_verify_twice():
    from tree_speculative_decoding_jf_gb300 import build
    build.build()
    from tree_speculative_decoding_jf_gb300 import jf
    lib = jf._lib
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed, (B, N, V, dtype) in enumerate([(3, 40, 151936, "bf16"), (2, 17, 5003, "f32")]):
        logits, draft, parent, w = _inputs(seed, B, N, V, dtype)
        dt = jf.JF_DTYPE_BF16 if dtype == "bf16" else jf.JF_DTYPE_F32
        # existing entry point, with its own workspace
        ref = _outputs(B, N)
        ws = torch.empty(jf.jf_tree_verify_workspace_size(B, N, V), dtype=torch.uint8, device="cuda")
        rc = lib.jf_tree_verify(_ptr(logits), dt, _ptr(draft), _ptr(parent), B, N, V,
                                _ptr(ref[0]), _ptr(ref[1]), _ptr(ref[2]), _ptr(ref[3]), _ptr(ws),
                                ws.numel(), _ptr(ref[4]), stream)
        assert rc == 0
        # allocation-free entry point
        got = _outputs(B, N)
        rc = lib.jf_tree_verify_static(_ptr(logits), dt, _ptr(draft), _ptr(parent), B, N, V,
                                       _ptr(got[0]), _ptr(got[1]), _ptr(got[2]), _ptr(got[3]),
                                       _ptr(got[4]), stream)
        assert rc == 0
        torch.cuda.synchronize()
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
        assert got[4].item() == 0 and got[1].min().item() >= 0
        ram, racc, rpath, rbonus = oracle.tree_verify(w)
        assert (got[0].cpu().numpy() == ram).all() and (got[1].cpu().numpy() == racc).all()
        assert (got[2].cpu().numpy() == rpath).all() and (got[3].cpu().numpy() == rbonus).all()


def test_static_verify_rejects_sizes_beyond_its_scratch():
    from tree_speculative_decoding_jf_gb300 import jf
    lib = jf._lib
    fake = ctypes.c_void_p(0x10000)     # never dereferenced: the call fails before launching
    B, N, V = 256, 4096, 151936         # 1M rows > 2^19 scratch entries
    rc = lib.jf_tree_verify_static(fake, jf.JF_DTYPE_BF16, fake, fake, B, N, V, None, fake,
                                   fake, fake, None, None)
    assert rc == 8 and jf.jf_status_string(rc) == "JF_ERR_SCRATCH_CAPACITY"
