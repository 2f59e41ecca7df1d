"""The bounded waits of the tree-attention kernels, exercised on the GPU.

Every wait of a CTA on its own pipeline (a K/V copy landing, a tensor-core step, a softmax
pass) gives up after a time limit, records JF_DEVERR_TIMEOUT and lets the kernel return;
the waits that drain the CTA's own copies and tensor-core work before it exits keep the
one-second limit.  A test hook lowers the pipeline limit to 50 us and makes the warps that
report "this key tile's data has landed" withhold that signal, so the tensor-core issuer
waits for a barrier phase that nothing completes.  The call must still return (the stream
completes), report the timeout bit, and leave the GPU usable: the next call in normal
operation must be correct, which also shows that every CTA released its tensor memory (a
later allocation on the same SM would otherwise never be granted)."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_decoding_jf_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module")
def jf():
    from tree_speculative_decoding_jf_gb300 import build
    build.build()
    from tree_speculative_decoding_jf_gb300 import jf as mod
    return mod


def run(jf, w, t, mask):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = jf.tree_attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                 t["prefix_len"], mask, scale=w.scale, with_lse=True, dev_err=err)
    torch.cuda.synchronize()
    return out, lse, int(err.item())


def test_attention_wait_limit_runs_out_then_recovers(jf):
    w = wl.config("c1_tiny_random16")
    t = wl.device_tensors(w, with_logits=False)
    mask, _, _ = jf.build_tree_mask(t["parent"], t["prefix_len"])
    torch.cuda.synchronize()
    jf.jf_debug_set_wait_limit_ns(50_000, withhold_arrivals=True)
    try:
        _, _, err = run(jf, w, t, mask)
    finally:
        jf.jf_debug_set_wait_limit_ns(0, withhold_arrivals=False)
    assert err & jf.DEVERR_TIMEOUT, f"device error bits {err:#x}"
    out, lse, err = run(jf, w, t, mask)
    assert err == 0
    ref_o, _ = oracle.tree_attention(w)
    got = out.float().cpu().numpy()
    assert (np.abs(got - ref_o) <= ATOL + RTOL * np.abs(ref_o)).all()
