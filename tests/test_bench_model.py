"""CPU checks of bench.py's algorithmic work model (the numerators of the roofline
fractions): a ragged call with every tree at full size counts exactly the fixed-size
work, smaller trees count strictly less, and the flop count matches a direct count of
visible (query row, key) pairs on a tiny workload."""
import importlib.util
import os

import numpy as np

from conftest import ROOT
from tree_speculative_decoding_jf_gb300 import workloads as wl


def _bench():
    spec = importlib.util.spec_from_file_location("bench_model", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_ragged_work_at_full_size_equals_fixed_size_work():
    b = _bench()
    w = wl.make_workload("m", 3, 20, 8, 2, 64, 64, np.array([5, 40, 130], np.int32),
                         tree="random_depth_limited", seed=3, with_logits=False)
    full = [w.N] * w.B
    assert b.attention_algorithmic_bytes(w, full) == b.attention_algorithmic_bytes(w)
    assert b.attention_algorithmic_flops(w, full) == b.attention_algorithmic_flops(w)
    small = [1, 7, 20]
    assert b.attention_algorithmic_bytes(w, small) < b.attention_algorithmic_bytes(w)
    assert b.attention_algorithmic_flops(w, small) < b.attention_algorithmic_flops(w)


def test_flops_count_visible_pairs():
    b = _bench()
    w = wl.make_workload("m", 2, 6, 4, 1, 8, 64, np.array([3, 0], np.int32),
                         tree="random_depth_limited", seed=4, with_logits=False)
    pairs = 0
    for s in range(w.B):
        for i in range(w.N):
            anc, x = 0, i
            while x >= 0:
                anc += 1
                x = w.parent[s, x]
            pairs += int(w.prefix_len[s]) + anc
    assert b.attention_algorithmic_flops(w) == 4 * w.D * w.Hq * pairs
