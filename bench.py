#!/usr/bin/env python3
"""Benchmark of the tree-speculative-decoding hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch of synthetic inputs already in
HBM: tree-mask build -> tree-causal paged attention -> greedy tree verify (argmax + walk).
The reported metric is the tree-causal paged attention call's time (µs per call) with its
HBM GB/s and TFLOP/s against the roofline.  Default workload: Qwen3-30B-A3B attention
shape, 8 sequences with 32768-token prefixes, budget-256 best-first trees, vocabulary
151936 (``--config`` picks another of the five).

Timing: each of the three calls is captured once into its own CUDA graph, and the whole
step once more into one graph.  W untimed warm-up steps, then K timed steps; a step
writes 256 MiB (twice the L2) so it starts from a cold L2, then replays the mask,
attention and verify graphs with CUDA events between them on the stream the kernels run
on.  ``value`` is the mean attention time over the K steps; the other calls go to
``breakdown_us``.  ``ms_per_step`` is the one-graph step, replayed K more times after an
L2 eviction each (``step_three_graphs`` is the step as the sum of the three graphs with
events between them).  The same run then
times the attention call alone for at least a second (so the clock sampler sees
sustained load), the attention calls of the budget-16 and budget-256 Qwen3-8B workloads,
the lossless (sampled) verification, the draft-tree build, the ragged attention call and
the KV compaction.  ``e2e`` times the
attention call through the plain API with pinned host buffers: the copies of its inputs
in and of its outputs back are inside the timed region.  Under torchrun every rank runs
its own replica (the path shards by sequence with no exchange), and the slowest rank's
time is reported.

``--impl reference`` times the fp64 CPU oracle's attention instead (on a bounded sample
of the query rows of the same workload, scaled to a full call).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tree_speculative_decoding_jf_gb300 import workloads as wl  # noqa: E402

METRIC = "tree-causal paged attention µs/call, HBM GB/s & TFLOP/s vs GB300 roofline"
DEFAULT_CONFIG = "c5_qwen3_30b_b8_tree256_32k"
# Other workloads whose attention call is timed in the same run (budgets 16 and 256).
SIDE_CONFIGS = ("c2_qwen3_8b_chain16", "c3_qwen3_8b_tree256")
SUSTAINED_S = 1.0                      # length of the attention-only loop
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one jf_tree_attention call
# (attention kernel + combine) from ncu captures of the current kernels (None until a
# capture of the current kernel exists for that workload); the capture commands are in
# the profile summaries.
NCU_TRAFFIC_BYTES = {
    "c5_qwen3_30b_b8_tree256_32k": 569551872 + 29477376 + 38097920 + 0,
    "c3_qwen3_8b_tree256": 20050944 + 0 + 16927488 + 0,
    "c4_qwen3_8b_b32_tree64_paged": 569012992 + 6938880,
    "c2_qwen3_8b_chain16": 8674304 + 0 + 2405120 + 0,
}


# ----------------------------------------------------------------------------- work model

def attention_algorithmic_bytes(w, tree_len=None) -> int:
    """K/V of every visible position read once per kv-head, Q read, O written, masks and
    block-table entries read (ragged trees: the first tree_len[b] nodes of sequence b)."""
    n = np.full(w.B, w.N, np.int64) if tree_len is None else np.asarray(tree_len, np.int64)
    kv_len = w.prefix_len.astype(np.int64) + n
    kv = int(kv_len.sum()) * w.Hkv * w.D * 2 * 2
    qo = 2 * int(n.sum()) * w.Hq * w.D * 2
    mask = int(n.sum()) * ((w.N + 63) // 64) * 8
    bt = int(((kv_len + w.page - 1) // w.page).sum()) * 4
    return kv + qo + mask + bt


def attention_algorithmic_flops(w, tree_len=None) -> int:
    """4 * D * Hq * sum_b (n_b * P_b + sum_{i < n_b} (depth_i + 1)): visible (query, key)
    pairs, n_b = N or tree_len[b]."""
    tot = 0
    for b in range(w.B):
        nb = w.N if tree_len is None else int(tree_len[b])
        par = w.parent[b]
        depth = np.zeros(nb, dtype=np.int64)
        for i in range(1, nb):
            depth[i] = depth[par[i]] + 1
        tot += nb * int(w.prefix_len[b]) + int((depth + 1).sum())
    return 4 * w.D * w.Hq * tot


def verify_algorithmic_bytes(w) -> int:
    esz = 4 if w.logits_dtype == "f32" else 2
    return w.B * w.N * w.V * esz + w.B * w.N * 4 * 4


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_attention_time(w, budget_s: float = 20.0):
    """Time the fp64 oracle's tree attention on a bounded sample of query rows and scale
    by row count to one full call.  Returns (seconds per call, sample description,
    threads used)."""
    import oracle
    rows_total = w.B * w.N * w.Hq
    rb, rh, ri = oracle.all_rows(w)
    rng = np.random.default_rng(0)
    order = rng.permutation(rows_total)
    n_probe = min(rows_total, 64)
    t0 = time.perf_counter()
    oracle.tree_attention_rows(w, rb[order[:n_probe]], rh[order[:n_probe]], ri[order[:n_probe]])
    per_row = max((time.perf_counter() - t0) / n_probe, 1e-7)
    n_att = int(min(rows_total, max(n_probe, budget_s / per_row)))
    sel = order[:n_att]
    t0 = time.perf_counter()
    oracle.tree_attention_rows(w, rb[sel], rh[sel], ri[sel])
    t_att = (time.perf_counter() - t0) * rows_total / n_att
    sample = (f"attention over {n_att} of {rows_total} query rows (random sample), scaled by "
              f"row count to one full call")
    threads = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    return t_att, sample, threads


# ----------------------------------------------------------------------------- GPU arm

def roofline(w, us, peaks, tree_len=None):
    """Bound (HBM or tensor, whichever ideal time is longer), achieved rate and fraction of
    the measured peak for an attention call of `us` microseconds."""
    abytes = attention_algorithmic_bytes(w, tree_len)
    aflops = attention_algorithmic_flops(w, tree_len)
    if abytes / (peaks["hbm_gbs"] * 1e9) >= aflops / (peaks["bf16_tflops"] * 1e12):
        r = {"bound": "hbm", "achieved": abytes / (us * 1e-6) / 1e9, "peak": peaks["hbm_gbs"],
             "unit": "GB/s"}
    else:
        r = {"bound": "tensor", "achieved": aflops / (us * 1e-6) / 1e12,
             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["algorithmic_bytes"] = abytes
    r["algorithmic_flops"] = aflops
    r["hbm_gbs_achieved"] = abytes / (us * 1e-6) / 1e9
    r["tflops_achieved"] = aflops / (us * 1e-6) / 1e12
    return r


def run_gpu(args, w, rank, world, peaks):
    import torch
    from tree_speculative_decoding_jf_gb300 import jf

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    t = wl.device_tensors(w, device=dev)
    B, N, Hq, Hkv, D, V = w.B, w.N, w.Hq, w.Hkv, w.D, w.V
    W = (N + 63) // 64
    mask = torch.empty((B, N, W), dtype=torch.int64, device=dev)
    depth = torch.empty((B, N), dtype=torch.int32, device=dev)
    pos = torch.empty((B, N), dtype=torch.int32, device=dev)
    out = torch.empty_like(t["q"])
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    ws_a_bytes = jf.jf_tree_attention_workspace_size(B, N, Hq, Hkv, D, w.max_pages, w.page)
    ws_a = torch.empty(max(16, ws_a_bytes), dtype=torch.uint8, device=dev)
    ws_v = torch.empty(jf.jf_tree_verify_workspace_size(B, N, V), dtype=torch.uint8, device=dev)
    argmax = torch.empty((B, N), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    path = torch.empty((B, N), dtype=torch.int32, device=dev)
    bonus = torch.empty((B,), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    attn_launches = 2 if ws_a_bytes > 0 else 1          # attention kernel (+ combine)
    launches_per_step = 1 + attn_launches + 2           # mask, attention, argmax + walk

    # Each hot-path call is captured once into its own CUDA graph, so host-side argument
    # marshalling stays out of the device timeline.
    def call_mask():
        jf.jf_build_tree_mask(t["parent"], t["prefix_len"], mask, depth, pos, err)

    def call_attn():
        jf.jf_tree_attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                             t["prefix_len"], mask, w.scale, out, lse, ws_a, err)

    def call_verify():
        jf.jf_tree_verify(t["logits"], t["draft"], t["parent"], acc, path, bonus, argmax, ws_v,
                          err)

    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(2):
            call_mask(); call_attn(); call_verify()
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)

    def capture(*fns):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for fn in fns:
                fn()
        return g

    g_mask, g_attn, g_ver = capture(call_mask), capture(call_attn), capture(call_verify)
    g_step = capture(call_mask, call_attn, call_verify)     # the whole step as one graph

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def step(k):
        """One step after an L2 eviction: mask, attention and verify graphs with events
        between them."""
        e = [ev() for _ in range(4)]
        flush.fill_(k & 0xFF)
        e[0].record(stream)
        g_mask.replay()
        e[1].record(stream)
        g_attn.replay()
        e[2].record(stream)
        g_ver.replay()
        e[3].record(stream)
        return e

    def timed(g, k):
        a, b_ = ev(), ev()
        flush.fill_(k & 0xFF)                     # evict L2 before every timed replay
        a.record(stream)
        g.replay()
        b_.record(stream)
        return a, b_

    def ms(pairs):
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b_) for a, b_ in pairs]

    for k in range(args.warmup):
        step(k)
        timed(g_step, k)
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)                              # let the sampler start before the loop
    step_ev = [step(k) for k in range(args.steps)]
    step1_ev = [timed(g_step, k) for k in range(args.steps)]
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    step_ms = [a.elapsed_time(b_) for a, b_ in step1_ev]
    step_ev_ms = [e[0].elapsed_time(e[3]) for e in step_ev]
    mask_ms = [e[0].elapsed_time(e[1]) for e in step_ev]
    attn_ms = [e[1].elapsed_time(e[2]) for e in step_ev]
    ver_ms = [e[2].elapsed_time(e[3]) for e in step_ev]
    # Sustained: the attention call alone for at least SUSTAINED_S seconds, still inside
    # the clock sampler's window.
    reps = args.steps if args.step_only else max(
        args.steps, int(SUSTAINED_S / max(statistics.mean(attn_ms) * 1e-3, 1e-6)) + 1)
    sus_ms = ms([timed(g_attn, k) for k in range(reps)])
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if err.item() != 0:
        raise RuntimeError(f"device error bits {err.item():#x} during the benchmark")

    if args.step_only:
        return dict(step_ms=step_ms, step_ev_ms=step_ev_ms, mask_ms=mask_ms, attn_ms=attn_ms, ver_ms=ver_ms, sus_ms=sus_ms,
                    clocks=clk, e2e=None, launches=2 * launches_per_step * args.steps, ws=ws_a_bytes)
    # ---- the attention calls of the budget-16 and budget-256 Qwen3-8B workloads
    side_lines = {}
    for name in SIDE_CONFIGS:
        if name == w.name or world > 1:
            continue
        sw = wl.config(name, with_logits=False)
        st = wl.device_tensors(sw, device=dev, with_logits=False)
        smask = torch.empty((sw.B, sw.N, (sw.N + 63) // 64), dtype=torch.int64, device=dev)
        jf.jf_build_tree_mask(st["parent"], st["prefix_len"], smask, None, None, err)
        sout = torch.empty_like(st["q"])
        slse = torch.empty((sw.B, sw.Hq, sw.N), dtype=torch.float32, device=dev)
        nws = jf.jf_tree_attention_workspace_size(sw.B, sw.N, sw.Hq, sw.Hkv, sw.D, sw.max_pages, sw.page)
        sws = torch.empty(max(16, nws), dtype=torch.uint8, device=dev)

        def call_side(st=st, smask=smask, sout=sout, slse=slse, sws=sws, sw=sw):
            jf.jf_tree_attention(st["q"], st["k_cache"], st["v_cache"], st["block_table"],
                                 st["prefix_len"], smask, sw.scale, sout, slse, sws, err)

        call_side()
        g_side = capture(call_side)
        for k in range(args.warmup):
            timed(g_side, k)
        side_ms = ms([timed(g_side, k) for k in range(max(args.steps, 50))])
        us = statistics.mean(side_ms) * 1e3
        rf = roofline(sw, us, peaks)
        side_lines[name] = {"attention_us": us, "bound": rf["bound"], "achieved": rf["achieved"],
                            "unit": rf["unit"], "frac": rf["frac"],
                            "traffic": NCU_TRAFFIC_BYTES.get(name)}
        del st, smask, sout, slse, sws, g_side
        torch.cuda.synchronize(dev)

    # ---- end to end through the C ABI with host buffers (pinned), copies timed: the
    # attention call with its inputs copied in (and its mask built) and its outputs
    # copied back.
    e2e = None
    if not args.no_e2e:
        keys = ("q", "k_cache", "v_cache", "block_table", "prefix_len", "parent")
        host = {k: t[k].cpu().pin_memory() for k in keys}
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        dt = {k: torch.empty_like(t[k]) for k in keys}
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = sum(x.numel() * x.element_size() for x in (h_out, h_lse))

        def e2e_call():
            for k in keys:
                dt[k].copy_(host[k], non_blocking=True)
            jf.jf_build_tree_mask(dt["parent"], dt["prefix_len"], mask, None, None, err)
            jf.jf_tree_attention(dt["q"], dt["k_cache"], dt["v_cache"], dt["block_table"],
                                 dt["prefix_len"], mask, w.scale, out, lse, ws_a, err)
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_call()
        torch.cuda.synchronize(dev)
        e2e_ms = []
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            a, b_ = ev(), ev()
            a.record(stream)
            e2e_call()
            b_.record(stream)
            b_.synchronize()
            e2e_ms.append(a.elapsed_time(b_))
        e2e = {"value": max_over_ranks(statistics.mean(e2e_ms) * 1e3, world), "unit": "µs/call",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}
        del host, dt
    # ---- lossless (stochastic) verification of the same trees (seeded random numbers,
    # temperature 1); not part of the step, which verifies greedily.
    su, sbu = wl.sampling_uniforms(B, N, w.seed)
    t_su, t_sbu = torch.from_numpy(su).to(dev), torch.from_numpy(sbu).to(dev)
    s_acc = torch.empty_like(acc)
    s_path = torch.empty_like(path)
    s_bonus = torch.empty_like(bonus)

    def call_sampled():
        jf.jf_tree_verify_sampled(t["logits"], t["draft"], t["parent"], t_su, t_sbu, 1.0, s_acc,
                                  s_path, s_bonus, ws_v, err)

    call_sampled()
    g_samp = capture(call_sampled)
    for k in range(args.warmup):
        timed(g_samp, k)
    samp_ms = ms([timed(g_samp, k) for k in range(args.steps)])

    # ---- vocabulary-sharded verification as one of 8 GPUs would run it (the target's
    # output layer split into 8 token ranges): this GPU's range keys, then the merge and
    # walk on all 8 ranges' keys.  The other ranges' keys are made once beforehand; the
    # all-gather between the two calls is not timed.  Not part of the step.
    S_v = 8
    cuts_v = [V * s // S_v for s in range(S_v + 1)]
    ch_v = max(jf.jf_tree_verify_shard_chunks(B, N, cuts_v[s + 1] - cuts_v[s]) for s in range(S_v))
    range0 = t["logits"][:, :, cuts_v[0]:cuts_v[1]].contiguous()
    keys_v = torch.stack([jf.tree_verify_shard_keys(
        t["logits"][:, :, cuts_v[s]:cuts_v[s + 1]].contiguous(), cuts_v[s], ch_v)
        for s in range(S_v)])
    v_am = torch.empty_like(argmax)
    v_acc, v_path, v_bonus = torch.empty_like(acc), torch.empty_like(path), torch.empty_like(bonus)
    ws_k = torch.empty((8 * B * N,), dtype=torch.uint8, device=dev)

    def call_sharded():
        jf.jf_tree_verify_shard_keys(range0, 0, keys_v[0])
        jf.jf_tree_verify_from_keys(keys_v, V, t["draft"], t["parent"], v_acc, v_path, v_bonus,
                                    ws_k, v_am, err)

    call_sharded()
    g_shard = capture(call_sharded)
    for k in range(args.warmup):
        timed(g_shard, k)
    shard_ms = ms([timed(g_shard, k) for k in range(args.steps)])
    torch.cuda.synchronize(dev)
    shard_same = bool((v_am == argmax).all() and (v_acc == acc).all() and (v_path == path).all()
                      and (v_bonus == bonus).all())
    del range0, keys_v

    # ---- before verification: best-first draft-tree construction from per-depth draft
    # logits (16 depths, 8 candidates per depth, the workload's budget); not part of the step.
    dl = wl.draft_logits(B, 16, V, seed=w.seed)
    t_dl = torch.from_numpy(dl.view(np.int16)).view(torch.bfloat16).to(dev)
    K_tree = 8
    tree_out = dict(cand_token=torch.empty((B, 16, K_tree), dtype=torch.int32, device=dev),
                    cand_logp=torch.empty((B, 16, K_tree), dtype=torch.float32, device=dev),
                    parent=torch.empty((B, N), dtype=torch.int32, device=dev),
                    draft=torch.empty((B, N), dtype=torch.int32, device=dev),
                    depth=torch.empty((B, N), dtype=torch.int32, device=dev))

    def call_tree():
        jf.jf_build_draft_tree(t_dl, K_tree, N, tree_out["cand_token"], tree_out["cand_logp"],
                               tree_out["parent"], tree_out["draft"], tree_out["depth"])

    call_tree()
    g_tree = capture(call_tree)
    for k in range(args.warmup):
        timed(g_tree, k)
    tree_ms = ms([timed(g_tree, k) for k in range(args.steps)])
    torch.cuda.synchronize(dev)
    tree_bytes = int(t_dl.numel()) * 2

    # ---- ragged trees: the same attention call with a per-sequence budget mix (seeded,
    # uniform in [N/4, N]); its mask is built once beforehand.  Not part of the step.
    rag_len = np.random.default_rng(w.seed + 1000).integers(max(1, N // 4), N + 1, B)
    t_rag = torch.from_numpy(rag_len.astype(np.int32)).to(dev)
    mask_r = torch.empty_like(mask)
    jf.jf_build_tree_mask_ragged(t["parent"], t["prefix_len"], t_rag, mask_r, None, None, err)

    def call_attn_ragged():
        jf.jf_tree_attention_ragged(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                    t["prefix_len"], t_rag, mask_r, w.scale, out, lse, ws_a, err)

    call_attn_ragged()
    g_rag = capture(call_attn_ragged)
    for k in range(args.warmup):
        timed(g_rag, k)
    rag_ms = ms([timed(g_rag, k) for k in range(args.steps)])

    # ---- the same ragged trees in the packed (cu_seqlens) layout: q, out and the mask
    # hold only real nodes; the call must match the ragged one row for row.
    cu_np = np.concatenate([[0], np.cumsum(rag_len)]).astype(np.int32)
    T_p = int(cu_np[-1])
    t_cu = torch.from_numpy(cu_np).to(dev)
    q_p = torch.cat([t["q"][b, :int(n)] for b, n in enumerate(rag_len)]).contiguous()
    par_p = torch.cat([t["parent"][b, :int(n)] for b, n in enumerate(rag_len)]).contiguous()
    mask_p = torch.empty((T_p, mask.shape[-1]), dtype=torch.int64, device=dev)
    jf.jf_build_tree_mask_packed(par_p, t["prefix_len"], t_cu, N, mask_p, None, None, err)
    out_p = torch.empty((T_p, Hq, D), dtype=torch.bfloat16, device=dev)
    lse_p = torch.empty((Hq, T_p), dtype=torch.float32, device=dev)

    def call_attn_packed():
        jf.jf_tree_attention_packed(q_p, t["k_cache"], t["v_cache"], t["block_table"],
                                    t["prefix_len"], t_cu, N, mask_p, w.scale, out_p, lse_p,
                                    ws_a, err)

    call_attn_packed()
    g_pk = capture(call_attn_packed)
    for k in range(args.warmup):
        timed(g_pk, k)
    pk_ms = ms([timed(g_pk, k) for k in range(args.steps)])
    torch.cuda.synchronize(dev)
    pk_same = all(torch.equal(out_p[int(cu_np[b]):int(cu_np[b + 1])].view(torch.int16),
                              out[b, :int(n)].view(torch.int16))
                  for b, n in enumerate(rag_len))
    del q_p, out_p, lse_p, mask_p
    torch.cuda.synchronize(dev)

    # ---- after verification: accepted-path KV compaction (not part of the step).  It
    # rewrites the cache in place, so it is timed last; replays repeat the same copies.
    new_prefix = torch.empty_like(t["prefix_len"])

    def call_compact():
        jf.jf_compact_accepted_kv(t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"],
                                  path, acc, new_prefix, err)

    g_compact = capture(call_compact)
    for k in range(args.warmup):
        timed(g_compact, k)
    compact_ms = ms([timed(g_compact, k) for k in range(args.steps)])

    # ---- the device side of one serving iteration as one graph: draft tree from the draft
    # logits, its mask, the attention call (its mask is the drafted tree's), greedy verify
    # of the drafted tokens and the KV compaction.  Replays repeat the same copies.
    def call_serving():
        call_tree()
        jf.jf_build_tree_mask(tree_out["parent"], t["prefix_len"], mask, depth, pos, err)
        call_attn()
        jf.jf_tree_verify(t["logits"], tree_out["draft"], tree_out["parent"], acc, path, bonus,
                          argmax, ws_v, err)
        call_compact()

    call_serving()
    g_serving = capture(call_serving)
    for k in range(args.warmup):
        timed(g_serving, k)
    serving_ms = ms([timed(g_serving, k) for k in range(args.steps)])
    torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    if err.item() != 0:
        raise RuntimeError(f"device error bits {err.item():#x} after the benchmark's calls")
    return dict(step_ms=step_ms, step_ev_ms=step_ev_ms, mask_ms=mask_ms, attn_ms=attn_ms, ver_ms=ver_ms, sus_ms=sus_ms,
                clocks=clk, e2e=e2e, launches=2 * launches_per_step * args.steps, ws=ws_a_bytes,
                compact_ms=compact_ms, accepted=acc.cpu().tolist(), tree_ms=tree_ms, samp_ms=samp_ms,
                serving_ms=serving_ms,
                samp_accepted=s_acc.cpu().tolist(), shard_ms=shard_ms, shard_same=shard_same,
                tree_bytes=tree_bytes, rag_ms=rag_ms, rag_len=rag_len.tolist(), side=side_lines,
                pk_ms=pk_ms, pk_same=pk_same)


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_dict(w, l2="flushed"):
    return {"workload": w.name, "batch": w.B, "tree_nodes": w.N, "q_heads": w.Hq,
            "kv_heads": w.Hkv, "head_dim": w.D, "vocab": w.V,
            "prefix_len": int(w.prefix_len[0]) if len(set(w.prefix_len.tolist())) == 1
            else [int(w.prefix_len.min()), int(w.prefix_len.max())],
            "page_size": w.page, "l2_between_steps": l2}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=wl.CONFIG_NAMES)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--step-only", action="store_true",
                    help="time only the step (no sustained loop, other workloads, e2e or CPU "
                         "baseline): short runs for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group(backend)

    peaks, peak_src = load_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        w = wl.config(args.config, with_logits=False)
        per_call = []
        sample = threads = None
        for _ in range(args.steps):
            s, sample, threads = oracle_attention_time(
                w, budget_s=max(0.2, args.cpu_budget / args.steps))
            per_call.append(s)
        v = statistics.mean(per_call) * 1e6
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": "µs/call",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": v / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, l2="n/a (CPU)"),
            "cpu_baseline": {"value": v, "unit": "µs/call", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "µs/call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return

    w = wl.config(args.config)
    r = run_gpu(args, w, rank, world, peaks)
    attn_us = max_over_ranks(statistics.mean(r["attn_ms"]) * 1e3, world)
    step_us = max_over_ranks(statistics.mean(r["step_ms"]) * 1e3, world)
    roof = roofline(w, attn_us, peaks)
    roof["traffic"] = NCU_TRAFFIC_BYTES.get(w.name)
    roof["kernel"] = "jf_tree_attention (attention kernel + combine)"
    roof["peak_source"] = "measured (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["attention_us"] = attn_us
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and not args.step_only and world == 1:
        s, sample, threads = oracle_attention_time(w, budget_s=args.cpu_budget)
        cpu = {"value": s * 1e6, "unit": "µs/call", "cores": threads, "kind": "oracle",
               "sample": sample}
    sus_us = statistics.mean(r["sus_ms"]) * 1e3
    if args.step_only:
        print(json.dumps({"metric": METRIC, "value": attn_us, "unit": "µs/call", "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_us / 1e3,
                          "higher_is_better": False, "config": config_dict(w), "roofline": roof,
                          "breakdown_us": {"step": step_us, "mask": statistics.mean(r["mask_ms"]) * 1e3,
                                           "verify": statistics.mean(r["ver_ms"]) * 1e3,
                                           "attention_sustained": sus_us},
                          "clocks": r["clocks"], "note": "step-only run (profiling)"}), flush=True)
        return
    line = {
        "metric": METRIC, "value": attn_us, "unit": "µs/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_us / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(w),
        "breakdown_us": {"step": step_us, "step_min": min(r["step_ms"]) * 1e3,
                         "step_three_graphs": statistics.mean(r["step_ev_ms"]) * 1e3,
                         "mask": statistics.mean(r["mask_ms"]) * 1e3, "attention": attn_us,
                         "attention_min": min(r["attn_ms"]) * 1e3,
                         "attention_median": statistics.median(r["attn_ms"]) * 1e3,
                         "attention_sustained": sus_us,
                         "attention_sustained_calls": len(r["sus_ms"]),
                         "attention_sustained_frac": roofline(w, sus_us, peaks)["frac"],
                         "verify": statistics.mean(r["ver_ms"]) * 1e3,
                         "verify_hbm_gbs": verify_algorithmic_bytes(w) /
                         (statistics.mean(r["ver_ms"]) * 1e-3) / 1e9,
                         "verify_sampled": statistics.mean(r["samp_ms"]) * 1e3,
                         "verify_sampled_hbm_gbs": verify_algorithmic_bytes(w) /
                         (statistics.mean(r["samp_ms"]) * 1e-3) / 1e9,
                         "verify_sampled_accepted_nodes": r["samp_accepted"],
                         "verify_vocab_shard8": statistics.mean(r["shard_ms"]) * 1e3,
                         "verify_vocab_shard8_equals_verify": r["shard_same"],
                         "other_workloads_attention": r["side"],
                         "draft_tree_build": statistics.mean(r["tree_ms"]) * 1e3,
                         "draft_tree_logits_hbm_gbs": r["tree_bytes"] /
                         (statistics.mean(r["tree_ms"]) * 1e-3) / 1e9,
                         "kv_compaction_after_verify": statistics.mean(r["compact_ms"]) * 1e3,
                         "serving_iteration": statistics.mean(r["serving_ms"]) * 1e3,
                         "kv_compaction_accepted_nodes": r["accepted"],
                         "attention_ragged": statistics.mean(r["rag_ms"]) * 1e3,
                         "attention_ragged_tree_len": r["rag_len"],
                         "attention_packed": statistics.mean(r["pk_ms"]) * 1e3,
                         "attention_packed_equals_ragged": r["pk_same"],
                         "attention_ragged_hbm_gbs": attention_algorithmic_bytes(w, r["rag_len"]) /
                         (statistics.mean(r["rag_ms"]) * 1e-3) / 1e9,
                         "attention_ragged_tflops": attention_algorithmic_flops(w, r["rag_len"]) /
                         (statistics.mean(r["rag_ms"]) * 1e-3) / 1e12},
        "roofline": roof, "cpu_baseline": cpu, "e2e": r["e2e"], "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
