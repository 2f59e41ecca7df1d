#!/usr/bin/env python3
"""Benchmark of the tree-speculative-decoding hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch of synthetic inputs already in
HBM: tree-mask build -> tree-causal paged attention -> greedy tree verify (argmax + walk).
Default workload: Qwen3-8B attention shape, one sequence, 2048-token prefix, 16-node
linear draft tree, vocabulary 151936 (``--config`` picks another of the five).

Timing: the step (three calls) is captured once into a CUDA graph; W untimed warm-up
steps, then K timed replays between CUDA events on the stream the kernels run on, each
after a 256 MiB write (twice the L2) so every step starts from a cold L2.  Each call is
also captured alone and timed the same way (K replays each) for the per-call breakdown;
the attention call's time is the one used for the roofline.  The e2e figure uses the plain API calls (no graphs) with pinned
host buffers and the copies inside the timed region.  Under torchrun every rank runs its
own replica (the path shards by sequence with no exchange), and the slowest rank's time is
reported.

``--impl reference`` times the fp64 CPU oracle instead (on a bounded sample of the same
workload, scaled to a full step).
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
DEFAULT_CONFIG = "c2_qwen3_8b_chain16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes per attention call from the ncu captures summarised under profiles/ (None
# until a capture of the current kernel exists for that workload).
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one jf_tree_attention call
# (attention kernel + combine) from `ncu --set full` captures of the current kernels; see
# profiles/tree_attention_<workload>_full.md for the commands.
NCU_TRAFFIC_BYTES = {
    "c2_qwen3_8b_chain16": 8659968 + 0 + 2404352 + 0,
    "c5_qwen3_30b_b8_tree256_32k": 568709888 + 27651584 + 38085120 + 4352,
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

def oracle_step_time(w, budget_s: float = 20.0):
    """Time the fp64 oracle on a bounded sample of one step and scale to a full step.
    Returns (seconds per full step, description of the sample, threads used)."""
    import oracle
    rows_total = w.B * w.N * w.Hq
    # attention: time a small probe, then size the sample to the budget
    rb, rh, ri = oracle.all_rows(w)
    rng = np.random.default_rng(0)
    order = rng.permutation(rows_total)
    n_probe = min(rows_total, 64)
    t0 = time.perf_counter()
    oracle.tree_attention_rows(w, rb[order[:n_probe]], rh[order[:n_probe]], ri[order[:n_probe]])
    per_row = max((time.perf_counter() - t0) / n_probe, 1e-7)
    n_att = int(min(rows_total, max(n_probe, budget_s * 0.7 / per_row)))
    sel = order[:n_att]
    t0 = time.perf_counter()
    oracle.tree_attention_rows(w, rb[sel], rh[sel], ri[sel])
    t_att = (time.perf_counter() - t0) * rows_total / n_att
    # mask: whole step (cheap)
    t0 = time.perf_counter()
    oracle.tree_mask(w.parent, w.prefix_len)
    t_mask = time.perf_counter() - t0
    # verify: argmax over a sample of rows, the walk over every sequence
    lrows = w.logits.reshape(w.B * w.N, w.V)
    n_lr = min(w.B * w.N, max(1, int(2e9 / max(1, w.V * 20))))
    t0 = time.perf_counter()
    am_part = oracle.argmax(lrows[:n_lr], w.logits_dtype)
    t_arg = (time.perf_counter() - t0) * (w.B * w.N) / n_lr
    am = np.zeros((w.B, w.N), np.int32)
    am.reshape(-1)[:n_lr] = am_part
    t0 = time.perf_counter()
    oracle.tree_walk(am, w.draft, w.parent)
    t_walk = time.perf_counter() - t0
    total = t_att + t_mask + t_arg + t_walk
    sample = (f"attention {n_att}/{rows_total} query rows, argmax {n_lr}/{w.B * w.N} logits rows, "
              f"mask and walk in full; scaled by row count to one full step")
    threads = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    return total, sample, threads


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args, w, rank, world):
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
    launches_per_step = 1 + (2 if ws_a_bytes > 0 else 1) + 2

    def step(tt, ev=None):
        if ev is not None:
            ev[0].record(stream)
        jf.jf_build_tree_mask(tt["parent"], tt["prefix_len"], mask, depth, pos, err, stream)
        if ev is not None:
            ev[1].record(stream)
        jf.jf_tree_attention(tt["q"], tt["k_cache"], tt["v_cache"], tt["block_table"],
                             tt["prefix_len"], mask, w.scale, out, lse, ws_a, err, stream)
        if ev is not None:
            ev[2].record(stream)
        jf.jf_tree_verify(tt["logits"], tt["draft"], tt["parent"], acc, path, bonus, argmax, ws_v,
                          err, stream)
        if ev is not None:
            ev[3].record(stream)

    # Each hot-path call is captured once into its own CUDA graph; a timed step replays the
    # three graphs between CUDA events, so host-side argument marshalling stays out of
    # the device timeline.
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

    g_step = capture(call_mask, call_attn, call_verify)     # the whole hot path
    g_parts = [capture(call_mask), capture(call_attn), capture(call_verify)]

    def timed(g, k):
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.fill_(k & 0xFF)                     # evict L2 before every timed replay
        a.record(stream)
        g.replay()
        b_.record(stream)
        return a, b_

    for k in range(args.warmup):
        timed(g_step, k)
        for g in g_parts:
            timed(g, k)
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)                              # let the sampler start before the loop
    step_ev = [timed(g_step, k) for k in range(args.steps)]
    part_ev = [[timed(g, k) for g in g_parts] for k in range(args.steps)]
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    step_ms = [a.elapsed_time(b_) for a, b_ in step_ev]
    mask_ms = [e[0][0].elapsed_time(e[0][1]) for e in part_ev]
    attn_ms = [e[1][0].elapsed_time(e[1][1]) for e in part_ev]
    ver_ms = [e[2][0].elapsed_time(e[2][1]) for e in part_ev]
    if err.item() != 0:
        raise RuntimeError(f"device error bits {err.item():#x} during the benchmark")

    # ---- end to end through the C ABI with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e:
        host = {k: v.cpu().pin_memory() for k, v in t.items()}
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_acc = torch.empty(acc.shape, dtype=acc.dtype).pin_memory()
        h_path = torch.empty(path.shape, dtype=path.dtype).pin_memory()
        h_bonus = torch.empty(bonus.shape, dtype=bonus.dtype).pin_memory()
        dt = {k: torch.empty_like(v) for k, v in t.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = sum(x.numel() * x.element_size() for x in (h_out, h_acc, h_path, h_bonus))

        def e2e_step():
            for k in host:
                dt[k].copy_(host[k], non_blocking=True)
            step(dt)
            h_out.copy_(out, non_blocking=True)
            h_acc.copy_(acc, non_blocking=True)
            h_path.copy_(path, non_blocking=True)
            h_bonus.copy_(bonus, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        e2e_ms = []
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_step()
            b_.record(stream)
            b_.synchronize()
            e2e_ms.append(a.elapsed_time(b_))
        e2e = {"value": statistics.mean(e2e_ms) * 1e3, "unit": "µs/call",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}
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
    tree_ev = [timed(g_tree, k) for k in range(args.steps)]
    torch.cuda.synchronize(dev)
    tree_ms = [a.elapsed_time(b_) for a, b_ in tree_ev]
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
    rag_ev = [timed(g_rag, k) for k in range(args.steps)]
    torch.cuda.synchronize(dev)
    rag_ms = [a.elapsed_time(b_) for a, b_ in rag_ev]

    # ---- after verification: accepted-path KV compaction (not part of the step).  It
    # rewrites the cache in place, so it is timed last; replays repeat the same copies.
    new_prefix = torch.empty_like(t["prefix_len"])

    def call_compact():
        jf.jf_compact_accepted_kv(t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"],
                                  path, acc, new_prefix, err)

    g_compact = capture(call_compact)
    for k in range(args.warmup):
        timed(g_compact, k)
    cmp_ev = [timed(g_compact, k) for k in range(args.steps)]
    torch.cuda.synchronize(dev)
    compact_ms = [a.elapsed_time(b_) for a, b_ in cmp_ev]
    if err.item() != 0:
        raise RuntimeError(f"device error bits {err.item():#x} in the KV compaction")
    return dict(step_ms=step_ms, mask_ms=mask_ms, attn_ms=attn_ms, ver_ms=ver_ms, clocks=clk,
                e2e=e2e, launches=2 * launches_per_step * args.steps, ws=ws_a_bytes,
                compact_ms=compact_ms, accepted=acc.cpu().tolist(), tree_ms=tree_ms,
                tree_bytes=tree_bytes, rag_ms=rag_ms, rag_len=rag_len.tolist())


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

    w = wl.config(args.config)
    peaks, peak_src = load_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        per_step = []
        sample = threads = None
        for _ in range(args.warmup):
            pass                                     # the oracle has no warm-up state
        for _ in range(args.steps):
            s, sample, threads = oracle_step_time(w, budget_s=max(1.0, args.cpu_budget / args.steps))
            per_step.append(s)
        v = statistics.mean(per_step) * 1e6
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

    r = run_gpu(args, w, rank, world)
    step_us = statistics.mean(r["step_ms"]) * 1e3
    step_us = max_over_ranks(step_us, world)
    attn_us = statistics.mean(r["attn_ms"]) * 1e3
    abytes = attention_algorithmic_bytes(w)
    aflops = attention_algorithmic_flops(w)
    t_hbm = abytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = aflops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": abytes / (attn_us * 1e-6) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": aflops / (attn_us * 1e-6) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = NCU_TRAFFIC_BYTES.get(w.name)
    roof["kernel"] = "jf_tree_attention (attention kernel + combine)"
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["algorithmic_bytes"] = abytes
    roof["algorithmic_flops"] = aflops
    roof["attention_us"] = attn_us
    roof["hbm_gbs_achieved"] = abytes / (attn_us * 1e-6) / 1e9
    roof["tflops_achieved"] = aflops / (attn_us * 1e-6) / 1e12
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        s, sample, threads = oracle_step_time(w, budget_s=args.cpu_budget)
        cpu = {"value": s * 1e6, "unit": "µs/call", "cores": threads, "kind": "oracle",
               "sample": sample}
    line = {
        "metric": METRIC, "value": step_us, "unit": "µs/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_us / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(w),
        "breakdown_us": {"mask": statistics.mean(r["mask_ms"]) * 1e3, "attention": attn_us,
                         "attention_min": min(r["attn_ms"]) * 1e3,
                         "attention_median": statistics.median(r["attn_ms"]) * 1e3,
                         "step_min": min(r["step_ms"]) * 1e3,
                         "verify": statistics.mean(r["ver_ms"]) * 1e3,
                         "verify_hbm_gbs": verify_algorithmic_bytes(w) /
                         (statistics.mean(r["ver_ms"]) * 1e-3) / 1e9,
                         "draft_tree_build": statistics.mean(r["tree_ms"]) * 1e3,
                         "draft_tree_logits_hbm_gbs": r["tree_bytes"] /
                         (statistics.mean(r["tree_ms"]) * 1e-3) / 1e9,
                         "kv_compaction_after_verify": statistics.mean(r["compact_ms"]) * 1e3,
                         "kv_compaction_accepted_nodes": r["accepted"],
                         "attention_ragged": statistics.mean(r["rag_ms"]) * 1e3,
                         "attention_ragged_tree_len": r["rag_len"],
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
