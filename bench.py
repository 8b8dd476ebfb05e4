"""Benchmark of the EAGLE draft-and-verify cycle on GB300.

One step = one full cycle (drafting with EAGLE-2 tree growth, rerank, tree-attention
verify, acceptance, KV compaction, drafter update) over one batch. Default workload: the
Llama-3.1-8B-shaped EAGLE-3 configuration with temperature-1 speculative sampling (batch 1,
1024-token prompt, k=10, depth 8, m=60), whose 8B batch-1 verify pass is the figure the
roofline reports; random-init bf16 weights and synthetic prompt ids. `--workload` selects
the other configurations. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica (no collective on the
data path); rank 0 prints value = tokens committed by all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from eagle_speculative_decoding_cycle_gb300 import synth  # noqa: E402

METRIC = "draft+verify cycle µs, tree tok/s & HBM GB/s; committed tok/s (τ) at bs=1"
UNIT = "tok/s"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s)"


def algorithmic_bytes(w: synth.Workload, ctx: float, batch: int = 1) -> dict:
    """Bytes one cycle over `batch` sequences of mean context `ctx` must move (bf16 weights
    and KV), split by phase: verify = all target layer weights + LM head, read once for the
    batch, + each sequence's ctx KV read and tree KV write; drafter = (depth - 1) expansions
    + 1 update, each FC + one layer + LM head (+ each sequence's drafter KV)."""
    m, t = w.model, w.tree
    H, F, V, d = m.hidden, m.ffn, m.vocab, m.head_dim
    qkv = m.qkv_out
    layer = (qkv * H + H * m.n_heads * d + 3 * H * F) * 2
    lm = V * H * 2
    kv_tok = 2 * m.n_layers * m.n_kv_heads * d * 2
    verify = int(m.n_layers * layer + lm + batch * (ctx + t.m + 1) * kv_tok)
    fc_in = 2 * H if w.drafter.kind == 1 else 3 * H
    dlayer = ((qkv * (H if w.drafter.kind == 1 else 2 * H)) + H * m.n_heads * d + 3 * H * F) * 2
    dstep = int(H * fc_in * 2 + dlayer + lm + batch * ctx * 2 * m.n_kv_heads * d * 2)
    drafter = t.depth * dstep
    return {"verify": verify, "drafter": drafter, "cycle": verify + drafter,
            "verify_weights": m.n_layers * layer + lm}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu), "--query-gpu=" + self.FIELDS,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


def dist_setup(backend: str = ""):
    """Rank, world size and local GPU from the torchrun environment; for N > 1 a process
    group for the timing reductions: NCCL on GPUs, gloo where no GPU is present."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier_max(ws: int, value: float, device) -> float:
    if ws == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier_sum(ws: int, value: float, device) -> float:
    if ws == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(ws: int) -> None:
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------------------------
# CPU oracle sample (the baseline; also the --impl reference arm)
# ---------------------------------------------------------------------------------------------
CPU_PROMPT = 32


def oracle_sample(wl: synth.Workload, weights_gpu, steps: int, warmup: int, budget_s: float):
    """Time the oracle as it stands on the workload's model and tree shapes at full depth, on
    the host cores: prefill of the first CPU_PROMPT prompt tokens (untimed), `warmup` untimed
    cycles, then up to `steps` timed cycles, stopping once `budget_s` seconds of cycles have
    run (at least one timed cycle). Weights reach the oracle as float32 arrays (an exact
    upcast of the bf16 values). Planting is off: a truncated prompt has no reference
    continuation, so the oracle commits what its random-init drafter and the acceptance rule
    give. Every reported figure is the time of cycles actually run."""
    from oracle.cycle import OracleSeq, build_model
    W = {k: v.to("cpu", torch.float32).numpy() for k, v in weights_gpu.items()}
    wlc = wl.replace(new_tokens=64)
    M = build_model(W, wlc)
    prompt = synth.make_prompts(wl)[0].numpy()[:CPU_PROMPT]
    n_ref = (steps + warmup + 2) * (wl.tree.depth + 1) + 8
    t0 = time.perf_counter()
    o = OracleSeq(M, wlc, capacity=len(prompt) + n_ref + 4 * (wl.tree.m + wl.tree.depth) + 16)
    o.prefill(prompt)
    setup_s = time.perf_counter() - t0
    for _ in range(warmup):
        o.cycle()
    times, committed = [], 0
    t_start = time.perf_counter()
    for _ in range(steps):
        c0 = len(o.committed)
        t0 = time.perf_counter()
        o.cycle()
        times.append(time.perf_counter() - t0)
        committed += len(o.committed) - c0
        if time.perf_counter() - t_start > budget_s:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    done = len(times)
    t_total = sum(times)
    return {"value": committed / t_total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "cycles": done, "s_per_cycle": t_total / done, "tau": committed / done, "setup_s": setup_s,
            "sample": (f"{done} timed oracle cycle(s) of {wl.name} at full depth ({wl.model.n_layers} layers, "
                       f"k{wl.tree.topk} D{wl.tree.depth} m{wl.tree.m}, T={wl.tree.temperature}) after a "
                       f"{len(prompt)}-token prompt prefill and {warmup} untimed cycle(s), planting off; numpy fp64 on "
                       f"{cores} host cores")}


def static_tree(kind: str, tree: synth.TreeShape) -> synth.TreeShape:
    """A static (EAGLE-1 style) tree for the workload's k and D, decided before any context
    is seen. "static-chain": one rank-0 child per depth (m = D). "static-prior": the m nodes
    with the largest prior acceptance, the prior of a node being the product over its path
    of a fixed per-rank weight (0.6, 0.15, 0.08, 0.05, 0.03, then 0.02), subject to at most
    k expanded nodes per depth (nodes are taken best-first, each after its parent)."""
    k, D, m = tree.topk, tree.depth, tree.m
    if kind == "static-chain":
        return dataclasses.replace(tree, m=D, static_parent=tuple(range(-1, D - 1)), static_rank=(0,) * D)
    w = [0.6, 0.15, 0.08, 0.05, 0.03] + [0.02] * max(0, k - 5)
    parent, rank, score, depth = [], [], [], []
    expanded = {d: set() for d in range(1, D + 1)}
    frontier = [(w[r], -1, r, 1) for r in range(k)]
    while len(parent) < m and frontier:
        frontier.sort(key=lambda x: -x[0])
        sc, p, r, d = frontier.pop(0)
        if p >= 0 and p not in expanded[d - 1] and len(expanded[d - 1]) >= k:
            continue
        if p >= 0:
            expanded[d - 1].add(p)
        parent.append(p)
        rank.append(r)
        i = len(parent) - 1
        if d < D:
            frontier += [(sc * w[c], i, c, d + 1) for c in range(k)]
    return dataclasses.replace(tree, m=len(parent), static_parent=tuple(parent), static_rank=tuple(rank))


# ---------------------------------------------------------------------------------------------
def run_ours(args, ws, rank, local):
    from eagle_speculative_decoding_cycle_gb300 import _lib as L
    from eagle_speculative_decoding_cycle_gb300 import api
    from eagle_speculative_decoding_cycle_gb300.build import build
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    # rank 0 compiles (if the sources changed); the other ranks then find its library
    if rank == 0:
        build()
    barrier(ws)
    if rank != 0:
        build()
    wl = synth.WORKLOADS[args.workload]
    if args.planted_p is not None:
        wl = wl.replace(tree=dataclasses.replace(wl.tree, planted_p=args.planted_p))
    if args.tree != "dynamic":
        wl = wl.replace(tree=static_tree(args.tree, wl.tree))
    t = wl.tree
    D = t.depth
    weights = synth.make_weights(wl, device=str(dev))
    torch.cuda.synchronize()
    prompts = synth.make_prompts(wl)
    B = len(prompts)
    K, W = args.steps, args.warmup
    n_ref = (W + K + args.prof_steps + 8) * (D + 1) + D + 2
    n_plain = 64
    max_ctx = max(len(p) for p in prompts) + 2 * n_ref + (W + K + args.prof_steps + 8) * (D + 1) + 64
    stream = torch.cuda.Stream(device=dev)
    eng = api.Engine(wl, weights, max_batch=B, max_ctx=max_ctx, stream=stream)
    prompts_d = [p.to(dev) for p in prompts]
    out_d = torch.zeros(B, D + 1, dtype=torch.int32, device=dev)
    cnt_d = torch.zeros(B, dtype=torch.int32, device=dev)

    with torch.cuda.stream(stream):
        # plain decoding (one token per sequence per step): the speedup baseline
        eng.prefill(prompts_d)
        plain = torch.zeros(B, n_plain, dtype=torch.int32, device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        eng.decode_plain(n_plain, plain)
        e1.record(stream)
        eng.sync()
        plain_ms_per_step = e0.elapsed_time(e1) / n_plain
        # the planted reference: each sequence's continuation by the GPU's own plain decoding,
        # which the verify pass reproduces bit for bit (greedy), so a planted run stays on it
        eng.prefill(prompts_d)
        first = eng.dump(L.DUMP_STATE)["root_tok"][:B].to(torch.int32)
        rest = torch.zeros(B, n_ref - 1, dtype=torch.int32, device=dev)
        eng.decode_plain(n_ref - 1, rest)
        eng.sync()
        ref = torch.cat([first.view(B, 1).to(dev), rest], 1).tolist()
    R = torch.tensor(ref, dtype=torch.int32, device=dev)
    ref_buf = R.clone()
    # speculative cycles, graph replay
    clocks = ClockSampler(local)
    with torch.cuda.stream(stream):
        eng.set_graph(True)
        eng.prefill(prompts_d, ref_buf)
        for _ in range(W):
            eng.cycle()
        eng.sync()
        st0 = eng.dump(L.DUMP_STATE)
        c0 = st0["committed"][:B].long()
        ctx0 = float(st0["ctx_len"][:B].double().mean())
        barrier(ws)
        torch.cuda.synchronize(dev)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(K):
            eng.cycle()
        s1.record(stream)
        eng.sync()
        torch.cuda.synchronize(dev)
        barrier(ws)
        st = eng.dump(L.DUMP_STATE)
        committed = int((st["committed"][:B].long() - c0).sum())
        ctx1 = float(st["ctx_len"][:B].double().mean())
        on_track = int(st["on_track"][:B].min())
    ms_local = s0.elapsed_time(s1)
    # per-launch GEMM timing inside real cycles (eager launches, events around each GEMM)
    with torch.cuda.stream(stream):
        eng.set_graph(False)
        eng.prefill(prompts_d, ref_buf)
        for _ in range(2):
            eng.cycle()
        eng.sync()
        eng.profile_begin(400 * max(1, args.prof_steps))
        for _ in range(args.prof_steps):
            eng.cycle()
        n_launch, gemm_ms, gemm_bytes = eng.profile_end()
        eng.sync()
        # verify-pass time in cycles that carry only the two events around it (per-launch
        # events would break the programmatic dependent launches between kernels)
        eng.profile_begin(0)
        for _ in range(max(3, args.prof_steps)):
            eng.cycle()
        eng.profile_end()
        n_verify, verify_ms = eng.profile_verify()
        eng.sync()
    clk = clocks.stop()
    # end to end through the public API with host buffers: prompt + reference H2D from pinned
    # memory, prefill, then K cycles each followed by a D2H read of the committed tokens
    lens = [len(p) for p in prompts]
    prompt_h = torch.cat(prompts).pin_memory()
    prompt_all = torch.empty(prompt_h.shape, dtype=torch.int32, device=dev)
    ref_h = R.cpu().pin_memory()
    out_h = torch.zeros(B, D + 1, dtype=torch.int32).pin_memory()
    cnt_h = torch.zeros(B, dtype=torch.int32).pin_memory()
    with torch.cuda.stream(stream):
        eng.set_graph(True)
        eng.prefill(prompts_d, ref_buf)        # capture the graph with these output buffers
        eng.cycle(out_d, cnt_d)
        eng.sync()
        torch.cuda.synchronize(dev)
        barrier(ws)
        t0 = time.perf_counter()
        prompt_all.copy_(prompt_h, non_blocking=True)
        ref_buf.copy_(ref_h, non_blocking=True)
        eng.prefill(list(torch.split(prompt_all, lens)), ref_buf)
        e2e_tok = B
        for _ in range(K):
            eng.cycle(out_d, cnt_d)
            out_h.copy_(out_d, non_blocking=True)
            cnt_h.copy_(cnt_d, non_blocking=True)
            stream.synchronize()
            e2e_tok += int(cnt_h.sum())
        e2e_s = time.perf_counter() - t0
        eng.sync()
    e2e_s = barrier_max(ws, e2e_s, dev)
    e2e_tok_all = barrier_sum(ws, e2e_tok, dev)
    graph_launches = eng.lib.eagle_cycle_kernel_launches(eng.h)
    ms = barrier_max(ws, ms_local, dev)
    committed_all = barrier_sum(ws, committed, dev)
    hbm_peak, peak_src = peaks()
    byt = algorithmic_bytes(wl, (ctx0 + ctx1) / 2, B)
    cycle_s = ms / 1e3 / K
    gemm_gbs = gemm_bytes / (gemm_ms / 1e3) / 1e9 if gemm_ms > 0 else None
    verify_us = verify_ms * 1e3 / max(n_verify, 1) if verify_ms > 0 else None
    verify_gbs = byt["verify"] / (verify_us / 1e6) / 1e9 if verify_us else None
    res = None
    if rank == 0:
        res = {
            "metric": METRIC, "value": committed_all / (ms / 1e3), "unit": UNIT, "n_gpus": ws, "steps": K,
            "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init N(0,0.02) weights, uniform prompt ids)",
            "config": {"workload": wl.name, "batch": B,
                       "prompt": lens[0] if B == 1 else f"{min(lens)}-{max(lens)} tokens, {sum(lens)} in all",
                       "tree": f"k{t.topk} D{t.depth} m{t.m}" + ("" if args.tree == "dynamic" else f" {args.tree}"),
                       "planted_p": t.planted_p,
                       "temperature": t.temperature, "parallelism": "replicas" if ws > 1 else "single GPU",
                       "l2": "inputs larger than L2 (13+ GB of weights streamed per cycle); no flush needed",
                       "graph_replay": True},
            "cycle_us": cycle_s * 1e6,
            "tau": committed / K / B,
            "tree_tok_s": ws * B * (t.m + 1) / cycle_s,
            "hbm_gbs": byt["cycle"] / cycle_s / 1e9,
            "algorithmic_bytes_per_cycle": byt,
            "plain_decode": {"ms_per_step": plain_ms_per_step, "tok_s": B * 1e3 / plain_ms_per_step},
            "speedup_vs_plain": (committed / K) / cycle_s / (B * 1e3 / plain_ms_per_step),
            "on_track": on_track,
            "reference": "planted reference = the GPU's own plain decoding of each sequence; on_track = 1 if the "
                         "timed cycles never left it (under sampling the committed tokens leave it at the first "
                         "non-greedy draw and planting goes inert)",
            # the benchmark spec's figure: the target's verify pass against the HBM roofline; the GEMM
            # that streams its weights is the kernel that explains it
            "roofline": {"bound": "hbm",
                         "what": "verify pass: all target layers over the B(m+1) tree rows and the fused LM-head "
                                 "epilogue (weights, LM head, context KV read, tree KV write), CUDA events around "
                                 "it inside profiled eager cycles",
                         "achieved": verify_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": (verify_gbs / hbm_peak) if verify_gbs else None,
                         # the pass's DRAM bytes, scaled from the captured verify-pass GEMM
                         # launches (DRAM per algorithmic byte); its weights are ~99% of its bytes
                         "traffic": (traffic_ratio() * byt["verify"]) if traffic_ratio() else None,
                         "traffic_source": "profiles/gemm_bf16_tc_verify_llama3.1-8b-2layers.md: DRAM bytes "
                                           "per algorithmic byte of three verify-pass GEMM launches x this "
                                           "pass's algorithmic bytes",
                         "peak_source": peak_src,
                         "algorithmic_bytes": byt["verify"], "us": verify_us,
                         "kernel": {"name": "gemm_bf16_tc (tcgen05 weight-streaming GEMM, every projection and "
                                            "LM-head launch of a cycle)",
                                    "achieved": gemm_gbs, "peak": hbm_peak, "unit": "GB/s",
                                    "frac": (gemm_gbs / hbm_peak) if gemm_gbs else None,
                                    # the captured launches' DRAM bytes per algorithmic byte,
                                    # scaled to this run's average launch
                                    "traffic": (traffic_ratio() * gemm_bytes / max(n_launch, 1))
                                    if traffic_ratio() else None,
                                    "timing": f"CUDA events around each of {n_launch} GEMM launches over "
                                              f"{args.prof_steps} cycles (eager launches on the engine stream)",
                                    "bytes_per_launch_avg": gemm_bytes / max(n_launch, 1),
                                    "us_per_launch_avg": gemm_ms * 1e3 / max(n_launch, 1)}},
            "verify_pass": {
                "passes": n_verify, "us": verify_us, "algorithmic_bytes": byt["verify"], "gbs": verify_gbs,
                "frac_of_hbm_peak": (verify_gbs / hbm_peak) if verify_gbs else None,
                # projections + LM head only (2 flops per weight per row); attention excluded
                "weight_tflops": (byt["verify_weights"] * B * (t.m + 1) / (verify_us / 1e6) / 1e12)
                if verify_us else None},
            "clocks": clk,
            "e2e": {"value": e2e_tok_all / e2e_s, "unit": UNIT,
                    "h2d_bytes_per_step": (prompt_h.numel() * 4 + R.numel() * 4) / K,
                    "d2h_bytes_per_step": B * ((D + 1) * 4 + 4),
                    "what": "public API with host buffers: pinned H2D of prompt + reference, prefill, then K "
                            "cycles each with a D2H read of its committed tokens and a host sync"},
            "gpu_launches": graph_launches * K if graph_launches else None,
        }
    return res, wl, weights


def traffic_ratio():
    """DRAM bytes per algorithmic byte of the GEMM launches in the committed ncu summary (a
    small case of the same kernel), if the GEMM kernel's sources are unchanged since the
    counters were taken (else None)."""
    p = os.path.join(ROOT, "profiles", "gemm_bf16_tc_verify_llama3.1-8b-2layers.md")
    try:
        vals = {}
        with open(p) as f:
            for line in f:
                if line.startswith("- ") and ": " in line:
                    k, v = line[2:].strip().split(": ", 1)
                    vals[k] = v.strip("` ")
        from eagle_speculative_decoding_cycle_gb300.build import gemm_digest
        if vals.get("gemm source digest") != gemm_digest():
            return None
        return float(vals["dram bytes per algorithmic byte"])
    except Exception:
        return None


def run_ncu_region(args):
    """Short run for an ncu launch list: set up the workload, then run `--steps` eager
    cycles and two plain-decode steps inside the NVTX range "profiled"."""
    from eagle_speculative_decoding_cycle_gb300 import _lib as L
    from eagle_speculative_decoding_cycle_gb300 import api
    from eagle_speculative_decoding_cycle_gb300.build import build
    build()
    dev = torch.device("cuda:0")
    wl = synth.WORKLOADS[args.workload]
    if args.layers:   # a shallower model of the same width: the small case for multi-pass captures
        wl = wl.replace(model=dataclasses.replace(wl.model, n_layers=args.layers),
                        drafter=dataclasses.replace(wl.drafter, fuse_layers=tuple(
                            min(f, args.layers - 1) for f in wl.drafter.fuse_layers)))
    D = wl.tree.depth
    weights = synth.make_weights(wl, device=str(dev))
    prompts = [p.to(dev) for p in synth.make_prompts(wl)]
    B = len(prompts)
    n_plain = (args.steps + 4) * (D + 1) + D + 2
    eng = api.Engine(wl, weights, max_batch=B,
                     max_ctx=max(len(p) for p in prompts) + n_plain + (args.steps + 8) * (D + 1) + 64)
    eng.prefill(prompts)
    first = eng.dump(L.DUMP_STATE)["root_tok"][:B].to(dev).to(torch.int32)
    plain = torch.zeros(B, n_plain, dtype=torch.int32, device=dev)
    eng.decode_plain(n_plain, plain)
    R = torch.cat([first.view(B, 1), plain], 1).contiguous()
    eng.prefill(prompts, R)
    eng.cycle()
    eng.sync()
    torch.cuda.synchronize()
    # the region is also bracketed by cudaProfilerStart/Stop: under `ncu --profile-from-start
    # off` only its launches are seen, so -s/-c count from the first cycle's first kernel
    out = torch.zeros(B, 2, dtype=torch.int32, device=dev)
    torch.cuda.profiler.start()
    torch.cuda.nvtx.range_push("profiled")
    for _ in range(args.steps):
        eng.cycle()
    eng.decode_plain(2, out)
    eng.sync()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    torch.cuda.profiler.stop()
    print(json.dumps({"ncu_region": True, "workload": wl.name, "batch": B, "cycles": args.steps, "plain_steps": 2}))


def run_gemm_probe(args):
    """One projection GEMM in isolation (weight larger than L2), timed with CUDA events:
    the kernel the roofline reports, at a verify-pass shape."""
    from eagle_speculative_decoding_cycle_gb300 import _lib as L
    from eagle_speculative_decoding_cycle_gb300.build import build
    build()
    lib = L.lib()
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(0)
    M, N, K = args.gemm_shape
    # enough weight copies, used in turn, that consecutive launches stream from HBM, not L2
    copies = max(1, -(-(320 << 20) // (N * K * 2)))
    Ws = [(torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16) for _ in range(copies)]
    X = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    out = torch.zeros(M, N, dtype=torch.float32, device=dev)
    nb = lib.eagle_op_gemm_scratch_bytes(M, N)
    scratch = torch.zeros(nb, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream().cuda_stream
    turn = {"i": 0}

    def call():
        W = Ws[turn["i"] % copies]
        turn["i"] += 1
        L.check(lib.eagle_op_gemm(L.DTYPE_BF16, st, W.data_ptr(), N, K, X.data_ptr(), M, 0, out.data_ptr(), N,
                                  scratch.data_ptr(), nb), "eagle_op_gemm")

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    # back-to-back launches replayed from a CUDA graph, so the host-side call overhead
    # (tensor-map encode, argument checks) is not timed; inputs are larger than L2 for the
    # verify-pass shapes, so consecutive launches stream the weight from HBM
    reps = 10 * copies
    gs = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gs):
        st = gs.cuda_stream
        graph.capture_begin()
        for _ in range(reps):
            call()
        graph.capture_end()
    ts = []
    with torch.cuda.stream(gs):
        graph.replay()
        torch.cuda.synchronize()
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(gs)
            graph.replay()
            e1.record(gs)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / reps)
    byt = N * K * 2 + M * K * 2 + M * N * 4
    us = statistics.median(ts) * 1e3
    hbm, src = peaks()
    print(json.dumps({"gemm": [M, N, K], "weight_copies": copies, "us_median": us, "us_min": min(ts) * 1e3,
                      "gbs": byt / us / 1e3, "frac": byt / us / 1e3 / hbm, "peak_source": src}))


def run_attn_probe(args):
    """The tree-mode attention kernel in isolation (contiguous cache larger than L2), timed
    with CUDA events over graph-replayed launches: B sequences of CTX context keys, ROWS tree
    rows each (a chain: row i sees rows 0..i), Llama-3.1-8B head geometry (32 query heads,
    8 KV heads, head dim 128), with the key splits of an engine serving B sequences."""
    from eagle_speculative_decoding_cycle_gb300 import _lib as L
    from eagle_speculative_decoding_cycle_gb300 import api
    from eagle_speculative_decoding_cycle_gb300.build import build
    build()
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(0)
    B, CTX, T = args.attn_shape
    nq, nkv, d = 32, 8, 128
    cap = CTX + T + 16
    R = B * T
    kc = torch.randn(B, nkv, cap, d, generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn(B, nkv, cap, d, generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn(R, nq, d, generator=g, device=dev).to(torch.bfloat16)
    row_seq = torch.arange(R, device=dev, dtype=torch.int32) // T
    row_slot = (CTX + torch.arange(R, device=dev, dtype=torch.int32) % T).to(torch.int32)
    ctx_len = torch.full((B,), CTX, dtype=torch.int32, device=dev)
    mw = (T + 63) // 64
    bits = torch.zeros(T, mw * 64, dtype=torch.bool)
    for i in range(T):
        bits[i, :i + 1] = True
    words = torch.zeros(T, mw, dtype=torch.int64)
    for w in range(mw):
        for b in range(64):
            words[:, w] |= bits[:, w * 64 + b].to(torch.int64) << b
    mask = words.repeat(B, 1).to(dev)
    gs = torch.cuda.Stream()

    def call():
        api.attention(q, kc, vc, row_seq, row_slot, ctx_len, T, 1, tree_T=T, mask=mask, stream=gs, max_batch=B)

    with torch.cuda.stream(gs):
        for _ in range(3):
            call()
    torch.cuda.synchronize()
    reps = 10
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gs):
        graph.capture_begin()
        for _ in range(reps):
            call()
        graph.capture_end()
    ts = []
    with torch.cuda.stream(gs):
        graph.replay()
        torch.cuda.synchronize()
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(gs)
            graph.replay()
            e1.record(gs)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / reps)
    byt = B * nkv * (CTX + T) * d * 2 * 2 + 2 * R * nq * d * 2
    us = statistics.median(ts) * 1e3
    hbm, src = peaks()
    print(json.dumps({"attention": {"batch": B, "ctx": CTX, "tree_rows": T, "nq": nq, "nkv": nkv, "d": d},
                      "us_median": us, "us_min": min(ts) * 1e3, "gbs": byt / us / 1e3, "frac": byt / us / 1e3 / hbm,
                      "peak_source": src}))


def run_plan_budget(args):
    """Measure the inputs of the batch-aware budget planner on this GPU, plan (k, m) per batch
    size, and apply each plan: for k in (4, 8, 10) the expected committed tokens of the m best
    nodes (1 + the sum of their path values, averaged over planted cycles) and the drafter's
    share of a cycle; the verify-pass time at batch 1, 4, 16 and 64 (k10, m60); then, per
    batch size, measured committed tokens per second with the workload's own (k, m) and with
    the planned one, set between cycles on one engine."""
    from eagle_speculative_decoding_cycle_gb300 import _lib as L
    from eagle_speculative_decoding_cycle_gb300 import api
    from eagle_speculative_decoding_cycle_gb300.build import build
    build()
    dev = torch.device("cuda:0")
    base = synth.WORKLOADS[args.workload]
    weights = synth.make_weights(base, device=str(dev))
    stream = torch.cuda.Stream(device=dev)
    prompt = synth.make_prompts(base)[0].to(dev)
    D = base.tree.depth
    n_cyc = 12
    cands = []
    for k in (4, 8, 10):
        t = dataclasses.replace(base.tree, topk=k, m=min(60, k + (D - 1) * k * k))
        wl = base.replace(tree=t)
        eng = api.Engine(wl, weights, max_ctx=len(prompt) + 6 * (n_cyc + 8) * (D + 1) + 64, stream=stream)
        with torch.cuda.stream(stream):
            eng.prefill([prompt])
            first = int(eng.dump(L.DUMP_STATE)["root_tok"][0])
            plain = torch.zeros(1, (n_cyc + 6) * (D + 1), dtype=torch.int32, device=dev)
            eng.decode_plain(plain.shape[1], plain)
            eng.sync()
            ref = torch.cat([torch.tensor([[first]], dtype=torch.int32, device=dev), plain], 1).contiguous()
            eng.prefill([prompt], ref)
            curve = np.zeros(t.n_gen)
            for i in range(n_cyc + 2):
                eng.cycle()
                eng.sync()
                if i >= 2:
                    logv = eng.dump(L.DUMP_NODES)[3][0].double().numpy()
                    curve += np.cumsum(np.sort(np.exp(logv))[::-1])
            curve = 1.0 + curve / n_cyc
            eng.prefill([prompt], ref)
            eng.set_graph(True)
            for _ in range(3):
                eng.cycle()
            eng.sync()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n_cyc):
                eng.cycle()
            e1.record(stream)
            eng.sync()
            cycle_us = e0.elapsed_time(e1) * 1e3 / n_cyc
            eng.set_graph(False)
            eng.profile_begin(0)
            for _ in range(3):
                eng.cycle()
            eng.profile_end()
            nv, vms = eng.profile_verify()
        eng.close()
        draft_us = max(0.0, cycle_us - vms * 1e3 / max(nv, 1))
        cands.append((k, draft_us, [float(x) for x in curve[:min(t.n_gen, 255)]]))
    rows, vus = [], []
    for B in (1, 4, 16, 64):
        wl = base.replace(batch=B)
        prompts = [prompt] * B
        eng = api.Engine(wl, weights, max_batch=B, max_ctx=len(prompt) + 12 * (D + 1) + 64, stream=stream)
        with torch.cuda.stream(stream):
            eng.prefill(prompts)
            eng.cycle()
            eng.sync()
            eng.profile_begin(0)
            for _ in range(3):
                eng.cycle()
            eng.profile_end()
            nv, vms = eng.profile_verify()
        eng.close()
        rows.append(B * (base.tree.m + 1))
        vus.append(vms * 1e3 / max(nv, 1))
    plans = {}
    for B in (1, 4, 16, 64):
        k, m, rate = api.plan_budget(cands, rows, vus, B)
        plans[B] = {"k": k, "m": m, "committed_tok_per_s": rate * 1e6}
    # apply each plan between cycles (eagle_set_tree_budget) on an engine created with the
    # largest k and m, against the workload's own (k, m) on the same engine; planted cycles
    # on the batch's own plain continuation, graph-replayed, committed tokens per second
    k_max = max(c[0] for c in cands)
    m_max = max(60, base.tree.m)
    big = base.replace(tree=dataclasses.replace(base.tree, topk=k_max, m=m_max))
    for B in (1, 4, 16, 64):
        prompts = [p.to(dev) for p in (synth.make_prompts(base.replace(batch=max(B, base.batch)))[:B])]
        n_meas = 8
        n_ref = (n_meas + 8) * (D + 1) + D + 2
        eng = api.Engine(big.replace(batch=B), weights, max_batch=B,
                         max_ctx=max(len(p) for p in prompts) + 2 * n_ref + 64, stream=stream)
        with torch.cuda.stream(stream):
            eng.prefill(prompts)
            first = eng.dump(L.DUMP_STATE)["root_tok"][:B].to(torch.int32).view(B, 1).to(dev)
            rest = torch.zeros(B, n_ref - 1, dtype=torch.int32, device=dev)
            eng.decode_plain(n_ref - 1, rest)
            eng.sync()
            ref = torch.cat([first, rest], 1).contiguous()
            meas = {}
            for label, (k, m) in (("default", (base.tree.topk, base.tree.m)),
                                  ("planned", (plans[B]["k"], plans[B]["m"]))):
                eng.set_graph(False)
                eng.set_tree_budget(k, m)
                eng.prefill(prompts, ref)
                eng.set_graph(True)
                for _ in range(2):
                    eng.cycle()
                eng.sync()
                c0 = int(eng.dump(L.DUMP_STATE)["committed"][:B].long().sum())
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(n_meas):
                    eng.cycle()
                e1.record(stream)
                eng.sync()
                c1 = int(eng.dump(L.DUMP_STATE)["committed"][:B].long().sum())
                ms = e0.elapsed_time(e1)
                meas[label] = {"k": k, "m": m, "committed_tok_per_s": (c1 - c0) / (ms / 1e3),
                               "cycle_ms": ms / n_meas, "tau": (c1 - c0) / n_meas / B}
            plans[B]["measured"] = meas
        eng.close()
    print(json.dumps({"plan_budget": {
        "workload": base.name, "verify_rows": rows, "verify_us": vus,
        "draft_us": {c[0]: c[1] for c in cands},
        "expected_tokens_at_m": {c[0]: {m: round(c[2][m - 1], 3) for m in (1, 4, 8, 16, 32, 60) if m <= len(c[2])}
                                 for c in cands},
        "plan": plans}}))


def run_reference(args, ws, rank, local):
    """The oracle as it stands, on the host cores, as the reference arm: full-depth cycles of
    the workload's shapes (see oracle_sample), one untimed warm-up cycle, then up to
    `--steps` timed cycles within `--ref-budget` seconds; the line reports the cycles it
    actually timed."""
    if rank != 0:
        return None
    wl = synth.WORKLOADS[args.workload]
    dev = torch.device(f"cuda:{local}") if torch.cuda.is_available() else torch.device("cpu")
    weights = synth.make_weights(wl, device=str(dev))
    t0 = time.perf_counter()
    cb = oracle_sample(wl, weights, args.steps, 1, budget_s=args.ref_budget)
    wall = time.perf_counter() - t0
    v = cb["value"]
    return {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws, "steps": cb["cycles"], "warmup": 1,
            "ms_per_step": cb["s_per_cycle"] * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": wl.name, "batch": wl.batch, "prompt": CPU_PROMPT},
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "requested_steps": args.steps, "requested_warmup": args.warmup,
            "consistency": {"timed_s": cb["s_per_cycle"] * cb["cycles"], "wall_s": wall}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=synth.LLAMA31_8B_SAMPLE.name, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--planted-p", type=float, default=None)
    ap.add_argument("--tree", default="dynamic", choices=["dynamic", "static-chain", "static-prior"],
                    help="tree policy: EAGLE-2 dynamic (default) or a static EAGLE-1 style shape")
    ap.add_argument("--prof-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-steps", type=int, default=2)
    ap.add_argument("--ref-budget", type=float, default=150.0)
    ap.add_argument("--gemm-shape", type=int, nargs=3, default=None, metavar=("M", "N", "K"),
                    help="only time one projection GEMM of this shape (for ncu and tuning)")
    ap.add_argument("--ncu-region", action="store_true",
                    help="only run a short NVTX-marked region for an ncu launch list")
    ap.add_argument("--attn-shape", type=int, nargs=3, default=None, metavar=("B", "CTX", "ROWS"),
                    help="time the tree-mode attention kernel alone (8B head geometry, contiguous cache)")
    ap.add_argument("--plan-budget", action="store_true",
                    help="measure the budget planner's inputs on this GPU and plan (k, m) per batch size")
    ap.add_argument("--layers", type=int, default=0,
                    help="with --ncu-region: truncate the target to this many layers (small profiling case)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.ncu_region:
        run_ncu_region(args)
        return
    if args.gemm_shape:
        run_gemm_probe(args)
        return
    if args.attn_shape:
        run_attn_probe(args)
        return
    if args.plan_budget:
        run_plan_budget(args)
        return
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, ws, rank, local)
    else:
        res, wl, weights = run_ours(args, ws, rank, local)
        if rank == 0 and ws == 1 and not args.no_cpu_baseline:
            cb = oracle_sample(wl, weights, args.cpu_steps, 0, budget_s=30.0)
            res["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
        elif rank == 0:
            res["cpu_baseline"] = None
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
