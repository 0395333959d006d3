#!/usr/bin/env python
"""Benchmark of the DFlash drafter gamma-block forward on one GB300 (per rank).

Metric: draft tokens/s = nb * (gamma - 1) / t_fwd over K timed steps, each step one
dflash_propose (the whole hot path: embedding, every layer, final norm, lm_head, argmax)
on a batch whose paged context K/V was written beforehand.  Synthetic, seeded inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line on rank 0.  Under torchrun each rank runs an independent replica
(the path shards by sequence; no collective on the data path): value = draft tokens of
all ranks / max over ranks of the timed region.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import WORKLOADS, make_weights, workload_taps  # noqa: E402

DEFAULT_WORKLOAD = "qwen3_8l_nb1_ctx4096"
METRIC = "draft tokens/s per gamma=16 block forward"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-logits", action="store_true", help="tokens only (logits=NULL)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ----------------------------------------------------------------------------- algorithmic work


def work_model(cfg, wl, logits: bool):
    """Algorithmic bytes / flops of one forward (every weight once, visible K/V once per
    (sequence, layer), block K/V writes, embedding rows, logits write)."""
    es = 4 if cfg.dtype == "f32" else 2
    H, F, V, hd, nh, nkv, L = cfg.hidden, cfg.n_ff, cfg.vocab, cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads, cfg.n_layers
    M = wl.nb * cfg.gamma
    layer_w = ((nh + 2 * nkv) * hd * H + H * nh * hd + 3 * F * H) * es + (2 * H + 2 * hd) * es
    lm_w = V * H * (1 if cfg.lm_head_dtype == "fp8" else es) + (V * 4 if cfg.lm_head_dtype == "fp8" else 0)
    keys = []
    for s in range(wl.nb):
        c = int(wl.ctx_lens[s])
        w = cfg.sliding_window
        keys.append([(min(c + cfg.gamma, w + cfg.gamma - 1) if (cfg.sliding(l) and w > 0) else c + cfg.gamma)
                     for l in range(L)])
    kv_read = sum(sum(k) for k in keys) * 2 * nkv * hd * es
    kv_write = L * M * 2 * nkv * hd * es
    nbytes = L * layer_w + lm_w + kv_read + kv_write + M * H * es + (M * V * es if logits else 0)
    flops = 2 * M * (L * ((nh + 2 * nkv) * hd * H + H * nh * hd + 3 * F * H) + V * H)
    flops += sum(sum(4 * cfg.gamma * nh * hd * k for k in ks) for ks in keys)
    per_kernel = {
        "qkv_gemm": ((nh + 2 * nkv) * hd * H * es + M * H * es, 2 * M * (nh + 2 * nkv) * hd * H),
        "o_proj_gemm": (H * nh * hd * es + M * nh * hd * es, 2 * M * H * nh * hd),
        "gate_up_gemm": (2 * F * H * es + M * H * es, 4 * M * F * H),
        "down_gemm": (H * F * es + M * F * es, 2 * M * H * F),
        "lm_head": (lm_w + M * H * es + (M * V * es if logits else 0), 2 * M * V * H),
        "attention": (kv_read / L + M * nh * hd * es * 2, sum(sum(4 * cfg.gamma * nh * hd * k for k in ks)
                                                               for ks in keys) / L),
        # the single-launch forward does the whole step's work in one kernel
        "persistent_forward": (nbytes, flops),
    }
    return nbytes, flops, per_kernel


# The sources that define each measured kernel (its own file and every header it includes).
KERNEL_SOURCES = {
    "persistent_forward": ("persist_tc.cu", "persist_tc.cuh", "gemm_epi.cuh", "gemm_tc.cuh", "tc_common.cuh",
                           "dflash_internal.cuh"),
}


def kernel_sources_sha(kernel: str = "persistent_forward", read=None) -> str:
    """Hash of the sources of `kernel`, to tell whether a stored ncu traffic figure still
    applies.  `read(name) -> bytes` overrides how a file under csrc/ is read."""
    import hashlib
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "block_diffusion_drafter_forward_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name), "rb") as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in sorted(KERNEL_SOURCES.get(kernel, ())):
        h.update(f.encode() + read(f))
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on these sources."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "dram_traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(f"{kernel}@{workload}")
    except (OSError, ValueError):
        return None
    if not rec or kernel not in KERNEL_SOURCES or rec.get("sources_sha") != kernel_sources_sha(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        with open(self.path) as fh:
            for ln in fh:
                p = [x.strip() for x in ln.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                               r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------- oracle timing


def oracle_threads() -> int:
    """Threads the oracle's numpy BLAS runs on: the usual thread-count variables when set, else
    every core (the OpenBLAS default)."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return min(int(v), os.cpu_count() or 1)
    return os.cpu_count() or 1


def oracle_timing(wl, budget_s: float = 20.0):
    """The CPU oracle (float64 numpy, as it stands) on a bounded sample of the workload:
    context K/V of one band precomputed, then its gamma-block forward + lm_head + argmax
    timed, repeated while within the budget."""
    from oracle.dflash_oracle import Oracle

    cfg = wl.cfg
    W = make_weights(cfg, wl.seed)
    o = Oracle(cfg, W, cache=True)
    s = 0
    c = int(wl.ctx_lens[s])
    f = o.ctx_features(workload_taps(wl, s, 0, c))
    ks, vs = o.ctx_kv(f, wl.ctx_positions(s, 0, c))
    del f
    times = []
    t_all = time.time()
    while True:
        t0 = time.perf_counter()
        h = o.forward_block(ks, vs, wl.ctx_positions(s, 0, c), int(wl.bonus[s]), c)
        o.drafts(h)
        times.append(time.perf_counter() - t0)
        if time.time() - t_all + times[-1] > budget_s or len(times) >= 5:
            break
    t = statistics.mean(times)
    return {"value": (cfg.gamma - 1) / t, "unit": "draft tokens/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"band 0 of {wl.name} (ctx {c}): float64 numpy gamma-block forward + lm_head + argmax, "
                      f"{len(times)} run(s), context K/V precomputed outside the timing"}


# ----------------------------------------------------------------------------- main


def aggregate_over_ranks(local_ms: float, tokens_per_rank: int, dist=None, device="cpu"):
    """Replicas: each rank timed its own batch.  Returns (max over ranks of the timed region in
    ms, whole-job tokens/s = tokens of all ranks / that max)."""
    import torch

    world = 1
    t = local_ms
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        buf = torch.tensor([local_ms], dtype=torch.float64, device=device)
        dist.all_reduce(buf, op=dist.ReduceOp.MAX)
        t = float(buf.item())
    return t, world * tokens_per_rank / (t / 1e3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, world, rank):
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]()
    wl.name = args.workload
    cfg = wl.cfg
    from oracle.dflash_oracle import Oracle
    W = make_weights(cfg, wl.seed)
    o = Oracle(cfg, W, cache=True)
    s = 0
    c = int(wl.ctx_lens[s])
    f = o.ctx_features(workload_taps(wl, s, 0, c))
    ks, vs = o.ctx_kv(f, wl.ctx_positions(s, 0, c))
    for _ in range(max(args.warmup, 0)):
        o.drafts(o.forward_block(ks, vs, wl.ctx_positions(s, 0, c), int(wl.bonus[s]), c))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.drafts(o.forward_block(ks, vs, wl.ctx_positions(s, 0, c), int(wl.bonus[s]), c))
    dt = time.perf_counter() - t0
    value = args.steps * (cfg.gamma - 1) / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "draft tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": wl.name, "nb_timed": 1, "ctx": c},
            "cpu_baseline": {"value": value, "unit": "draft tokens/s", "cores": oracle_threads(), "kind": "oracle",
                             "sample": f"band 0 of {wl.name}: one gamma-block forward + lm_head + argmax per step "
                                       "(float64 numpy oracle); context K/V precomputed before the timing"},
            "e2e": {"value": value, "unit": "draft tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    import torch

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    from block_diffusion_drafter_forward_gb300 import Drafter, dflash_profile, dflash_profile_read
    from synth.inputs import taps_table
    from synth.torch_io import to_torch, upload_weights

    wl = WORKLOADS[args.workload]()
    wl.name = args.workload
    cfg = wl.cfg
    logits_on = not args.no_logits
    W = make_weights(cfg, wl.seed)
    tensors = upload_weights(W)
    drafter = Drafter(cfg, tensors, num_pages=wl.num_pages, max_batch=wl.nb, max_pages_per_seq=wl.max_pages_per_seq,
                      max_write_rows=4096)
    table = to_torch(taps_table(wl), cfg.dtype)
    page_tables = to_torch(wl.page_tables, "i32")
    for s in range(wl.nb):
        c = int(wl.ctx_lens[s])
        idx = (int(wl.tap_offsets[s]) + torch.arange(c, device="cuda")) % wl.taps_rows
        drafter.write_ctx_kv(table[idx].contiguous(), to_torch(wl.ctx_positions(s, 0, c), "i32"), page_tables[s], 0)
    del table
    torch.cuda.synchronize()
    bonus = to_torch(wl.bonus, "i32")
    ctx_lens = to_torch(wl.ctx_lens, "i32")
    M = wl.nb * cfg.gamma
    dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    logits = torch.empty((M, cfg.vocab), dtype=dt, device="cuda") if logits_on else None
    drafts = torch.empty((wl.nb, cfg.gamma - 1), dtype=torch.int32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        drafter.propose(bonus, ctx_lens, page_tables, wl.max_ctx_len, drafts=drafts, logits=logits)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()

    # ---- device-timed region: K steps (one CUDA-graph replay each), L2 flushed before each,
    # events on the launch stream
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    tokens_per_step = wl.nb * (cfg.gamma - 1)
    total_ms, value = aggregate_over_ranks(sum(step_ms), tokens_per_step * args.steps, dist, "cuda")
    ms_per_step = total_ms / args.steps

    # ---- per-kernel durations: the same K steps again, replaying the graph captured with
    # CUDA events around every kernel (the events serialise the kernels, so this pass is
    # only used for per-kernel times; the value above comes from the plain replay)
    dflash_profile(drafter.handle, True)
    step()
    torch.cuda.synchronize()
    dflash_profile(drafter.handle, True)
    for i in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    prof = dflash_profile_read(drafter.handle)
    dflash_profile(drafter.handle, False)
    prof_steps = args.steps

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timing
    h_bonus = torch.from_numpy(wl.bonus.copy()).pin_memory()
    h_ctx = torch.from_numpy(wl.ctx_lens.copy()).pin_memory()
    h_pt = torch.from_numpy(wl.page_tables.copy()).pin_memory()
    h_drafts = torch.empty((wl.nb, cfg.gamma - 1), dtype=torch.int32).pin_memory()
    d_bonus, d_ctx, d_pt = torch.empty_like(bonus), torch.empty_like(ctx_lens), torch.empty_like(page_tables)
    e2e_ms = 0.0
    for i in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        d_bonus.copy_(h_bonus, non_blocking=True)
        d_ctx.copy_(h_ctx, non_blocking=True)
        d_pt.copy_(h_pt, non_blocking=True)
        drafter.propose(d_bonus, d_ctx, d_pt, wl.max_ctx_len, drafts=drafts, logits=logits)
        h_drafts.copy_(drafts, non_blocking=True)
        b.record(stream)
        b.synchronize()
        e2e_ms += a.elapsed_time(b)
    e2e_ms, e2e_value = aggregate_over_ranks(e2e_ms, tokens_per_step * args.steps, dist, "cuda")
    e2e = {"value": e2e_value, "unit": "draft tokens/s",
           "h2d_bytes_per_step": int(h_bonus.numel() * 4 + h_ctx.numel() * 4 + h_pt.numel() * 4),
           "d2h_bytes_per_step": int(h_drafts.numel() * 4)}

    # ---- context-K/V writer (the step before the path): rows/s at n = 16 and n = 4096,
    # rewriting rows of sequence 0 with their own taps (same values), events on the stream
    writer = {}
    c0 = int(wl.ctx_lens[0])
    tab = to_torch(taps_table(wl), cfg.dtype)
    for n in (16, 4096):
        n = min(n, c0)
        if n <= 0:
            continue
        idx = (int(wl.tap_offsets[0]) + torch.arange(n, device="cuda")) % wl.taps_rows
        taps0 = tab[idx].contiguous()
        pos0 = to_torch(wl.ctx_positions(0, 0, n), "i32")
        for _ in range(3):
            drafter.write_ctx_kv(taps0, pos0, page_tables[0], 0)
        reps = 20 if n <= 64 else 5
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            drafter.write_ctx_kv(taps0, pos0, page_tables[0], 0)
        b.record(stream)
        b.synchronize()
        ms = a.elapsed_time(b) / reps
        wbytes = (cfg.hidden * cfg.tap_dim + cfg.n_layers * 2 * cfg.kv_dim * cfg.hidden) * (4 if cfg.dtype == "f32" else 2)
        wbytes += n * cfg.tap_dim * (4 if cfg.dtype == "f32" else 2) + n * cfg.n_layers * 2 * cfg.kv_dim * (4 if cfg.dtype == "f32" else 2)
        wflops = 2.0 * n * (cfg.hidden * cfg.tap_dim + cfg.n_layers * 2 * cfg.kv_dim * cfg.hidden)
        writer[f"n{n}"] = {"rows_per_s": n / (ms / 1e3), "us_per_call": 1e3 * ms,
                           "hbm_frac": wbytes / (ms / 1e3) / (peaks()[0]["hbm_gbs"] * 1e9),
                           "tensor_frac": wflops / (ms / 1e3) / (peaks()[0]["bf16_tflops"] * 1e12)}
    del tab

    # ---- roofline of the dominant kernel
    pk, src = peaks()
    nbytes, flops, per_kernel = work_model(cfg, wl, logits_on)
    kernels = {k: v for k, v in prof.items() if v[1] > 0 and k != "copy"}
    launches = sum(v[1] for v in kernels.values())
    dom = max(kernels, key=lambda k: kernels[k][0])
    dom_ms, dom_n = kernels[dom]
    roof = None
    if dom in per_kernel:
        b_per, f_per = per_kernel[dom]
        t_launch = dom_ms / dom_n / 1e3
        bw = b_per / t_launch / 1e9
        tf = f_per / t_launch / 1e12
        peak_tf = pk["bf16_tflops"]
        if f_per / max(b_per, 1) > peak_tf * 1e3 / pk["hbm_gbs"]:
            roof = {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": tf / peak_tf}
        else:
            roof = {"bound": "hbm", "achieved": bw, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": bw / pk["hbm_gbs"]}
        roof.update({"kernel": dom, "traffic": measured_traffic(dom, wl.name), "peak_source": src,
                     "algorithmic_bytes_per_launch": b_per, "launch_us": 1e6 * t_launch})
    t_roof = max(nbytes / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))

    line = {
        "metric": METRIC, "value": value, "unit": "draft tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if cfg.dtype == "f32" else "bf16", "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "nb": wl.nb, "ctx_mean": float(np.mean(wl.ctx_lens)),
                   "layers": cfg.n_layers, "hidden": cfg.hidden, "vocab": cfg.vocab,
                   "lm_head": cfg.lm_head_dtype, "logits_written": logits_on,
                   "l2": "256 MB buffer written before every timed step (outside the events)",
                   "parallelism": f"replicas x{world}"},
        "fwd_per_s": value / tokens_per_step,
        "step_roofline": {"bytes": nbytes, "flops": flops, "t_roof_us": 1e6 * t_roof,
                          "frac": t_roof / (ms_per_step / 1e3), "peak_source": src},
        "roofline": roof,
        "kernels_ms_per_step": {k: v[0] / prof_steps for k, v in kernels.items()},
        "gpu_launches": int(launches),
        "e2e": e2e,
        "writer": writer,
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["clocks"] = clk.summary()
        line["cpu_baseline"] = oracle_timing(wl)
    elif rank == 0:
        line["clocks"] = clk.summary()
    if rank == 0:
        print(json.dumps(line), flush=True)
    drafter.close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
