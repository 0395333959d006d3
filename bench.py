#!/usr/bin/env python
"""Benchmark of the DFlash drafter gamma-block forward on one GB300 (per rank).

Metric: draft tokens/s = nb * (gamma - 1) / t_fwd over K timed steps, each step one
dflash_propose (the whole hot path: embedding, every layer, final norm, lm_head, argmax)
on a batch whose paged context K/V was written beforehand.  Synthetic, seeded inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                  [--sweep] [--no-extra] [--no-logits] [--no-cpu-baseline]

Prints one JSON line on rank 0.  Under torchrun each rank runs an independent replica
(the path shards by sequence; no collective on the data path): value = draft tokens of
all ranks / max over ranks of the timed region.  Beside the headline workload (one
sequence, context 4096) the line carries the 32-sequence ragged batch under "nb32", a
median over --long-reps replays, the context-K/V writer's rate, every kernel's fraction of
its own roofline, and the CPU oracle timed on the host cores (all cores and one thread).
--sweep adds the FP8-lm_head batches nb = 1, 4, 16, 64 at context 32768.
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
    "attention": ("attn_tc.cu", "attn_tc.cuh", "tc_common.cuh", "dflash_internal.cuh"),
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


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=30).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_leg(workload: str, budget_s: float, max_runs: int, warmup: int = 0):
    """The CPU oracle (float64 numpy, as it stands) on a bounded sample of the workload:
    the context K/V of band 0 precomputed, then its gamma-block forward + lm_head + argmax
    timed, repeated while within the budget.  Runs in whatever process calls it; the BLAS
    thread count is fixed by that process's environment."""
    from oracle.dflash_oracle import Oracle

    wl = WORKLOADS[workload]()
    cfg = wl.cfg
    W = make_weights(cfg, wl.seed)
    o = Oracle(cfg, W, cache=True)
    s = 0
    c = int(wl.ctx_lens[s])
    f = o.ctx_features(workload_taps(wl, s, 0, c))
    ks, vs = o.ctx_kv(f, wl.ctx_positions(s, 0, c))
    del f
    for _ in range(max(warmup, 0)):
        o.drafts(o.forward_block(ks, vs, wl.ctx_positions(s, 0, c), int(wl.bonus[s]), c))
    times = []
    t_all = time.time()
    while True:
        t0 = time.perf_counter()
        h = o.forward_block(ks, vs, wl.ctx_positions(s, 0, c), int(wl.bonus[s]), c)
        o.drafts(h)
        times.append(time.perf_counter() - t0)
        if time.time() - t_all + times[-1] > budget_s or len(times) >= max_runs:
            break
    return {"runs": len(times), "s_per_forward": statistics.mean(times), "total_s": sum(times),
            "threads": oracle_threads(), "ctx": c, "gamma": cfg.gamma}


def run_oracle_leg(workload: str, threads: int, budget_s: float, max_runs: int, warmup: int = 0):
    """oracle_leg in a fresh interpreter whose BLAS thread count is set to `threads` before numpy
    loads (an exec'd child: nothing of a CUDA context is inherited)."""
    env = dict(os.environ)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(threads)
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-leg", workload, "--leg-budget", str(budget_s),
           "--leg-runs", str(max_runs), "--warmup", str(warmup)]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=3600)
    if r.returncode != 0:
        raise RuntimeError(f"oracle leg failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_timing(workload: str):
    """The bench's cpu_baseline: the oracle on the host cores, once with the BLAS on every core
    and once single-threaded, each on band 0 of the workload (bounded runs)."""
    ncpu = os.cpu_count() or 1
    multi = run_oracle_leg(workload, ncpu, 15.0, 5)
    single = run_oracle_leg(workload, 1, 25.0, 3)
    g = multi["gamma"]
    model = cpu_model()
    return {"value": (g - 1) / multi["s_per_forward"], "unit": "draft tokens/s", "cores": multi["threads"],
            "kind": "oracle", "cpu_model": model,
            "sample": f"band 0 of {workload} (ctx {multi['ctx']}): float64 numpy gamma-block forward + lm_head + "
                      f"argmax, {multi['runs']} run(s) with the BLAS on {multi['threads']} threads; context K/V "
                      "precomputed outside the timing",
            "single_thread": {"value": (g - 1) / single["s_per_forward"], "unit": "draft tokens/s", "cores": 1,
                              "runs": single["runs"]}}


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
    """The reference arm: the oracle, as it stands, on the host cores (every core, the BLAS thread
    count set explicitly), one gamma-block forward per step on band 0 of the workload."""
    if rank != 0:
        return
    ncpu = os.cpu_count() or 1
    leg = run_oracle_leg(args.workload, ncpu, 1e9, args.steps, warmup=args.warmup)
    g = leg["gamma"]
    dt = leg["total_s"]
    value = args.steps * (g - 1) / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "draft tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": args.workload, "nb_timed": 1, "ctx": leg["ctx"]},
            "cpu_baseline": {"value": value, "unit": "draft tokens/s", "cores": leg["threads"], "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"band 0 of {args.workload}: one gamma-block forward + lm_head + argmax per "
                                       f"step (float64 numpy oracle, BLAS on {leg['threads']} threads); context "
                                       "K/V precomputed before the timing"},
            "e2e": {"value": value, "unit": "draft tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def kernel_fractions(prof, per_kernel, steps, pk):
    """Per kernel kind: mean launch time and the fraction of its own roofline (algorithmic
    bytes or flops of one launch over that time, against the measured peak of its bound)."""
    out = {}
    ridge = pk["bf16_tflops"] * 1e3 / pk["hbm_gbs"]
    for k, (ms, n) in prof.items():
        if n <= 0 or k == "copy":
            continue
        e = {"ms_per_step": ms / steps, "launches_per_step": n / steps}
        if k in per_kernel:
            b_per, f_per = per_kernel[k]
            t = ms / n / 1e3
            if f_per / max(b_per, 1) > ridge:
                e.update(bound="tensor", achieved=f_per / t / 1e12, unit="TFLOP/s",
                         frac=f_per / t / 1e12 / pk["bf16_tflops"])
            else:
                e.update(bound="hbm", achieved=b_per / t / 1e9, unit="GB/s", frac=b_per / t / 1e9 / pk["hbm_gbs"])
        out[k] = e
    return out


class Bench:
    """One workload on this rank's GPU: the drafter, its paged context written, and the buffers of
    one propose step."""

    def __init__(self, name: str, logits_on: bool, max_write_rows: int = 4096):
        import torch
        from block_diffusion_drafter_forward_gb300 import Drafter
        from synth.inputs import taps_table
        from synth.torch_io import to_torch, upload_weights

        self.torch = torch
        wl = WORKLOADS[name]()
        wl.name = name
        self.wl, self.cfg = wl, wl.cfg
        cfg = wl.cfg
        self.logits_on = logits_on
        W = make_weights(cfg, wl.seed)
        self.tensors = upload_weights(W)
        self.drafter = Drafter(cfg, self.tensors, num_pages=wl.num_pages, max_batch=wl.nb,
                               max_pages_per_seq=wl.max_pages_per_seq, max_write_rows=max_write_rows)
        self.table = to_torch(taps_table(wl), cfg.dtype)
        self.page_tables = to_torch(wl.page_tables, "i32")
        for s in range(wl.nb):
            c = int(wl.ctx_lens[s])
            idx = (int(wl.tap_offsets[s]) + torch.arange(c, device="cuda")) % wl.taps_rows
            self.drafter.write_ctx_kv(self.table[idx].contiguous(), to_torch(wl.ctx_positions(s, 0, c), "i32"),
                                      self.page_tables[s], 0)
        torch.cuda.synchronize()
        self.bonus = to_torch(wl.bonus, "i32")
        self.ctx_lens = to_torch(wl.ctx_lens, "i32")
        M = wl.nb * cfg.gamma
        dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
        self.logits = torch.empty((M, cfg.vocab), dtype=dt, device="cuda") if logits_on else None
        self.drafts = torch.empty((wl.nb, cfg.gamma - 1), dtype=torch.int32, device="cuda")
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.stream = torch.cuda.current_stream()
        self.tokens_per_step = wl.nb * (cfg.gamma - 1)

    def step(self):
        self.drafter.propose(self.bonus, self.ctx_lens, self.page_tables, self.wl.max_ctx_len, drafts=self.drafts,
                             logits=self.logits)

    def timed(self, steps: int):
        """Per-step device times (ms) of `steps` graph replays, L2 flushed before each (outside
        the events), events on the launch stream."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            self.flush.zero_()
            evs[i][0].record(self.stream)
            self.step()
            evs[i][1].record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def profile(self, steps: int):
        """Per-kernel time: the same steps replaying the graph captured with CUDA events around
        every kernel (the events serialise the kernels; only used for per-kernel times)."""
        from block_diffusion_drafter_forward_gb300 import dflash_profile, dflash_profile_read
        torch = self.torch
        dflash_profile(self.drafter.handle, True)
        self.step()
        torch.cuda.synchronize()
        dflash_profile(self.drafter.handle, True)
        for _ in range(steps):
            self.flush.zero_()
            self.step()
        torch.cuda.synchronize()
        prof = dflash_profile_read(self.drafter.handle)
        dflash_profile(self.drafter.handle, False)
        return prof

    def roofline(self, prof, steps: int, ms_per_step: float):
        pk, src = peaks()
        nbytes, flops, per_kernel = work_model(self.cfg, self.wl, self.logits_on)
        kernels = {k: v for k, v in prof.items() if v[1] > 0 and k != "copy"}
        dom = max(kernels, key=lambda k: kernels[k][0])
        fr = kernel_fractions(prof, per_kernel, steps, pk)
        roof = None
        if dom in per_kernel and "frac" in fr[dom]:
            d = fr[dom]
            dom_ms, dom_n = kernels[dom]
            roof = {"bound": d["bound"], "achieved": d["achieved"],
                    "peak": pk["bf16_tflops"] if d["bound"] == "tensor" else pk["hbm_gbs"], "unit": d["unit"],
                    "frac": d["frac"], "kernel": dom, "traffic": measured_traffic(dom, self.wl.name),
                    "peak_source": src, "algorithmic_bytes_per_launch": per_kernel[dom][0],
                    "launch_us": 1e3 * dom_ms / dom_n}
        t_roof = max(nbytes / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
        step_roof = {"bytes": nbytes, "flops": flops, "t_roof_us": 1e6 * t_roof,
                     "frac": t_roof / (ms_per_step / 1e3), "peak_source": src}
        return roof, step_roof, fr, int(sum(v[1] for v in kernels.values()))

    def close(self):
        self.drafter.close()
        del self.tensors, self.table, self.flush


def extra_workload(name: str, steps: int, warmup: int, logits_on: bool):
    """A workload beside the headline one: its median step time over `steps` replays, the step
    roofline, the dominant kernel's roofline and every kernel's fraction of its own bound."""
    b = Bench(name, logits_on)
    for _ in range(max(warmup, 3)):
        b.step()
    ms = b.timed(steps)
    med = statistics.median(ms)
    prof = b.profile(min(steps, 20))
    roof, step_roof, fr, _ = b.roofline(prof, min(steps, 20), med)
    out = {"workload": name, "nb": b.wl.nb, "ctx_mean": float(np.mean(b.wl.ctx_lens)),
           "ctx_max": int(b.wl.max_ctx_len), "steps": steps, "ms_per_step_median": med,
           "ms_per_step_mean": statistics.mean(ms), "value": b.tokens_per_step / (med / 1e3),
           "unit": "draft tokens/s", "fwd_per_s": 1e3 / med, "step_roofline": step_roof, "roofline": roof,
           "kernels": fr, "persistent": bool(b.drafter.persistent)}
    b.close()
    return out


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-logits", action="store_true", help="tokens only (logits=NULL)")
    ap.add_argument("--no-extra", action="store_true", help="skip the 32-sequence batch and the long run")
    ap.add_argument("--sweep", action="store_true",
                    help="also time the FP8-lm_head workloads at nb = 1, 4, 16, 64 (context 32768)")
    ap.add_argument("--long-reps", type=int, default=300, help="replays of the median-of-reps leg")
    ap.add_argument("--oracle-leg", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--leg-budget", type=float, default=15.0, help=argparse.SUPPRESS)
    ap.add_argument("--leg-runs", type=int, default=5, help=argparse.SUPPRESS)
    return ap.parse_args()


def main():
    args = parse()
    if args.oracle_leg:
        print(json.dumps(oracle_leg(args.oracle_leg, args.leg_budget, args.leg_runs, args.warmup)), flush=True)
        return
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
    from synth.inputs import taps_table
    from synth.torch_io import to_torch

    logits_on = not args.no_logits
    b = Bench(args.workload, logits_on)
    wl, cfg = b.wl, b.cfg
    warm = max(args.warmup, 3)
    for _ in range(warm):
        b.step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()

    # ---- device-timed region: exactly K steps (one CUDA-graph replay each), L2 flushed before
    # each, events on the launch stream; clocks sampled from a soak of untimed replays before it
    # through the end of the timed region
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_soak = time.time()
        while time.time() - t_soak < 1.0:
            for _ in range(50):
                b.step()
            torch.cuda.synchronize()
        step_ms = b.timed(args.steps)
    if dist:
        dist.barrier()
    total_ms, value = aggregate_over_ranks(sum(step_ms), b.tokens_per_step * args.steps, dist, "cuda")
    ms_per_step = total_ms / args.steps

    prof_steps = min(args.steps, 50)
    prof = b.profile(prof_steps)

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timing
    h_bonus = torch.from_numpy(wl.bonus.copy()).pin_memory()
    h_ctx = torch.from_numpy(wl.ctx_lens.copy()).pin_memory()
    h_pt = torch.from_numpy(wl.page_tables.copy()).pin_memory()
    h_drafts = torch.empty((wl.nb, cfg.gamma - 1), dtype=torch.int32).pin_memory()
    d_bonus, d_ctx, d_pt = torch.empty_like(b.bonus), torch.empty_like(b.ctx_lens), torch.empty_like(b.page_tables)
    e2e_ms = 0.0
    for i in range(args.steps):
        b.flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(b.stream)
        d_bonus.copy_(h_bonus, non_blocking=True)
        d_ctx.copy_(h_ctx, non_blocking=True)
        d_pt.copy_(h_pt, non_blocking=True)
        b.drafter.propose(d_bonus, d_ctx, d_pt, wl.max_ctx_len, drafts=b.drafts, logits=b.logits)
        h_drafts.copy_(b.drafts, non_blocking=True)
        e1.record(b.stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms, e2e_value = aggregate_over_ranks(e2e_ms, b.tokens_per_step * args.steps, dist, "cuda")
    e2e = {"value": e2e_value, "unit": "draft tokens/s",
           "h2d_bytes_per_step": int(h_bonus.numel() * 4 + h_ctx.numel() * 4 + h_pt.numel() * 4),
           "d2h_bytes_per_step": int(h_drafts.numel() * 4)}

    # ---- median over many replays (after the K steps above), as a check on the K-step mean
    long_ms = b.timed(args.long_reps) if not args.no_extra and args.long_reps > 0 else []

    # ---- context-K/V writer (the step before the path): rows/s at n = 16 and n = 4096,
    # rewriting rows of sequence 0 with their own taps (same values), events on the stream
    writer = {}
    c0 = int(wl.ctx_lens[0])
    es = 4 if cfg.dtype == "f32" else 2
    for n in (16, 4096):
        n = min(n, c0)
        if n <= 0:
            continue
        idx = (int(wl.tap_offsets[0]) + torch.arange(n, device="cuda")) % wl.taps_rows
        taps0 = b.table[idx].contiguous()
        pos0 = to_torch(wl.ctx_positions(0, 0, n), "i32")
        for _ in range(3):
            b.drafter.write_ctx_kv(taps0, pos0, b.page_tables[0], 0)
        reps = 20 if n <= 64 else 5
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(b.stream)
        for _ in range(reps):
            b.drafter.write_ctx_kv(taps0, pos0, b.page_tables[0], 0)
        e1.record(b.stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1) / reps
        wbytes = (cfg.hidden * cfg.tap_dim + cfg.n_layers * 2 * cfg.kv_dim * cfg.hidden) * es
        wbytes += n * cfg.tap_dim * es + n * cfg.n_layers * 2 * cfg.kv_dim * es
        wflops = 2.0 * n * (cfg.hidden * cfg.tap_dim + cfg.n_layers * 2 * cfg.kv_dim * cfg.hidden)
        writer[f"n{n}"] = {"rows_per_s": n / (ms / 1e3), "us_per_call": 1e3 * ms,
                           "hbm_frac": wbytes / (ms / 1e3) / (peaks()[0]["hbm_gbs"] * 1e9),
                           "tensor_frac": wflops / (ms / 1e3) / (peaks()[0]["bf16_tflops"] * 1e12)}

    # batched writer: 32 sequences x 128 new rows in one call (rows of all sequences stacked),
    # against the same rows written by 32 per-sequence calls; rows land on sequence 0's first
    # 128 slots (same values as before), so the pool is unchanged
    if c0 >= 128:
        nseq, per = 32, 128
        idx = (int(wl.tap_offsets[0]) + torch.arange(per, device="cuda")) % wl.taps_rows
        taps1 = b.table[idx].contiguous()
        taps_b = taps1.repeat(nseq, 1)
        pos_b = to_torch(np.tile(wl.ctx_positions(0, 0, per), nseq), "i32")
        rs_b = torch.zeros(nseq * per, dtype=torch.int32, device="cuda")
        ri_b = to_torch(np.tile(np.arange(per, dtype=np.int32), nseq), "i32")
        pt0 = b.page_tables[:1].contiguous()
        pos1 = to_torch(wl.ctx_positions(0, 0, per), "i32")

        def timed_calls(fn, reps):
            for _ in range(2):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(b.stream)
            for _ in range(reps):
                fn()
            e1.record(b.stream)
            e1.synchronize()
            return e0.elapsed_time(e1) / reps

        ms_b = timed_calls(lambda: b.drafter.write_ctx_kv_batch(taps_b, pos_b, rs_b, ri_b, pt0), 5)
        ms_s = timed_calls(lambda: [b.drafter.write_ctx_kv(taps1, pos1, b.page_tables[0], 0) for _ in range(nseq)], 3)
        n = nseq * per
        wflops = 2.0 * n * (cfg.hidden * cfg.tap_dim + cfg.n_layers * 2 * cfg.kv_dim * cfg.hidden)
        writer["batched_32x128"] = {"rows_per_s": n / (ms_b / 1e3), "us_per_call": 1e3 * ms_b,
                                    "tensor_frac": wflops / (ms_b / 1e3) / (peaks()[0]["bf16_tflops"] * 1e12),
                                    "per_sequence_calls_us": 1e3 * ms_s, "speedup": ms_s / ms_b}

    roof, step_roof, fr, launches = b.roofline(prof, prof_steps, ms_per_step)
    launches_per_step = launches / prof_steps
    line = {
        "metric": METRIC, "value": value, "unit": "draft tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": warm, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if cfg.dtype == "f32" else "bf16", "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "nb": wl.nb, "ctx_mean": float(np.mean(wl.ctx_lens)),
                   "layers": cfg.n_layers, "hidden": cfg.hidden, "vocab": cfg.vocab,
                   "lm_head": cfg.lm_head_dtype, "logits_written": logits_on,
                   "l2": "256 MB buffer written before every timed step (outside the events)",
                   "parallelism": f"replicas x{world}"},
        "fwd_per_s": value / b.tokens_per_step,
        "step_roofline": step_roof,
        "roofline": roof,
        "kernels": fr,
        "kernels_ms_per_step": {k: v["ms_per_step"] for k, v in fr.items()},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "e2e": e2e,
        "writer": writer,
    }
    if long_ms:
        med = statistics.median(long_ms)
        line["median_of_reps"] = {"reps": len(long_ms), "ms_per_step": med, "value": b.tokens_per_step / (med / 1e3),
                                  "step_roofline_frac": step_roof["t_roof_us"] / 1e3 / med}
    b.close()
    del b
    torch.cuda.empty_cache()

    # ---- the other half of the headline metric: the 32-sequence ragged batch (nb = 32, context
    # U[512, 8192]); and, on request, the FP8-lm_head sweep
    if not args.no_extra and wl.name == DEFAULT_WORKLOAD:
        line["nb32"] = extra_workload("qwen3_8l_nb32_ragged", 100, 10, logits_on)
        torch.cuda.empty_cache()
    if args.sweep:
        line["sweep"] = {}
        for nb in (1, 4, 16, 64):
            name = f"fp8head_nb{nb}_ctx32768"
            line["sweep"][name] = extra_workload(name, 50 if nb < 64 else 20, 5, logits_on)
            torch.cuda.empty_cache()
    line["clocks"] = clk.summary()
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = oracle_timing(wl.name)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
