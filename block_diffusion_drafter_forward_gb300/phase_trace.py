"""Per-phase timeline of the single-launch forward (one sequence).

Builds the library with DFLASH_PHASE_TRACE=1 into its own file, runs the 8-layer bf16 drafter
at nb = 1 (default context 4096) on cuda:0, and prints, for every phase of the last launch,
when the CTAs passed its barrier, committed their last MMA, had their split-K partials and
arrived, as median / max over CTAs in microseconds after the previous phase's last arrival.

  python -m block_diffusion_drafter_forward_gb300.phase_trace [--ctx N] [--raw FILE]

The stamps are %globaltimer reads (nanoseconds); the stamping adds a few percent to the step.
"""
from __future__ import annotations

import argparse
import os
import sys
import tempfile

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
TRACE_LIB = os.path.join(PKG, "libdflash_trace.so")
SLOTS = ("barrier", "act", "w_first", "mma_last", "acc", "counted", "landed", "arrive", "epi_done", "contrib",
         "reduced", "epi_body", "fenced")


def phase_names(L: int):
    names = ["embed"]
    for l in range(L):
        names += [f"L{l} qkv", f"L{l} attention", f"L{l} combine", f"L{l} o_proj", f"L{l} gate/up", f"L{l} down"]
    return names + ["lm_head"]


def read_trace(path: str):
    with open(path, "rb") as fh:
        G, P, S = np.frombuffer(fh.read(12), dtype=np.int32)
        t = np.frombuffer(fh.read(), dtype=np.uint64).astype(np.int64).reshape(G, P, S)
    return t


def table(t: np.ndarray, L: int):
    """Rows of (phase, duration, {slot: (median, max)}) in us, each relative to the previous
    phase's last arrival (the first phase: to the earliest stamp)."""
    G, P, S = t.shape
    names = phase_names(L)
    valid = t > 0
    t0 = int(t[valid].min())
    prev = t0
    rows = []
    for ph in range(P):
        arr = t[:, ph, SLOTS.index("arrive")]
        last = int(arr[arr > 0].max()) if (arr > 0).any() else prev
        cols = {}
        for k, name in enumerate(SLOTS[:S]):  # older traces hold fewer slots
            v = t[:, ph, k]
            v = v[v > 0]
            if v.size:
                cols[name] = (float(np.median(v) - prev) / 1e3, float(v.max() - prev) / 1e3)
        rows.append((names[ph] if ph < len(names) else str(ph), (last - prev) / 1e3, cols))
        prev = last
    return rows, (prev - t0) / 1e3


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--ctx", type=int, default=4096)
    ap.add_argument("--raw", default=None, help="keep the raw stamps in this file")
    args = ap.parse_args()
    sys.path.insert(0, ROOT)
    from block_diffusion_drafter_forward_gb300 import build

    build.build(verbose=True, defines=("DFLASH_PHASE_TRACE=1",), lib_path=TRACE_LIB,
                build_dir=os.path.join(ROOT, "_build", "trace"))
    from block_diffusion_drafter_forward_gb300 import _lib

    _lib.load(TRACE_LIB)
    import torch

    from block_diffusion_drafter_forward_gb300 import Drafter
    from synth import CONFIGS, make_weights, make_workload
    from synth.inputs import taps_table
    from synth.torch_io import to_torch, upload_weights

    torch.cuda.set_device(0)
    cfg = CONFIGS["qwen3_8l_bf16"]
    wl = make_workload(cfg, 2, [args.ctx])
    d = Drafter(cfg, upload_weights(make_weights(cfg, wl.seed)), num_pages=wl.num_pages, max_batch=1,
                max_pages_per_seq=wl.max_pages_per_seq)
    assert d.persistent, "the single-launch forward is not available on this device"
    table_rows = to_torch(taps_table(wl), cfg.dtype)
    pt = to_torch(wl.page_tables, "i32")
    c = args.ctx
    idx = (int(wl.tap_offsets[0]) + torch.arange(c, device="cuda")) % wl.taps_rows
    d.write_ctx_kv(table_rows[idx].contiguous(), to_torch(wl.ctx_positions(0, 0, c), "i32"), pt[0], 0)
    bonus, ctx = to_torch(wl.bonus, "i32"), to_torch(wl.ctx_lens, "i32")
    logits = torch.empty((16, cfg.vocab), dtype=torch.bfloat16, device="cuda")
    drafts = torch.empty((1, 15), dtype=torch.int32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(5):
        d.propose(bonus, ctx, pt, c, drafts=drafts, logits=logits)
    flush.zero_()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    d.propose(bonus, ctx, pt, c, drafts=drafts, logits=logits)
    b.record()
    torch.cuda.synchronize()
    path = args.raw or os.path.join(tempfile.mkdtemp(), "trace.bin")
    os.environ["DFLASH_TRACE_FILE"] = path
    assert d.device_status() == 0
    t = read_trace(path)
    rows, total = table(t, cfg.n_layers)
    print(f"step {a.elapsed_time(b) * 1e3:.1f} us (events), {total:.1f} us from first to last stamp")
    hdr = f"{'phase':14s} {'dur':>6s}  " + "  ".join(f"{s:>13s}" for s in SLOTS)
    print(hdr)
    for name, dur, cols in rows:
        cells = "  ".join(f"{cols[s][0]:6.1f}/{cols[s][1]:6.1f}" if s in cols else f"{'-':>13s}" for s in SLOTS)
        print(f"{name:14s} {dur:6.1f}  {cells}")
    d.close()


if __name__ == "__main__":
    main()
