"""Shared plumbing for the GPU tests: build a drafter from a seeded workload, fill its
context K/V through the library, run the oracle on sampled bands, compare."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from synth import make_weights, workload_taps
from synth.inputs import taps_table
from synth.torch_io import from_torch, to_torch, upload_weights

TOL = {  # relative max error max|gpu - oracle| / max|oracle| per tensor, and argmax margin
    "f32": dict(hidden=1e-4, logits=1e-4, margin=1e-3),
    "bf16": dict(hidden=2e-2, logits=3e-2, margin=0.1),
}


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class DevView:
    """Zero-copy torch view of a raw device pointer (the library-owned K/V pool)."""

    def __init__(self, ptr: int, n: int, typestr: str):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False), "version": 3}


def pool_view(drafter) -> torch.Tensor:
    ptr, nbytes, strides = drafter.kv_layout()
    esz = strides[5]
    t = torch.as_tensor(DevView(ptr, nbytes // esz, "<f4" if esz == 4 else "<u2"), device="cuda")
    return t if esz == 4 else t.view(torch.bfloat16)


def pool_rows(drafter, layer: int, kv: int, head: int, pages: np.ndarray, offs: np.ndarray) -> np.ndarray:
    """Read rows (page, offset) of a K (kv=0) or V (kv=1) head out of the pool -> [n, hd]."""
    _, _, st = drafter.kv_layout()
    hd = drafter.cfg.head_dim
    pool = pool_view(drafter)
    j = torch.as_tensor(offs, device="cuda", dtype=torch.int64)[:, None]
    d = torch.arange(hd, device="cuda", dtype=torch.int64)[None, :]
    if kv == 0:
        inner = ((j // 8) * (hd // 8) + d // 8) * 64 + (j % 8) * 8 + d % 8
    else:
        inner = ((d // 8) * 2 + j // 8) * 64 + (d % 8) * 8 + j % 8
    base = (layer * st[0] + torch.as_tensor(pages, device="cuda", dtype=torch.int64)[:, None] * st[1]
            + kv * st[2] + head * st[3])
    return as_f64(pool[base + inner])


class Rig:
    """Drafter + device inputs for one workload, context already written."""

    def __init__(self, wl, max_write_rows: int = 4096, max_batch=None, write=True):
        from block_diffusion_drafter_forward_gb300 import Drafter

        self.wl = wl
        self.cfg = wl.cfg
        self.W = make_weights(wl.cfg, wl.seed)
        self.tensors = upload_weights(self.W)
        self.drafter = Drafter(wl.cfg, self.tensors, num_pages=wl.num_pages, max_batch=max_batch or wl.nb,
                               max_pages_per_seq=wl.max_pages_per_seq, max_write_rows=max_write_rows)
        self.bonus = to_torch(wl.bonus, "i32")
        self.ctx_lens = to_torch(wl.ctx_lens, "i32")
        self.page_tables = to_torch(wl.page_tables, "i32")
        if write:
            self.write_all()

    def taps_dev(self, s: int, first: int, n: int) -> torch.Tensor:
        if not hasattr(self, "_table"):
            self._table = to_torch(taps_table(self.wl), self.cfg.dtype)
        idx = (int(self.wl.tap_offsets[s]) + torch.arange(first, first + n, device="cuda")) % self.wl.taps_rows
        return self._table[idx].contiguous()

    def write_all(self, chunk: int = 0) -> None:
        for s in range(self.wl.nb):
            c = int(self.wl.ctx_lens[s])
            step = chunk or c
            for first in range(0, c, max(step, 1)):
                n = min(step, c - first)
                pos = to_torch(self.wl.ctx_positions(s, first, n), "i32")
                self.drafter.write_ctx_kv(self.taps_dev(s, first, n), pos, self.page_tables[s], first)

    def propose(self, logits=True, hidden=True):
        nb, g = self.wl.nb, self.cfg.gamma
        dt = torch.float32 if self.cfg.dtype == "f32" else torch.bfloat16
        z = torch.empty((nb * g, self.cfg.vocab), dtype=dt, device="cuda") if logits else None
        h = torch.empty((nb * g, self.cfg.hidden), dtype=dt, device="cuda") if hidden else None
        d = self.drafter.propose(self.bonus, self.ctx_lens, self.page_tables, self.wl.max_ctx_len, logits=z,
                                 hidden=h)
        torch.cuda.synchronize()
        return d, z, h

    def oracle_band(self, s: int, oracle):
        c = int(self.wl.ctx_lens[s])
        taps = workload_taps(self.wl, s, 0, c)
        return oracle.run_sequence(taps, self.wl.ctx_positions(s, 0, c), int(self.wl.bonus[s]))


def check_band(rig, s, ref, drafts, z, h, tol):
    """Compare band s of the GPU outputs with the oracle's; returns a dict of errors."""
    g = rig.cfg.gamma
    hs = as_f64(h[s * g:(s + 1) * g])
    zs = as_f64(z[s * g:(s + 1) * g]) if z is not None else None
    out = {"hidden": rel_err(hs, ref["h"])}
    if zs is not None:
        out["logits"] = rel_err(zs, ref["logits"])
    dt = drafts[s].cpu().numpy().astype(np.int64)
    sure = ref["margin"] > tol["margin"]
    out["n_sure"] = int(sure.sum())
    out["mismatch"] = int((dt[sure] != ref["tokens"][sure]).sum())
    log = os.environ.get("DFLASH_PARITY_LOG")
    if log:
        with open(log, "a") as fh:
            fh.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", ""), "band": s, **out}) + "\n")
    assert out["hidden"] <= tol["hidden"], (s, out)
    if zs is not None:
        assert out["logits"] <= tol["logits"], (s, out)
    assert out["mismatch"] == 0, (s, out, dt, ref["tokens"], ref["margin"])
    return out
