"""Seeded synthetic drafter weights and workloads.

Everything here is a pure function of (config, seed): the same bits come out on
every machine.  bf16 tensors are produced as raw bf16 bit patterns (uint16),
fp32 tensors as float32, tokens / page ids as int32.  Nothing in this file
performs the drafter's arithmetic; it only draws numbers.

Distributions (stand-ins for checkpoints and for the target model's tapped
hidden states, which are not available):
  * projection / embedding / lm_head weights: N(0, 0.02)
  * RMSNorm weights (ln_in, ln_post, q_norm, k_norm, hidden_norm, norm): 1 + N(0, 0.05)
  * tapped target hidden states: N(0, 1)
  * bonus tokens: uniform over the vocabulary
  * page tables: one random permutation of a shared page pool, cut into
    per-sequence runs (plus one spare page that no sequence owns).

bf16 normals are drawn as a 16-bit uniform integer u and mapped through the
table mu + sigma * Phi^-1((u + 0.5) / 65536), rounded to bf16 (round to nearest
even).  That is a 65536-level quantised normal: far finer than bf16 itself.
fp32 normals come straight from numpy's standard_normal.
"""
from __future__ import annotations

import math
import os
import statistics
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np

_CHUNK = 1 << 22


@dataclass(frozen=True)
class DrafterConfig:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_ff: int
    n_layers: int
    vocab: int
    n_taps: int
    target_hidden: int
    gamma: int = 16
    mask_token_id: int = 4
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    # YaRN: (factor, original_max_position_embeddings, beta_fast, beta_slow) or None
    yarn: Optional[Tuple[float, float, float, float]] = None
    sliding_window: int = 0
    layer_sliding: Tuple[bool, ...] = ()
    markov_rank: int = 0          # DSpark Markov head rank (0: none)
    dtype: str = "bf16"          # 'f32' or 'bf16': weights, activations and KV cache
    lm_head_dtype: str = "bf16"  # same as dtype, or 'fp8' (e4m3 + per-row fp32 scale)
    layer_weight_dtype: str = "bf16"  # 'bf16', or 'fp8': q/k/v/o/gate/up/down of every layer in e4m3
    page_size: int = 16

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def tap_dim(self) -> int:
        return self.n_taps * self.target_hidden

    def sliding(self, layer: int) -> bool:
        return bool(self.layer_sliding[layer]) if self.layer_sliding else False


# The five drafter shapes.  C2/C3/C5 share the 8-layer architecture.
_C2_ARCH = dict(hidden=2048, n_q_heads=32, n_kv_heads=4, head_dim=128, n_ff=6144,
                n_layers=8, vocab=151936, n_taps=5, target_hidden=2048)

CONFIGS: Dict[str, DrafterConfig] = {
    "tiny_fp32": DrafterConfig(
        name="tiny_fp32", hidden=256, n_q_heads=4, n_kv_heads=1, head_dim=64, n_ff=512,
        n_layers=1, vocab=2048, n_taps=3, target_hidden=256, dtype="f32", lm_head_dtype="f32"),
    "qwen3_8l_bf16": DrafterConfig(name="qwen3_8l_bf16", **_C2_ARCH),
    "wide_5l_yarn_bf16": DrafterConfig(
        name="wide_5l_yarn_bf16", hidden=5376, n_q_heads=64, n_kv_heads=8, head_dim=128,
        n_ff=10752, n_layers=5, vocab=262144, n_taps=6, target_hidden=5376,
        yarn=(32.0, 8192.0, 32.0, 1.0), sliding_window=2048,
        layer_sliding=(True, True, True, True, False)),
    "qwen3_8l_fp8head": DrafterConfig(name="qwen3_8l_fp8head", lm_head_dtype="fp8", **_C2_ARCH),
    # shapes the C ABI accepts beside the five above, each on a different kernel route:
    # the tiny fp32 drafter with an e4m3 lm_head (CUDA-core FP8 GEMV), a bf16 drafter with
    # 4 query heads per kv head (CUDA-core attention between tensor-core projections), and a
    # bf16 drafter with 8 query heads per kv head too small for the single-launch forward
    "tiny_fp32_fp8head": DrafterConfig(
        name="tiny_fp32_fp8head", hidden=256, n_q_heads=4, n_kv_heads=1, head_dim=64, n_ff=512,
        n_layers=1, vocab=2048, n_taps=3, target_hidden=256, dtype="f32", lm_head_dtype="fp8"),
    "small_gqa4_bf16": DrafterConfig(
        name="small_gqa4_bf16", hidden=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, n_ff=2048,
        n_layers=2, vocab=8192, n_taps=2, target_hidden=1024),
    # the FP8 drafter lane: every layer's seven projections and the lm_head in e4m3
    "qwen3_8l_fp8w": DrafterConfig(name="qwen3_8l_fp8w", lm_head_dtype="fp8", layer_weight_dtype="fp8",
                                   **_C2_ARCH),
    "tiny_fp32_fp8w": DrafterConfig(
        name="tiny_fp32_fp8w", hidden=256, n_q_heads=4, n_kv_heads=1, head_dim=64, n_ff=512,
        n_layers=1, vocab=2048, n_taps=3, target_hidden=256, dtype="f32", lm_head_dtype="f32",
        layer_weight_dtype="fp8"),
    # DSpark Markov head (rank 256, as in the pages' DSpark drafter) on the 8-layer drafter, and
    # a rank-32 head on the tiny fp32 drafter
    "qwen3_8l_markov": DrafterConfig(name="qwen3_8l_markov", markov_rank=256, **_C2_ARCH),
    "tiny_fp32_markov": DrafterConfig(
        name="tiny_fp32_markov", hidden=256, n_q_heads=4, n_kv_heads=1, head_dim=64, n_ff=512,
        n_layers=1, vocab=2048, n_taps=3, target_hidden=256, dtype="f32", lm_head_dtype="f32",
        markov_rank=32),
    "small_gqa8_bf16": DrafterConfig(
        name="small_gqa8_bf16", hidden=1024, n_q_heads=8, n_kv_heads=1, head_dim=128, n_ff=2048,
        n_layers=2, vocab=8192, n_taps=2, target_hidden=1024),
}


@dataclass
class Workload:
    """One batch of nb sequences to draft for, with their paged context."""
    cfg: DrafterConfig
    name: str
    seed: int
    ctx_lens: np.ndarray          # int32 [nb]
    bonus: np.ndarray             # int32 [nb]
    page_tables: np.ndarray       # int32 [nb, max_pages_per_seq], -1 past each run
    num_pages: int
    taps_rows: int                # R: rows in the shared tap table
    tap_offsets: np.ndarray       # int64 [nb]: row i of sequence s is table row (off_s + i) % R
    _taps_table: Optional[np.ndarray] = field(default=None, repr=False)

    @property
    def nb(self) -> int:
        return int(self.ctx_lens.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.page_tables.shape[1])

    @property
    def max_ctx_len(self) -> int:
        return int(self.ctx_lens.max())

    def ctx_positions(self, s: int, first: int, n: int) -> np.ndarray:
        """Absolute positions of context rows first..first+n-1 (row i sits at position i)."""
        del s
        return np.arange(first, first + n, dtype=np.int32)


# ----------------------------------------------------------------------------- drawing


def _tensor_key(name: str) -> int:
    return zlib.crc32(name.encode("utf-8"))


_NORMAL_TABLE: Optional[np.ndarray] = None


def _normal_table() -> np.ndarray:
    global _NORMAL_TABLE
    if _NORMAL_TABLE is None:
        nd = statistics.NormalDist()
        _NORMAL_TABLE = np.array([nd.inv_cdf((u + 0.5) / 65536.0) for u in range(65536)],
                                 dtype=np.float64)
    return _NORMAL_TABLE


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + r) >> 16).astype(np.uint16)


_BF16_TABLES: Dict[Tuple[float, float], np.ndarray] = {}


def _bf16_table(mu: float, sigma: float) -> np.ndarray:
    key = (mu, sigma)
    if key not in _BF16_TABLES:
        _BF16_TABLES[key] = _f32_to_bf16_bits((mu + sigma * _normal_table()).astype(np.float32))
    return _BF16_TABLES[key]


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def draw(seed: int, name: str, shape, mu: float, sigma: float, dtype: str) -> np.ndarray:
    """N(mu, sigma) tensor of `shape` as bf16 bits (uint16) or float32, chunked by a
    counter so the result does not depend on the thread count."""
    n = int(np.prod(shape))
    key = _tensor_key(name)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    if dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
        tab = _bf16_table(mu, sigma)

        def job(c):
            s, e = c * _CHUNK, min(n, (c + 1) * _CHUNK)
            g = np.random.Generator(np.random.PCG64([seed, key, c]))
            np.take(tab, g.integers(0, 65536, size=e - s, dtype=np.uint16), out=out[s:e])
    elif dtype == "f32":
        out = np.empty(n, dtype=np.float32)

        def job(c):
            s, e = c * _CHUNK, min(n, (c + 1) * _CHUNK)
            g = np.random.Generator(np.random.PCG64([seed, key, c]))
            out[s:e] = (mu + sigma * g.standard_normal(e - s)).astype(np.float32)
    else:
        raise ValueError(dtype)
    if nchunks == 1:
        job(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(job, range(nchunks)))
    return out.reshape(shape)


# ----------------------------------------------------------------------------- weights


class Weights:
    """Lazily drawn drafter weights (HF layout: Linear weights are [out, in] row-major).

    `get(name)` draws a tensor on first use; `keep=False` draws without caching, so a
    caller can stream tensors to the device without holding all of them on the host.
    Names: fc, hidden_norm, norm, embed, lm_head, and L{l}.{ln_in, wq, wk, wv, q_norm,
    k_norm, wo, ln_post, w_gate, w_up, w_down}.
    """

    LAYER_TENSORS = ("ln_in", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ln_post",
                     "w_gate", "w_up", "w_down")

    def __init__(self, cfg: DrafterConfig, seed: int):
        self.cfg = cfg
        self.seed = seed
        self._cache: Dict[str, np.ndarray] = {}

    def spec(self, name: str):
        c = self.cfg
        H, F = c.hidden, c.n_ff
        if name == "fc":
            return (H, c.tap_dim), 0.0, 0.02
        if name in ("hidden_norm", "norm"):
            return (H,), 1.0, 0.05
        if name in ("embed", "lm_head"):
            return (c.vocab, H), 0.0, 0.02
        # DSpark Markov head: a unit-variance previous-token table and a projection scaled so
        # the bias w2 . w1[prev] has about unit spread, the spread of the logits themselves
        if name == "markov_w1":
            return (c.vocab, c.markov_rank), 0.0, 1.0
        if name == "markov_w2":
            return (c.vocab, c.markov_rank), 0.0, 1.0 / math.sqrt(c.markov_rank)
        layer, t = name.split(".")
        assert layer[0] == "L" and 0 <= int(layer[1:]) < c.n_layers, name
        return {
            "ln_in": ((H,), 1.0, 0.05),
            "ln_post": ((H,), 1.0, 0.05),
            "q_norm": ((c.head_dim,), 1.0, 0.05),
            "k_norm": ((c.head_dim,), 1.0, 0.05),
            "wq": ((c.q_dim, H), 0.0, 0.02),
            "wk": ((c.kv_dim, H), 0.0, 0.02),
            "wv": ((c.kv_dim, H), 0.0, 0.02),
            "wo": ((H, c.q_dim), 0.0, 0.02),
            "w_gate": ((F, H), 0.0, 0.02),
            "w_up": ((F, H), 0.0, 0.02),
            "w_down": ((H, F), 0.0, 0.02),
        }[t]

    def names(self) -> List[str]:
        out = ["fc", "hidden_norm", "norm", "embed", "lm_head"]
        if self.cfg.markov_rank > 0:
            out += ["markov_w1", "markov_w2"]
        for l in range(self.cfg.n_layers):
            out += [f"L{l}.{t}" for t in self.LAYER_TENSORS]
        return out

    def get(self, name: str, keep: bool = True) -> np.ndarray:
        if name in self._cache:
            return self._cache[name]
        shape, mu, sigma = self.spec(name)
        a = draw(self.seed, "w/" + name, shape, mu, sigma, self.cfg.dtype)
        if keep:
            self._cache[name] = a
        return a

    def drop(self, name: str) -> None:
        self._cache.pop(name, None)

    def layer(self, l: int) -> Dict[str, np.ndarray]:
        return {t: self.get(f"L{l}.{t}") for t in self.LAYER_TENSORS}


def make_weights(cfg: DrafterConfig, seed: int) -> Weights:
    return Weights(cfg, seed)


# ----------------------------------------------------------------------------- workloads


def make_workload(cfg: DrafterConfig, seed: int, ctx_lens, name: str = "",
                  taps_rows: Optional[int] = None, bonus=None,
                  extra_pages_per_seq: int = 0) -> Workload:
    """Batch of len(ctx_lens) sequences.  Each sequence gets ceil((c+gamma)/16) pages
    (room for its context plus the transient gamma block) + `extra_pages_per_seq`,
    drawn from one random permutation of a shared pool with one spare page."""
    ctx = np.asarray(ctx_lens, dtype=np.int32).reshape(-1)
    nb = ctx.shape[0]
    ps, g = cfg.page_size, cfg.gamma
    rng = np.random.Generator(np.random.PCG64([seed, _tensor_key("workload")]))
    need = [(int(c) + g + ps - 1) // ps + extra_pages_per_seq for c in ctx]
    num_pages = int(sum(need)) + 1
    perm = rng.permutation(num_pages).astype(np.int32)
    mpps = max(need)
    pt = np.full((nb, mpps), -1, dtype=np.int32)
    at = 0
    for s in range(nb):
        pt[s, :need[s]] = perm[at:at + need[s]]
        at += need[s]
    if bonus is None:
        bonus = rng.integers(0, cfg.vocab, size=nb, dtype=np.int64)
    bonus = np.asarray(bonus, dtype=np.int32).reshape(nb)
    R = int(taps_rows) if taps_rows else int(min(max(int(ctx.max()), 1), 16384))
    offs = (np.zeros(nb, dtype=np.int64) if R >= int(ctx.max()) and nb == 1
            else rng.integers(0, R, size=nb, dtype=np.int64))
    return Workload(cfg=cfg, name=name or cfg.name, seed=seed, ctx_lens=ctx, bonus=bonus,
                    page_tables=pt, num_pages=num_pages, taps_rows=R, tap_offsets=offs)


def taps_table(wl: Workload) -> np.ndarray:
    if wl._taps_table is None:
        wl._taps_table = draw(wl.seed, "taps", (wl.taps_rows, wl.cfg.tap_dim), 0.0, 1.0,
                              wl.cfg.dtype)
    return wl._taps_table


def workload_taps(wl: Workload, s: int, first: int, n: int) -> np.ndarray:
    """Tapped target hidden states for context rows first..first+n-1 of sequence s,
    [n, n_taps * target_hidden], taps concatenated in target_layer_ids order."""
    idx = (int(wl.tap_offsets[s]) + np.arange(first, first + n, dtype=np.int64)) % wl.taps_rows
    return taps_table(wl)[idx]


def _c3_ctx(seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64([seed, _tensor_key("c3_ctx")]))
    return rng.integers(512, 8192 + 1, size=32, dtype=np.int64).astype(np.int32)


# Named workloads at full size (the bench's and the full-size parity tests' inputs).
WORKLOADS = {
    "tiny_fp32_nb1_ctx64": lambda: make_workload(CONFIGS["tiny_fp32"], 1, [64]),
    "qwen3_8l_nb1_ctx4096": lambda: make_workload(CONFIGS["qwen3_8l_bf16"], 2, [4096]),
    "qwen3_8l_nb32_ragged": lambda: make_workload(CONFIGS["qwen3_8l_bf16"], 3, _c3_ctx(3)),
    "wide_5l_yarn_nb1_ctx16384": lambda: make_workload(CONFIGS["wide_5l_yarn_bf16"], 4, [16384]),
    "fp8head_nb1_ctx32768": lambda: make_workload(CONFIGS["qwen3_8l_fp8head"], 5, [32768],
                                                  taps_rows=8192),
    "fp8head_nb4_ctx32768": lambda: make_workload(CONFIGS["qwen3_8l_fp8head"], 5, [32768] * 4,
                                                  taps_rows=8192),
    "fp8head_nb16_ctx32768": lambda: make_workload(CONFIGS["qwen3_8l_fp8head"], 5, [32768] * 16,
                                                   taps_rows=8192),
    "fp8head_nb64_ctx32768": lambda: make_workload(CONFIGS["qwen3_8l_fp8head"], 5, [32768] * 64,
                                                   taps_rows=8192),
    # the FP8 drafter lane (layer weights and lm_head in e4m3) on the headline shape
    "fp8w_nb1_ctx4096": lambda: make_workload(CONFIGS["qwen3_8l_fp8w"], 6, [4096]),
    "fp8w_nb32_ragged": lambda: make_workload(CONFIGS["qwen3_8l_fp8w"], 7, _c3_ctx(3)),
}
