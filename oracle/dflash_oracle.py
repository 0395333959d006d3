"""CPU oracle of the DFlash drafter gamma-block forward.  TEST INFRASTRUCTURE ONLY.

Only the tests, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg may
import this module; the product path never does.  It shares no code with the CUDA
library: it reads the same seeded inputs (bf16 bit patterns / fp32 values) and
computes everything in float64 numpy, one plain step after another, with no
blocking, fusion or reordering beyond the definition.

What it follows (page = the source listing it is read from):
  * memra-engine `dflash.rs` (docs.rs, memra-engine 0.94.0):
      - `DflashDraft::ctx_features`: f = hidden_norm(fc(taps))
      - `DflashDraft::ingest_ctx`: per layer K = rope(k_norm(Wk f)) (* mscale), V = Wv f
      - `DflashDraft::forward_round` / `forward_block`: the per-layer block forward
      - `DflashDraft::load`, YaRN block: per-dim divisors and mscale = 0.1 ln(factor) + 1
      - `generate_spec_dflash`, draft step: block = [last, MASK x (b-1)], positions
        start..start+b-1, drafts = argmax(lm_head(h rows 1..b-1))
  * spark_model `dflash_head/from_weights.rs` (Atlas docs):
      - kernel table comment: vanilla RMSNorm out = x * w / RMS(x)
      - inv_freq table block: plain inv_freq = theta^(-2j/d); YaRN ramp with the
        +0.001 guard when high == low
      - paged pool block: BF16 cache, 16 tokens per page
      - FP8 "Phase G" block: weight-only e4m3 with a per-output-row fp32 scale
  * spark_model `layers/dflash_head.rs` (Atlas docs): batched propose stacks
    sequences seq-major, gamma rows each; row 0 of each band is the anchor echo.
  * DSpark Markov head (memra `dflash.rs` draft step, Markov chain block; Atlas
    `dflash_head.rs` DSpark fields): `markov_chain` below.

Readings where the pages leave a step open (each is also listed in the design notes):
  eps inside the square root; NeoX rotate-half RoPE over the full head_dim;
  GQA head map g = h // (nh / nkv); sliding-window mask iff p_q - p_k >= W;
  argmax ties go to the lowest vocabulary index; FP8 scale = fp32(rowmax|w|) / 448
  with e4m3 round-to-nearest-even and saturation to +-448.

Parity: every function below is pinned by tests/test_oracle_pins.py against closed
forms, brute force, invariants or independent library routines.  The composition
(`Oracle.forward_block` end to end) has no external value to compare with and is
"parity unpinned" beyond the composition of its pinned steps.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# ----------------------------------------------------------------------------- dtypes


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_to_f64(a)
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------- elementwise


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Vanilla RMSNorm over the last axis: x * w / sqrt(mean(x^2) + eps)
    (from_weights.rs, kernel table: `rms_norm_vanilla`, not the 1+w form)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)) (dflash.rs forward_round: `silu_mul`)."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


# ----------------------------------------------------------------------------- RoPE


def rope_inv_freq(head_dim: int, theta: float,
                  yarn: Optional[Tuple[float, float, float, float]] = None
                  ) -> Tuple[np.ndarray, float]:
    """Per-pair inverse frequencies [head_dim/2] and the post-rotation scale.

    Plain: inv_freq_j = theta^(-2j/d) (from_weights.rs inv_freq table).
    YaRN (factor, orig, beta_fast, beta_slow) (dflash.rs `load`, YaRN block;
    from_weights.rs YaRN arm):
        corr(r) = d ln(orig / (2 pi r)) / (2 ln theta)
        low = max(floor(corr(beta_fast)), 0), high = min(ceil(corr(beta_slow)), d - 1)
        ramp_j = clamp((j - low) / (high - low), 0, 1)   (high - low + 0.001 if equal)
        extrapolation share ex_j = 1 - ramp_j
        inv_freq_j = (base_j / factor) (1 - ex_j) + base_j ex_j,  base_j = theta^(-2j/d)
        mscale = 0.1 ln(factor) + 1, applied to q and k after the rotation.
    """
    d = float(head_dim)
    half = head_dim // 2
    j = np.arange(half, dtype=np.float64)
    base = theta ** (-2.0 * j / d)
    if yarn is None:
        return base, 1.0
    factor, orig, beta_fast, beta_slow = (float(v) for v in yarn)

    def corr(r: float) -> float:
        return d * math.log(orig / (r * 2.0 * math.pi)) / (2.0 * math.log(theta))

    low = max(math.floor(corr(beta_fast)), 0.0)
    high = min(math.ceil(corr(beta_slow)), d - 1.0)
    denom = (high - low) if abs(high - low) >= 1e-6 else (high - low + 0.001)
    ramp = np.clip((j - low) / denom, 0.0, 1.0)
    ex = 1.0 - ramp
    inv = (base / factor) * (1.0 - ex) + base * ex
    return inv, 0.1 * math.log(factor) + 1.0


def yarn_divisors(head_dim: int, theta: float, yarn) -> np.ndarray:
    """ff_j = base_j / inv_freq_j, the per-dim divisors memra uploads for `rope_neox_ff`."""
    base, _ = rope_inv_freq(head_dim, theta, None)
    inv, _ = rope_inv_freq(head_dim, theta, yarn)
    return base / inv


def rope(x: np.ndarray, pos: np.ndarray, inv_freq: np.ndarray, mscale: float = 1.0) -> np.ndarray:
    """NeoX rotate-half RoPE over the last axis (length d), positions broadcast over the
    leading axis: for j < d/2, with a = x_j, b = x_{j+d/2}, t = pos * inv_freq_j:
        out_j = a cos t - b sin t,  out_{j+d/2} = b cos t + a sin t;  then * mscale.
    x: [n, ..., d], pos: [n]."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    t = np.asarray(pos, dtype=np.float64).reshape((-1,) + (1,) * (x.ndim - 1)) * inv_freq
    c, s = np.cos(t), np.sin(t)
    a, b = x[..., :half], x[..., half:]
    out = np.concatenate([a * c - b * s, b * c + a * s], axis=-1)
    return out * mscale


# ----------------------------------------------------------------------------- attention


def block_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray,
                    k_pos: np.ndarray, window: int = 0) -> np.ndarray:
    """Non-causal GQA attention of the block queries over all keys
    (dflash.rs forward_round: `sdpa_naive(..., causal=false)`), explicit softmax.

    q [nq, nh, d], k/v [nk, nkv, d], positions int.  Query head h uses kv head
    h // (nh / nkv).  Score scale 1/sqrt(d).  With window W > 0 a key is masked for a
    query iff q_pos - k_pos >= W (keys at or after the query are never masked).
    Returns [nq, nh, d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, nh, d = q.shape
    nkv = k.shape[1]
    group = nh // nkv
    kh = np.repeat(k, group, axis=1)          # [nk, nh, d]: head h -> kv head h // group
    vh = np.repeat(v, group, axis=1)
    s = np.einsum("qhd,khd->hqk", q, kh) / math.sqrt(d)
    if window and window > 0:
        rel = np.asarray(q_pos, dtype=np.int64)[:, None] - np.asarray(k_pos, dtype=np.int64)[None, :]
        s = np.where((rel >= window)[None, :, :], -np.inf, s)
    m = np.max(s, axis=-1, keepdims=True)
    p = np.exp(s - m)
    p = p / np.sum(p, axis=-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", p, vh)


# ----------------------------------------------------------------------------- paging


def page_slots(page_table: np.ndarray, first: int, n: int, page_size: int = 16) -> np.ndarray:
    """Slot of logical rows first..first+n-1: page_table[i // ps] * ps + i % ps
    (from_weights.rs / dflash_head.rs: `fill_slots_from_block_table`). int64."""
    i = np.arange(first, first + n, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int64)
    return pt[i // page_size] * page_size + (i % page_size)


class PagedPool:
    """Paged K/V store: one pool of pages per layer, `page_size` rows per page.
    Logical row i of a sequence lives in page page_table[i // ps] at offset i % ps."""

    def __init__(self, n_layers: int, num_pages: int, n_kv: int, head_dim: int, page_size: int = 16):
        self.ps = page_size
        self.k = np.full((n_layers, num_pages * page_size, n_kv, head_dim), np.nan)
        self.v = np.full((n_layers, num_pages * page_size, n_kv, head_dim), np.nan)

    def store(self, layer: int, page_table, first: int, k: np.ndarray, v: np.ndarray) -> None:
        sl = page_slots(page_table, first, k.shape[0], self.ps)
        self.k[layer, sl] = k
        self.v[layer, sl] = v

    def gather(self, layer: int, page_table, n: int) -> Tuple[np.ndarray, np.ndarray]:
        sl = page_slots(page_table, 0, n, self.ps)
        return self.k[layer, sl], self.v[layer, sl]


# ----------------------------------------------------------------------------- FP8 e4m3


E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 ('fn': no infinities, S.1111.111 is NaN), bias 7.
    normal: (-1)^s 2^(e-7) (1 + m/8); subnormal (e == 0): (-1)^s 2^-6 (m/8)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64)))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return s * val


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even encode of float values into E4M3, saturating finite
    values (and +-inf) to +-448; NaN -> 0x7F.  Works on the exact float64 value."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.int64)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, 1e30))
    # subnormal range |x| < 2^-6: code = rint(|x| / 2^-9) (0..8; 8 is the smallest normal)
    sub = np.rint(np.ldexp(np.minimum(a, 2.0 ** -6), 9)).astype(np.int64)
    # normal range: |x| = 2^e * f, f in [1, 2)
    mant, ex = np.frexp(a)              # a = mant * 2^ex, mant in [0.5, 1)
    e = ex.astype(np.int64) - 1
    f = mant * 2.0
    q = np.rint((f - 1.0) * 8.0).astype(np.int64)
    carry = q == 8
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 0, q)
    norm_code = ((e + 7) << 3) | q
    norm_code = np.where(e > 8, 0x7E, norm_code)
    norm_code = np.minimum(norm_code, 0x7E)        # 0x7F would be NaN: saturate to 448
    code = np.where(a < 2.0 ** -6, sub, norm_code)
    code = np.where(nan, 0x7F, code | sign)
    return code.astype(np.uint8)


def fp8_quantize_rows(w: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-output-row e4m3 quantisation (from_weights.rs FP8 block: weight-only FP8
    with a per-row fp32 scale; scale rule rowmax/448):
        scale_v = fp32(max_k |w_vk|) / 448          (fp32 IEEE division)
        q_vk    = e4m3_rne_satfinite(fp32(w_vk / scale_v))
    A zero row gets scale 1.  w: float32 array [V, K].  Returns (uint8 [V, K], f32 [V])."""
    w = np.asarray(w, dtype=np.float32)
    rowmax = np.max(np.abs(w), axis=1)
    scale = (rowmax / np.float32(E4M3_MAX)).astype(np.float32)
    scale = np.where(rowmax == 0, np.float32(1.0), scale).astype(np.float32)
    ratio = (w / scale[:, None]).astype(np.float32)
    return e4m3_encode(ratio), scale


# ----------------------------------------------------------------------------- DSpark Markov chain


def markov_chain(z: np.ndarray, bonus: int, w1: np.ndarray, w2: np.ndarray):
    """Semi-autoregressive Markov fix-up of one band's draft logits (memra-engine dflash.rs,
    draft step of generate_spec_dflash, the SEMI-AR MARKOV CHAIN block; Atlas dflash_head.rs,
    DSpark heads: markov_w1 [V, rank] prev-token table, markov_w2 [V, rank] = Linear(rank, V)).

    z: [b-1, V] logits of block rows 1..b-1.  Left to right, starting from the bonus token:
        chain_0 = bonus
        for k = 0 .. b-2:
            f      = w1[chain_k]                       (rank-vector of the previous token)
            z_k   += w2 @ f                            (bias_v = sum_j w2[v, j] f_j)
            chain_{k+1} = argmax_v z_k                 (ties -> lowest id)
    Returns (adjusted logits [b-1, V], tokens chain_1..chain_{b-1} [b-1], top-1 minus top-2
    margins of the adjusted rows [b-1])."""
    z = np.array(z, dtype=np.float64, copy=True)
    w1 = np.asarray(w1, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    prev = int(bonus)
    tokens = np.empty(z.shape[0], dtype=np.int64)
    margins = np.empty(z.shape[0], dtype=np.float64)
    for k in range(z.shape[0]):
        z[k] += w2 @ w1[prev]
        idx, margin = Oracle.argmax_rows(z[k:k + 1])
        prev = int(idx[0])
        tokens[k] = prev
        margins[k] = margin[0]
    return z, tokens, margins


# ----------------------------------------------------------------------------- the drafter


class Oracle:
    """The drafter forward written out.  `weights.get(name, keep)` returns the raw
    tensors (bf16 bits or fp32) named as in synth.inputs.Weights; `keep` says whether
    the source may cache it."""

    def __init__(self, cfg, weights, cache: bool = False):
        self.cfg = cfg
        self.w = weights
        self.cache = cache
        self._f64: Dict[str, np.ndarray] = {}
        self.inv_freq, self.mscale = rope_inv_freq(cfg.head_dim, cfg.rope_theta, cfg.yarn)
        self._fp8 = None

    def W(self, name: str) -> np.ndarray:
        if name in self._f64:
            return self._f64[name]
        a = to_f64(self.w.get(name, keep=self.cache), self.cfg.dtype)
        if self.cache:
            self._f64[name] = a
        return a

    # the seven projections of a layer that the FP8 drafter lane stores in e4m3
    FP8_LAYER = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")

    def Wproj(self, l: int, t: str) -> np.ndarray:
        """Projection weight of layer l as the block forward uses it: the stored weight, or, with
        FP8 layer weights (from_weights.rs Phase G: q/k/v/o/gate/up/down quantised to e4m3 with a
        per-output-row fp32 scale), its decoded codes times the row scales."""
        name = f"L{l}.{t}"
        if getattr(self.cfg, "layer_weight_dtype", "bf16") != "fp8" or t not in self.FP8_LAYER:
            return self.W(name)
        key = name + "#fp8"
        if key in self._f64:
            return self._f64[key]
        codes, scale = fp8_quantize_rows(self.W(name).astype(np.float32))
        a = e4m3_decode(codes) * scale.astype(np.float64)[:, None]
        if self.cache:
            self._f64[key] = a
        return a

    # ---- context path: dflash.rs ctx_features + ingest_ctx

    def ctx_features(self, taps: np.ndarray) -> np.ndarray:
        """f = hidden_norm(fc(taps)); taps [n, n_taps * Ht] (raw) -> [n, H]."""
        t = to_f64(taps, self.cfg.dtype)
        y = t @ self.W("fc").T
        return rms_norm(y, self.W("hidden_norm"), self.cfg.rms_eps)

    def ctx_kv_layer(self, l: int, f: np.ndarray, pos: np.ndarray):
        """Layer l's cached context K (k_norm per head, RoPE at pos, * mscale) and raw V."""
        c = self.cfg
        n = f.shape[0]
        k = (f @ self.W(f"L{l}.wk").T).reshape(n, c.n_kv_heads, c.head_dim)
        v = (f @ self.W(f"L{l}.wv").T).reshape(n, c.n_kv_heads, c.head_dim)
        k = rms_norm(k, self.W(f"L{l}.k_norm"), c.rms_eps)
        k = rope(k, pos, self.inv_freq, self.mscale)
        return k, v

    def ctx_kv(self, f: np.ndarray, pos: np.ndarray):
        """K, V for every layer: lists of [n, nkv, hd]."""
        ks, vs = [], []
        for l in range(self.cfg.n_layers):
            k, v = self.ctx_kv_layer(l, f, pos)
            ks.append(k)
            vs.append(v)
        return ks, vs

    # ---- block path: dflash.rs forward_round + final norm

    def block_tokens(self, bonus: int, width: Optional[int] = None) -> np.ndarray:
        """[bonus, mask x (b - 1)], b = width (default gamma)."""
        g = self.cfg.gamma if width is None else int(width)
        tok = np.full(g, self.cfg.mask_token_id, dtype=np.int64)
        tok[0] = bonus
        return tok

    def embed_rows(self, tokens: np.ndarray) -> np.ndarray:
        e = self.w.get("embed", keep=False)
        return to_f64(e[np.asarray(tokens, dtype=np.int64)], self.cfg.dtype)

    def forward_block(self, k_ctx: Sequence[np.ndarray], v_ctx: Sequence[np.ndarray],
                      ctx_pos: np.ndarray, bonus: int, ctx_len: int,
                      layer_hook=None, block_pos0: Optional[int] = None,
                      width: Optional[int] = None) -> np.ndarray:
        """One block forward for one sequence over its cached context K/V (per layer
        [ctx_len, nkv, hd]); returns the final normed hidden [b, H], b = width (default gamma;
        the Atlas head's active block width, dflash_head.rs).
        Block row r takes RoPE position block_pos0 + r, block_pos0 = ctx_len by default (the
        draft starts at the committed length; Atlas's q_rope_pos overrides it).  The sliding
        window is measured on row indices of the sequence: context row i at i, block row r at
        ctx_len + r (these equal the RoPE positions whenever the positions are 0, 1, 2, ...)."""
        c = self.cfg
        g = c.gamma if width is None else int(width)
        nh, nkv, hd = c.n_q_heads, c.n_kv_heads, c.head_dim
        p0 = ctx_len if block_pos0 is None else int(block_pos0)
        pos_b = np.arange(p0, p0 + g, dtype=np.int64)
        idx_b = np.arange(ctx_len, ctx_len + g, dtype=np.int64)
        key_idx = np.arange(ctx_len + g, dtype=np.int64)
        x = self.embed_rows(self.block_tokens(bonus, g))
        for l in range(c.n_layers):
            L = lambda t: self.Wproj(l, t)  # noqa: E731
            xn = rms_norm(x, L("ln_in"), c.rms_eps)
            q = (xn @ L("wq").T).reshape(g, nh, hd)
            kb = (xn @ L("wk").T).reshape(g, nkv, hd)
            vb = (xn @ L("wv").T).reshape(g, nkv, hd)
            q = rope(rms_norm(q, L("q_norm"), c.rms_eps), pos_b, self.inv_freq, self.mscale)
            kb = rope(rms_norm(kb, L("k_norm"), c.rms_eps), pos_b, self.inv_freq, self.mscale)
            keys = np.concatenate([k_ctx[l][:ctx_len], kb], axis=0)
            vals = np.concatenate([v_ctx[l][:ctx_len], vb], axis=0)
            window = c.sliding_window if c.sliding(l) else 0
            a = block_attention(q, keys, vals, idx_b, key_idx, window).reshape(g, nh * hd)
            x1 = x + a @ L("wo").T
            n = rms_norm(x1, L("ln_post"), c.rms_eps)
            act = silu(n @ L("w_gate").T) * (n @ L("w_up").T)
            x = x1 + act @ L("w_down").T
            if layer_hook is not None:
                layer_hook(l, dict(xn=xn, q=q, kb=kb, vb=vb, attn=a, x1=x1, x=x))
        return rms_norm(x, self.W("norm"), c.rms_eps)

    def forward_uncached(self, f_ctx: np.ndarray, ctx_pos: np.ndarray, bonus: int) -> np.ndarray:
        """The first-light form (dflash.rs `forward_block` over ctx features): every
        layer projects K/V for [ctx_f ; block-normed] afresh, k-norms and ropes all
        keys, and attends.  The cached form above must give the same result."""
        c = self.cfg
        g, nh, nkv, hd = c.gamma, c.n_q_heads, c.n_kv_heads, c.head_dim
        n = f_ctx.shape[0]
        pos_b = np.arange(n, n + g, dtype=np.int64)
        pos_all = np.concatenate([np.asarray(ctx_pos, dtype=np.int64), pos_b])
        x = self.embed_rows(self.block_tokens(bonus))
        for l in range(c.n_layers):
            L = lambda t: self.Wproj(l, t)  # noqa: E731
            xn = rms_norm(x, L("ln_in"), c.rms_eps)
            q = (xn @ L("wq").T).reshape(g, nh, hd)
            # context rows through the stored K/V weights (the fused context-K/V weight stays
            # bf16 on the FP8 lane), block rows through the block's projections
            k = np.concatenate([f_ctx @ self.W(f"L{l}.wk").T, xn @ L("wk").T], axis=0).reshape(n + g, nkv, hd)
            v = np.concatenate([f_ctx @ self.W(f"L{l}.wv").T, xn @ L("wv").T], axis=0).reshape(n + g, nkv, hd)
            q = rope(rms_norm(q, L("q_norm"), c.rms_eps), pos_b, self.inv_freq, self.mscale)
            k = rope(rms_norm(k, L("k_norm"), c.rms_eps), pos_all, self.inv_freq, self.mscale)
            window = c.sliding_window if c.sliding(l) else 0
            a = block_attention(q, k, v, np.arange(n, n + g), np.arange(n + g), window).reshape(g, nh * hd)
            x1 = x + a @ L("wo").T
            n1 = rms_norm(x1, L("ln_post"), c.rms_eps)
            x = x1 + (silu(n1 @ L("w_gate").T) * (n1 @ L("w_up").T)) @ L("w_down").T
        return rms_norm(x, self.W("norm"), c.rms_eps)

    # ---- lm_head + argmax: dflash.rs draft step

    def fp8_lm_head(self):
        if self._fp8 is None:
            lm = self.w.get("lm_head", keep=False)
            self._fp8 = fp8_quantize_rows(to_f64(lm, self.cfg.dtype).astype(np.float32))
        return self._fp8

    def logits(self, h: np.ndarray, rows: Optional[np.ndarray] = None,
               chunk: int = 16384) -> np.ndarray:
        """z = lm_head h for the rows of h (all gamma rows by default) -> [rows, V].
        FP8 head: z_v = scale_v * sum_k dec(q_vk) h_k."""
        c = self.cfg
        hh = np.asarray(h, dtype=np.float64)
        out = np.empty((hh.shape[0], c.vocab), dtype=np.float64)
        if c.lm_head_dtype == "fp8":
            codes, scale = self.fp8_lm_head()
            for s in range(0, c.vocab, chunk):
                e = min(c.vocab, s + chunk)
                out[:, s:e] = (hh @ e4m3_decode(codes[s:e]).T) * scale[s:e].astype(np.float64)
            return out
        lm = self.w.get("lm_head", keep=False)
        for s in range(0, c.vocab, chunk):
            e = min(c.vocab, s + chunk)
            out[:, s:e] = hh @ to_f64(lm[s:e], c.dtype).T
        return out

    @staticmethod
    def argmax_rows(z: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        """Per-row argmax (ties -> lowest index) and the top-1 minus top-2 margin."""
        idx = np.argmax(z, axis=1)
        top2 = np.partition(z, -2, axis=1)[:, -2:]
        margin = top2[:, 1] - top2[:, 0]
        return idx.astype(np.int64), margin

    def drafts(self, h: np.ndarray):
        """Draft tokens = argmax over the vocabulary of rows 1..b-1 of a b-row block (row 0 is
        the anchor echo and is dropped).  Returns (logits [b, V], tokens [b-1], margins [b-1])."""
        z = self.logits(h)
        tok, margin = self.argmax_rows(z[1:])
        return z, tok, margin

    # ---- DSpark Markov head: dflash.rs draft step, semi-AR Markov chain

    def drafts_markov(self, h: np.ndarray, bonus: int):
        """Drafts with the DSpark Markov fix-up (see markov_chain): logits of rows 1..gamma-1,
        then the left-to-right chain from the bonus token.  Returns (row-0 logits [V],
        adjusted logits [gamma-1, V], tokens [gamma-1], margins [gamma-1])."""
        z = self.logits(h)
        w1 = to_f64(self.w.get("markov_w1", keep=self.cache), self.cfg.dtype)
        w2 = to_f64(self.w.get("markov_w2", keep=self.cache), self.cfg.dtype)
        adj, tok, margin = markov_chain(z[1:], bonus, w1, w2)
        return z[0], adj, tok, margin

    # ---- whole sequence: features -> cache -> block forward

    def run_sequence(self, taps: np.ndarray, ctx_pos: np.ndarray, bonus: int,
                     block_pos0: Optional[int] = None, width: Optional[int] = None):
        """Context of len(taps) rows, then one block: returns dict of K, V, h, z, tokens."""
        f = self.ctx_features(taps)
        ks, vs = self.ctx_kv(f, ctx_pos)
        h = self.forward_block(ks, vs, ctx_pos, bonus, taps.shape[0], block_pos0=block_pos0, width=width)
        z, tok, margin = self.drafts(h)
        return dict(f=f, k=ks, v=vs, h=h, logits=z, tokens=tok, margin=margin)
