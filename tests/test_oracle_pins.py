"""Pins for the CPU oracle: closed forms, brute force, invariants and independent
library routines (torch CPU in float64), so that a dropped term, a wrong sign, a
wrong index or a transposed operand in the oracle fails here."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O
from synth import CONFIGS, make_weights, make_workload, workload_taps

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


class DictWeights:
    """Weights source with per-name overrides (float32 values) over a seeded set."""

    def __init__(self, base, over):
        self.base, self.over = base, over

    def get(self, name, keep=True):
        return self.over[name] if name in self.over else self.base.get(name, keep)


# ----------------------------------------------------------------------------- RMSNorm


def test_rms_norm_hand_example():
    # x = [3, 4]: mean square 12.5, rms = 3.5355339; w = [1, 2]
    y = O.rms_norm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    np.testing.assert_allclose(y, [3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], rtol=1e-15)


def test_rms_norm_matches_torch_and_invariants():
    x = RNG.standard_normal((7, 96))
    w = 1 + 0.05 * RNG.standard_normal(96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), eps=1e-6)
    np.testing.assert_allclose(O.rms_norm(x, w, 1e-6), ref.numpy(), rtol=1e-13, atol=1e-14)
    y1 = O.rms_norm(x, np.ones(96), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y1 ** 2, axis=-1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(O.rms_norm(37.5 * x, w, 0.0), O.rms_norm(x, w, 0.0), rtol=1e-12)


def test_silu_matches_torch():
    z = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(O.silu(z), torch.nn.functional.silu(torch.from_numpy(z)).numpy(),
                               rtol=1e-14, atol=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0


# ----------------------------------------------------------------------------- RoPE


def test_inv_freq_plain_closed_form():
    inv, ms = O.rope_inv_freq(128, 1e6)
    assert ms == 1.0 and inv[0] == 1.0
    # ratio between consecutive pairs is theta^(2/d); last pair is theta^(-(d-2)/d)
    np.testing.assert_allclose(inv[:-1] / inv[1:], 10 ** (6 * 2 / 128), rtol=1e-12)
    np.testing.assert_allclose(inv[-1], 10 ** (-6 * 126 / 128), rtol=1e-12)


def test_rope_pairing_is_rotate_half():
    # a unit vector on dim j must rotate into dim j + d/2 (NeoX), not j + 1 (interleaved)
    d, p = 64, 7
    inv, _ = O.rope_inv_freq(d, 1e6)
    for j in (0, 5, 31):
        x = np.zeros((1, d))
        x[0, j] = 1.0
        y = O.rope(x, np.array([p]), inv)
        expect = np.zeros(d)
        expect[j] = math.cos(p * inv[j])
        expect[j + d // 2] = math.sin(p * inv[j])
        np.testing.assert_allclose(y[0], expect, atol=1e-15)


def test_rope_matches_complex_rotation():
    d = 128
    inv, _ = O.rope_inv_freq(d, 1e6)
    x = RNG.standard_normal((5, 3, d))
    pos = np.array([0, 1, 17, 4095, 32767])
    y = O.rope(x, pos, inv)
    z = (x[..., : d // 2] + 1j * x[..., d // 2:]) * np.exp(1j * pos[:, None, None] * inv)
    np.testing.assert_allclose(y[..., : d // 2], z.real, atol=1e-12)
    np.testing.assert_allclose(y[..., d // 2:], z.imag, atol=1e-12)


def test_rope_identity_norm_and_relative():
    d = 128
    inv, _ = O.rope_inv_freq(d, 1e6)
    q = RNG.standard_normal((1, d))
    k = RNG.standard_normal((1, d))
    np.testing.assert_array_equal(O.rope(q, np.array([0]), inv), q)
    y = O.rope(q, np.array([1234]), inv)
    pair = lambda v: v[0, : d // 2] ** 2 + v[0, d // 2:] ** 2  # noqa: E731
    np.testing.assert_allclose(pair(y), pair(q), rtol=1e-12)
    dots = [float((O.rope(q, np.array([p + 5]), inv) @ O.rope(k, np.array([p]), inv).T)[0, 0])
            for p in (0, 100, 3000)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)
    ms = 1.3
    np.testing.assert_allclose(O.rope(q, np.array([9]), inv, ms), ms * O.rope(q, np.array([9]), inv))


def test_yarn_wide_drafter_divisors():
    # head_dim 128, theta 1e6, factor 32, original 8192, beta_fast 32, beta_slow 1:
    # corr(32) = 17.17 -> low 17, corr(1) = 33.23 -> high 34 (ramp spans 17 dims).
    # Rearranged closed form: ff_j = factor / (1 + (factor - 1) * ex_j), ex_j = 1 - ramp_j.
    ff = O.yarn_divisors(128, 1e6, (32.0, 8192.0, 32.0, 1.0))
    j = np.arange(64)
    ramp = np.clip((j - 17) / 17.0, 0, 1)
    expect = 32.0 / (1.0 + 31.0 * (1.0 - ramp))
    np.testing.assert_allclose(ff, expect, rtol=1e-12)
    assert np.all(ff[:18] == 1.0) and np.all(np.abs(ff[34:] - 32.0) < 1e-12)
    assert abs(ff[26] - 2.0528) < 1e-4 and abs(ff[33] - 11.3333) < 1e-4
    _, ms = O.rope_inv_freq(128, 1e6, (32.0, 8192.0, 32.0, 1.0))
    assert abs(ms - (1 + 0.1 * math.log(32))) < 1e-15 and abs(ms - 1.346574) < 1e-6


def test_yarn_ramp_guard_when_low_equals_high():
    # original 8192, beta_slow 1400: corr = 128 ln(8192 / (2 pi 1400)) / (2 ln 1e6) = -0.33,
    # so high = ceil = 0; beta_fast 3000 gives corr < 0 and low = max(floor, 0) = 0.  With
    # low == high the ramp's denominator is the 0.001 guard: dim 0 keeps its frequency and
    # every other dim is divided by the full factor
    d, theta, orig = 128, 1e6, 8192.0
    corr = lambda r: d * math.log(orig / (2 * math.pi * r)) / (2 * math.log(theta))  # noqa: E731
    assert -1 < corr(1400.0) <= 0 and corr(3000.0) < 0
    ff = O.yarn_divisors(d, theta, (8.0, orig, 3000.0, 1400.0))
    assert ff[0] == 1.0
    np.testing.assert_allclose(ff[1:], 8.0, rtol=1e-12)


def test_yarn_factor_one_is_plain():
    a, _ = O.rope_inv_freq(128, 1e6)
    b, ms = O.rope_inv_freq(128, 1e6, (1.0, 8192.0, 32.0, 1.0))
    np.testing.assert_allclose(a, b, rtol=1e-15)
    assert ms == 1.0


# ----------------------------------------------------------------------------- attention


def brute_attention(q, k, v, qp, kp, window):
    """Per (row, head) loop with an online (running max) softmax."""
    nq, nh, d = q.shape
    nkv = k.shape[1]
    out = np.zeros_like(q)
    for r in range(nq):
        for h in range(nh):
            g = h * nkv // nh
            m, l, acc = -np.inf, 0.0, np.zeros(d)
            for j in range(k.shape[0]):
                if window and qp[r] - kp[j] >= window:
                    continue
                s = float(q[r, h] @ k[j, g]) / math.sqrt(d)
                mn = max(m, s)
                acc = acc * math.exp(m - mn) + math.exp(s - mn) * v[j, g]
                l = l * math.exp(m - mn) + math.exp(s - mn)
                m = mn
            out[r, h] = acc / l
    return out


@pytest.mark.parametrize("window", [0, 5, 12])
def test_attention_brute_force(window):
    q = RNG.standard_normal((4, 6, 8))
    k = RNG.standard_normal((21, 2, 8))
    v = RNG.standard_normal((21, 2, 8))
    kp = np.concatenate([np.arange(17), 17 + np.arange(4)])
    qp = 17 + np.arange(4)
    np.testing.assert_allclose(O.block_attention(q, k, v, qp, kp, window),
                               brute_attention(q, k, v, qp, kp, window), rtol=1e-12, atol=1e-12)


def test_attention_gqa_equals_mha_replicated():
    q = RNG.standard_normal((16, 8, 16))
    k = RNG.standard_normal((40, 2, 16))
    v = RNG.standard_normal((40, 2, 16))
    p = np.arange(40)
    a = O.block_attention(q, k, v, p[-16:], p)
    b = O.block_attention(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), p[-16:], p)
    np.testing.assert_allclose(a, b, rtol=1e-13)


def test_attention_matches_torch_sdpa():
    q = RNG.standard_normal((16, 8, 32))
    k = RNG.standard_normal((50, 2, 32))
    v = RNG.standard_normal((50, 2, 32))
    p = np.arange(50)
    a = O.block_attention(q, k, v, p[-16:], p)
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(np.repeat(k, 4, axis=1)).permute(1, 0, 2)
    tv = torch.from_numpy(np.repeat(v, 4, axis=1)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=False)
    np.testing.assert_allclose(a, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_attention_window_special_cases():
    q = RNG.standard_normal((16, 4, 16))
    k = RNG.standard_normal((100, 1, 16))
    v = RNG.standard_normal((100, 1, 16))
    kp, qp = np.arange(100), 84 + np.arange(16)
    full = O.block_attention(q, k, v, qp, kp, 0)
    np.testing.assert_allclose(O.block_attention(q, k, v, qp, kp, 100), full, rtol=1e-14)
    # window 1: each query sees only keys at or after its own position
    w1 = O.block_attention(q, k, v, qp, kp, 1)
    for r in range(16):
        sel = kp >= qp[r]
        np.testing.assert_allclose(
            w1[r:r + 1], O.block_attention(q[r:r + 1], k[sel], v[sel], qp[r:r + 1], kp[sel]),
            rtol=1e-13)
    # constant value rows give exactly that row
    vc = np.broadcast_to(RNG.standard_normal((1, 1, 16)), (100, 1, 16))
    np.testing.assert_allclose(O.block_attention(q, k, vc, qp, kp, 7), np.broadcast_to(vc[:1], (16, 4, 16)),
                               rtol=1e-12)


# ----------------------------------------------------------------------------- paging


def test_page_slots_and_paged_equals_contiguous():
    rng = np.random.default_rng(7)
    n, ps, npages = 77, 16, 13
    pt = rng.permutation(npages)[:(n + ps - 1) // ps]
    sl = O.page_slots(pt, 0, n, ps)
    assert [int(s) for s in sl] == [int(pt[i // 16]) * 16 + i % 16 for i in range(n)]
    assert len(set(sl.tolist())) == n
    pool = O.PagedPool(2, npages, 2, 8, ps)
    k = rng.standard_normal((n, 2, 8))
    v = rng.standard_normal((n, 2, 8))
    pool.store(1, pt, 0, k[:30], v[:30])
    pool.store(1, pt, 30, k[30:], v[30:])
    kk, vv = pool.gather(1, pt, n)
    np.testing.assert_array_equal(kk, k)
    np.testing.assert_array_equal(vv, v)
    assert np.isnan(pool.k[0]).all()


# ----------------------------------------------------------------------------- bf16 inputs


def test_bf16_decode_all_patterns_vs_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns warn when widened
        got = O.bf16_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # sign of zero and the infinities survive
    assert np.signbit(got[0x8000]) and not np.signbit(got[0]) and got[0x7F80] == np.inf and got[0xFF80] == -np.inf


# ----------------------------------------------------------------------------- FP8 e4m3


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(nan, np.isnan(got))
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_e4m3_roundtrip_and_spec_points():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    np.testing.assert_array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)
    # OCP OFP8 E4M3: max normal 448 = 0.1111.110, min normal 2^-6 = 0.0001.000,
    # min subnormal 2^-9 = 0.0000.001; NaN = S.1111.111.
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    xs = np.array([float(r[0]) for r in rows])
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint8)
    np.testing.assert_array_equal(O.e4m3_encode(xs), want)


def test_e4m3_encode_matches_torch_cast():
    # 10^7 values over every binade in range
    x = np.concatenate([RNG.standard_normal(2_000_000) * s for s in (0.003, 0.1, 1, 30, 200)])
    x = np.clip(x, -448, 448).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_encode(x), ref)


def test_e4m3_encode_ties_to_even_at_every_midpoint():
    # the exact midpoint between each pair of neighbouring finite codes (subnormal and normal,
    # both signs) rounds to the code with the even mantissa; a hair either side rounds to the
    # nearer code
    pos = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))    # 0 .. 448, increasing
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2
    codes = np.arange(0x7E, dtype=np.uint8)
    even = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    np.testing.assert_array_equal(O.e4m3_encode(mid), even)
    np.testing.assert_array_equal(O.e4m3_encode(-mid), even | 0x80)
    step = (hi - lo) / 64
    np.testing.assert_array_equal(O.e4m3_encode(mid - step), codes)
    np.testing.assert_array_equal(O.e4m3_encode(mid + step), codes + 1)
    ref = torch.from_numpy(mid.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ref, even)


def test_fp8_quantize_rows():
    w = (RNG.standard_normal((64, 300)) * 0.02).astype(np.float32)
    w[5] = 0.0
    codes, scale = O.fp8_quantize_rows(w)
    assert scale.dtype == np.float32 and scale[5] == 1.0 and not codes[5].any()
    np.testing.assert_array_equal(scale[:5], (np.abs(w[:5]).max(1) / np.float32(448)).astype(np.float32))
    dec = O.e4m3_decode(codes) * scale[:, None]
    # the largest element of each row lands on +-448 (or just below through fp32 division)
    amax = np.argmax(np.abs(w), axis=1)
    assert np.all(np.abs(O.e4m3_decode(codes[np.arange(64), amax])[np.arange(64) != 5]) == 448.0)
    # normal-range error bound: half a mantissa step (1/16 relative to the binade)
    rel = np.abs(dec - w) / np.maximum(np.abs(w), 2.0 ** -6 * scale[:, None])
    assert rel.max() <= 1.0 / 16 + 1e-7


# ----------------------------------------------------------------------------- forward


def tiny():
    cfg = CONFIGS["tiny_fp32"]
    wl = make_workload(cfg, 1, [64])
    return cfg, wl, make_weights(cfg, 1)


def test_argmax_ties_lowest_index():
    z = np.array([[0.0, 2.0, 2.0, 1.0], [5.0, 5.0, 5.0, 5.0]])
    idx, margin = O.Oracle.argmax_rows(z)
    assert idx.tolist() == [1, 0] and margin.tolist() == [0.0, 0.0]


def test_forward_cached_equals_uncached():
    cfg, wl, W = tiny()
    o = O.Oracle(cfg, W, cache=True)
    taps = workload_taps(wl, 0, 0, 64)
    pos = wl.ctx_positions(0, 0, 64)
    f = o.ctx_features(taps)
    ks, vs = o.ctx_kv(f, pos)
    a = o.forward_block(ks, vs, pos, 77, 64)
    b = o.forward_uncached(f, pos, 77)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_forward_shift_invariance():
    # shifting every position (context and block) by the same offset leaves the
    # forward unchanged: RoPE only sees relative offsets and nothing else reads positions
    cfg, wl, W = tiny()
    o = O.Oracle(cfg, W, cache=True)
    f = o.ctx_features(workload_taps(wl, 0, 0, 64))
    pos = np.arange(64)
    ks, vs = o.ctx_kv(f, pos)
    k2, v2 = o.ctx_kv(f, pos + 1000)
    a = o.forward_block(ks, vs, pos, 5, 64)
    b = o.forward_block(k2, v2, pos + 1000, 5, 64, block_pos0=1064)
    np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9)
    c = o.forward_block(k2, v2, pos + 1000, 5, 64, block_pos0=1070)
    assert np.abs(a - c).max() > 1e-3


def test_forward_context_permutation_invariance():
    cfg, wl, W = tiny()
    o = O.Oracle(cfg, W, cache=True)
    f = o.ctx_features(workload_taps(wl, 0, 0, 64))
    pos = np.arange(64)
    ks, vs = o.ctx_kv(f, pos)
    perm = np.random.default_rng(3).permutation(64)
    a = o.forward_block(ks, vs, pos, 5, 64)
    b = o.forward_block([k[perm] for k in ks], [v[perm] for v in vs], pos[perm], 5, 64)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_forward_identity_layer():
    # with o_proj and down_proj zero, each layer passes the residual through, so the
    # output is norm(embed[token]) row by row
    cfg, wl, W = tiny()
    over = {"L0.wo": np.zeros((cfg.hidden, cfg.q_dim), np.float32),
            "L0.w_down": np.zeros((cfg.hidden, cfg.n_ff), np.float32)}
    o = O.Oracle(cfg, DictWeights(W, over))
    f = o.ctx_features(workload_taps(wl, 0, 0, 64))
    ks, vs = o.ctx_kv(f, np.arange(64))
    h = o.forward_block(ks, vs, np.arange(64), 9, 64)
    e = W.get("embed")[[9] + [cfg.mask_token_id] * 15].astype(np.float64)
    np.testing.assert_allclose(h, O.rms_norm(e, W.get("norm"), cfg.rms_eps), rtol=1e-12)


def test_forward_single_block_key_context_free():
    # a context of 0 rows: attention sees only the gamma block keys
    cfg, wl, W = tiny()
    o = O.Oracle(cfg, W, cache=True)
    empty = [np.zeros((0, 1, 64))]
    h0 = o.forward_block(empty, empty, np.zeros(0), 3, 0)
    hu = o.forward_uncached(np.zeros((0, cfg.hidden)), np.zeros(0), 3)
    np.testing.assert_allclose(h0, hu, rtol=1e-12, atol=1e-12)
    assert np.isfinite(h0).all()


def test_drafts_drop_anchor_row():
    cfg, wl, W = tiny()
    o = O.Oracle(cfg, W, cache=True)
    h = RNG.standard_normal((16, cfg.hidden))
    z, tok, _ = o.drafts(h)
    lm = W.get("lm_head").astype(np.float64)
    np.testing.assert_allclose(z, h @ lm.T, rtol=1e-12)
    assert tok.tolist() == np.argmax(h[1:] @ lm.T, axis=1).tolist() and tok.shape == (15,)


class _ScaledNorms(O.Oracle):
    """The oracle with some weights multiplied by exact float64 factors."""

    def __init__(self, cfg, weights, scales, mscale):
        super().__init__(cfg, weights, cache=True)
        self.scales = scales
        self.mscale = mscale

    def W(self, name):
        a = super().W(name)
        return a * self.scales[name] if name in self.scales else a


def test_yarn_mscale_multiplies_both_q_and_k():
    """Where the YaRN mscale sits in the whole forward (context K of every layer, the block's q
    and k).  RMSNorm is linear in its weight and RoPE is linear in its input, so multiplying q
    and k by mscale after the rotation is the same as multiplying the q_norm and k_norm weights
    by mscale and rotating with mscale 1 (the YaRN frequencies unchanged).  The YaRN forward must
    equal that, and must differ from the forms that scale only q, only k, or neither."""
    import dataclasses
    cfg = dataclasses.replace(CONFIGS["tiny_fp32"], name="tiny_yarn", n_layers=2, yarn=(32.0, 8192.0, 32.0, 1.0))
    W = make_weights(cfg, 1)
    wl = make_workload(cfg, 1, [64])
    taps = workload_taps(wl, 0, 0, 64)
    pos = np.arange(5000, 5064)                       # angles far from zero
    o = O.Oracle(cfg, W, cache=True)
    m = o.mscale
    assert abs(m - (1 + 0.1 * math.log(32))) < 1e-15
    ref = o.run_sequence(taps, pos, 77)

    def variant(q, k):
        sc = {}
        for l in range(cfg.n_layers):
            if q:
                sc[f"L{l}.q_norm"] = m
            if k:
                sc[f"L{l}.k_norm"] = m
        return _ScaledNorms(cfg, W, sc, 1.0).run_sequence(taps, pos, 77)

    both = variant(True, True)
    rel = lambda a, b: np.abs(a - b).max() / np.abs(b).max()  # noqa: E731
    for l in range(cfg.n_layers):
        assert rel(both["k"][l], ref["k"][l]) < 1e-13
        np.testing.assert_array_equal(both["v"][l], ref["v"][l])
    assert rel(both["h"], ref["h"]) < 1e-12 and rel(both["logits"], ref["logits"]) < 1e-12
    for q, k in ((True, False), (False, True), (False, False)):
        assert rel(variant(q, k)["h"], ref["h"]) > 1e-3, (q, k)


# ----------------------------------------------------------------------------- layer wiring
# Probes with elementary weight matrices: E[i, j] = 1 sends input feature j to output feature i
# under the [out, in] row-major layout of every projection.  The tiny drafter's q and o
# projections are square (q_dim == hidden), so a transposed operand there changes no shape; the
# probes make it land on the wrong feature instead.


def _elem(rows, cols, i, j, val=1.0):
    m = np.zeros((rows, cols), np.float32)
    m[i, j] = val
    return m


def _layer0(cfg, W, over, bonus=9, ctx=64):
    wl = make_workload(cfg, 1, [ctx])
    o = O.Oracle(cfg, DictWeights(W, over))
    f = o.ctx_features(workload_taps(wl, 0, 0, ctx))
    ks, vs = o.ctx_kv(f, np.arange(ctx))
    seen = {}
    o.forward_block(ks, vs, np.arange(ctx), bonus, ctx, layer_hook=lambda l, d: seen.setdefault(l, d))
    x0 = W.get("embed")[[bonus] + [cfg.mask_token_id] * (cfg.gamma - 1)].astype(np.float64)
    return seen[0], x0


def _torch_rms(x, w, eps):
    t = torch.nn.functional.rms_norm(torch.from_numpy(x), (x.shape[-1],), torch.from_numpy(w), eps=eps)
    return t.numpy()


def test_o_proj_and_mlp_wiring():
    cfg, _, W = tiny()
    H, F, qd = cfg.hidden, cfg.n_ff, cfg.q_dim
    over = {"L0.wo": _elem(H, qd, 5, 200),             # attention feature 200 -> residual feature 5
            "L0.w_gate": _elem(F, H, 7, 11, 2.0),       # act 7 gated by 2 * n[11]
            "L0.w_up": _elem(F, H, 7, 13),              # ... times n[13]
            "L0.w_down": _elem(H, F, 9, 7)}             # act 7 -> residual feature 9
    d, x0 = _layer0(cfg, W, over)
    # attention residual: x1 = x + o_proj(attn) touches feature 5 only, by attn[:, 200]
    dx1 = d["x1"] - x0
    np.testing.assert_array_equal(np.delete(dx1, 5, axis=1), 0.0)
    np.testing.assert_allclose(dx1[:, 5], d["attn"][:, 200], rtol=1e-12, atol=1e-15)
    assert np.abs(d["attn"][:, 200]).min() > 1e-6
    # MLP residual on x1 (not on x): feature 9 only, by silu(gate) * up of the post-normed x1
    n = _torch_rms(d["x1"], W.get("L0.ln_post").astype(np.float64), cfg.rms_eps)
    act = torch.nn.functional.silu(torch.from_numpy(2.0 * n[:, 11])).numpy() * n[:, 13]
    dx = d["x"] - d["x1"]
    np.testing.assert_array_equal(np.delete(dx, 9, axis=1), 0.0)
    np.testing.assert_allclose(dx[:, 9], act, rtol=1e-12, atol=1e-15)
    # silu takes the gate: with the roles swapped the values differ
    swapped = torch.nn.functional.silu(torch.from_numpy(n[:, 13])).numpy() * 2.0 * n[:, 11]
    assert np.abs(swapped - act).max() > 1e-3


def test_q_proj_orientation_and_head_split():
    cfg, _, W = tiny()
    H, qd, hd = cfg.hidden, cfg.q_dim, cfg.head_dim
    i, j = 2 * hd + 3, 17                              # input feature 17 -> head 2, dim 3
    d, _ = _layer0(cfg, W, {"L0.wq": _elem(qd, H, i, j)})
    q = d["q"]                                          # [gamma, nh, hd] after q_norm and RoPE
    raw = d["xn"][:, j]
    for h in range(cfg.n_q_heads):
        nz = np.flatnonzero(np.abs(q[:, h]).max(axis=0))
        # one nonzero raw dim: q_norm keeps it alone, RoPE pairs it with its rotate-half partner
        assert nz.tolist() == ([3, 3 + hd // 2] if h == 2 else []), (h, nz)
    # q_norm of a one-hot head vector: |v| / sqrt(v^2 / hd + eps) * w; RoPE keeps the pair norm
    w3 = float(W.get("L0.q_norm")[3])
    expect = np.abs(raw) / np.sqrt(raw ** 2 / hd + cfg.rms_eps) * abs(w3)
    np.testing.assert_allclose(np.hypot(q[:, 2, 3], q[:, 2, 3 + hd // 2]), expect, rtol=1e-12)


def test_uniform_values_give_identical_rows():
    # no context and bonus == mask: the gamma block rows carry the same token, so every
    # layer's V rows are equal (V takes no RoPE) and each softmax-weighted sum returns that
    # row, whatever the position-dependent scores; every final hidden row is then equal
    cfg, _, W = tiny()
    o = O.Oracle(cfg, W)
    empty = [np.zeros((0, cfg.n_kv_heads, cfg.head_dim))] * cfg.n_layers
    seen = {}
    h = o.forward_block(empty, empty, np.zeros(0), cfg.mask_token_id, 0,
                        layer_hook=lambda l, d: seen.setdefault(l, d))
    np.testing.assert_allclose(h, np.broadcast_to(h[0], h.shape), rtol=1e-12, atol=1e-14)
    q = seen[0]["q"]
    assert np.abs(q - q[0]).max() > 1e-3              # the queries do differ by position
    # a distinct bonus token breaks it
    h2 = o.forward_block(empty, empty, np.zeros(0), 9, 0)
    assert np.abs(h2[1:] - h2[0]).max() > 1e-3


def test_ctx_features_are_hidden_normed_projections():
    # f = hidden_norm(fc taps): dividing out the norm weight leaves rows of unit RMS, and a
    # scaled tap row gives the same feature row up to the eps term (eps / mean(y^2) ~ 3e-6
    # here: the norm follows the linear map)
    cfg, wl, W = tiny()
    o = O.Oracle(cfg, W)
    taps = workload_taps(wl, 0, 0, 8).astype(np.float64)
    f = o.ctx_features(taps)
    w = W.get("hidden_norm").astype(np.float64)
    rms = np.sqrt(np.mean((f / w) ** 2, axis=1))
    y = taps @ W.get("fc").astype(np.float64).T
    np.testing.assert_allclose(rms, np.sqrt(np.mean(y ** 2, axis=1) / (np.mean(y ** 2, axis=1) + cfg.rms_eps)),
                               rtol=1e-12)
    np.testing.assert_allclose(o.ctx_features(7.0 * taps), f, rtol=1e-5, atol=1e-6)  # taps enter as fp32
    # fc rows index output features: a one-hot fc row picks one tap column
    over = {"fc": _elem(cfg.hidden, cfg.n_taps * cfg.target_hidden, 3, 100)}
    g = O.Oracle(cfg, DictWeights(W, over)).ctx_features(taps)
    np.testing.assert_array_equal(np.delete(g, 3, axis=1), 0.0)
    # one nonzero feature t of H: t / sqrt(t^2 / H + eps) = sign(t) sqrt(H) / sqrt(1 + eps H / t^2)
    t = taps[:, 100].astype(np.float32).astype(np.float64)
    np.testing.assert_allclose(g[:, 3], np.sign(t) * np.sqrt(cfg.hidden) * w[3]
                               / np.sqrt(1 + cfg.rms_eps * cfg.hidden / t ** 2), rtol=1e-12)


def test_forward_window_rule_at_the_layer_level():
    # a window covering every key (p - j <= 64 + 15 < 80) is exactly full attention; a window one
    # shorter masks key 0 for the last block row (p - j = 79 >= 79) and changes the output; the
    # window applies only on the layers marked sliding
    import dataclasses
    base = dataclasses.replace(CONFIGS["tiny_fp32"], n_layers=2)
    W = make_weights(base, 1)
    wl = make_workload(base, 1, [64])
    taps, pos = workload_taps(wl, 0, 0, 64), np.arange(64)

    def run(**kw):
        o = O.Oracle(dataclasses.replace(base, **kw), W)
        ks, vs = o.ctx_kv(o.ctx_features(taps), pos)
        return o.forward_block(ks, vs, pos, 5, 64)

    full = run()
    np.testing.assert_array_equal(run(sliding_window=80, layer_sliding=(True, True)), full)
    # W = 79 takes key 0 from row 15 in layer 0 only; the other rows change through that row's
    # block key in layer 1
    short = run(sliding_window=79, layer_sliding=(True, False))
    assert np.abs(short - full).max() > 1e-9
    a = run(sliding_window=20, layer_sliding=(True, False))
    b = run(sliding_window=20, layer_sliding=(False, True))
    assert np.abs(a - b).max() > 1e-3 and np.abs(a - full).max() > 1e-3


def test_fp8_lm_head_is_exact_on_the_e4m3_grid():
    # lm_head rows that are e4m3 values times 2^-k (with a +-448 entry, so the row scale is
    # exactly 2^-k) quantise without loss: the FP8 logits equal the full-precision ones
    import dataclasses
    cfg = dataclasses.replace(CONFIGS["tiny_fp32"], lm_head_dtype="fp8")
    W = make_weights(cfg, 1)
    rng = np.random.default_rng(7)
    V, H = cfg.vocab, cfg.hidden
    codes = rng.integers(0, 256, size=(V, H)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38                      # no NaN codes
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vals[:, 0] = np.where(rng.random(V) < 0.5, 448.0, -448.0)
    k = rng.integers(4, 14, size=V)
    lm = (vals * np.ldexp(1.0, -k)[:, None]).astype(np.float32)
    assert np.array_equal(lm.astype(np.float64), vals * np.ldexp(1.0, -k)[:, None])
    o = O.Oracle(cfg, DictWeights(W, {"lm_head": lm}))
    q, scale = o.fp8_lm_head()
    np.testing.assert_array_equal(scale, np.ldexp(1.0, -k).astype(np.float32))
    h = RNG.standard_normal((cfg.gamma, H))
    np.testing.assert_allclose(o.logits(h), h @ lm.astype(np.float64).T, rtol=1e-13, atol=1e-13)


def test_logits_do_not_depend_on_the_vocabulary_chunking():
    import dataclasses
    for head in ("f32", "fp8"):
        cfg = dataclasses.replace(CONFIGS["tiny_fp32"], lm_head_dtype=head)
        o = O.Oracle(cfg, make_weights(cfg, 1))
        h = RNG.standard_normal((cfg.gamma, cfg.hidden))
        np.testing.assert_allclose(o.logits(h, chunk=300), o.logits(h), rtol=1e-13, atol=1e-15)
        # rows are independent: a subset of rows gives the same rows
        np.testing.assert_allclose(o.logits(h[3:5], chunk=7), o.logits(h)[3:5], rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------- DSpark Markov chain


def test_markov_zero_projection_is_the_plain_argmax():
    z = RNG.standard_normal((15, 40))
    w1 = RNG.standard_normal((40, 8))
    adj, tok, margin = O.markov_chain(z, 3, w1, np.zeros((40, 8)))
    np.testing.assert_array_equal(adj, z)
    idx, m = O.Oracle.argmax_rows(z)
    assert tok.tolist() == idx.tolist() and np.allclose(margin, m)


def test_markov_shift_chain_closed_form():
    """w1 = identity and w2 = alpha * (the permutation v -> v + 3 mod V): each step's bias is
    alpha on the successor of the previous token, so the chain walks bonus + 3, bonus + 6, ...
    whatever the (small) logits, and each adjusted row is z plus alpha at that token."""
    V, alpha, bonus = 11, 100.0, 4
    perm = np.zeros((V, V))
    for v in range(V):
        perm[(v + 3) % V, v] = 1.0               # w2 @ e_v = e_{v+3}
    z = 0.1 * RNG.standard_normal((15, V))
    adj, tok, margin = O.markov_chain(z, bonus, np.eye(V), alpha * perm)
    expect = [(bonus + 3 * (k + 1)) % V for k in range(15)]
    assert tok.tolist() == expect
    for k in range(15):
        row = z[k].copy()
        row[expect[k]] += alpha
        np.testing.assert_allclose(adj[k], row, rtol=0, atol=1e-12)
    assert np.all(margin > alpha - 1)


def test_markov_bias_uses_the_realised_previous_token():
    """Row 0's plain argmax is token 1, but the bias of the bonus (0) moves it to 2; row 1's bias
    must then come from 2 (giving 4), not from the plain argmax 1 (giving 3) or the bonus (2)."""
    V = 5
    w2 = np.zeros((V, V))
    w2[2, 0] = 2.0       # prev 0 -> +2 on token 2
    w2[3, 1] = 1.0       # prev 1 -> +1 on token 3
    w2[4, 2] = 1.0       # prev 2 -> +1 on token 4
    z = np.zeros((2, V))
    z[0, 1] = 1.0
    _, tok, _ = O.markov_chain(z, 0, np.eye(V), w2)
    assert tok.tolist() == [2, 4]


def test_markov_matches_explicit_loops():
    """A rank smaller than the vocabulary, random tables, against plain Python loops over the
    definition bias_v = sum_j w2[v][j] * w1[prev][j] with a first-maximum argmax."""
    V, R, b = 13, 4, 6
    rng = np.random.default_rng(7)
    z = rng.standard_normal((b - 1, V))
    w1 = rng.standard_normal((V, R))
    w2 = rng.standard_normal((V, R))
    prev, toks, rows = 9, [], []
    for k in range(b - 1):
        row = [float(z[k][v]) + sum(float(w2[v][j]) * float(w1[prev][j]) for j in range(R)) for v in range(V)]
        best = 0
        for v in range(1, V):
            if row[v] > row[best]:
                best = v
        toks.append(best)
        rows.append(row)
        prev = best
    adj, tok, _ = O.markov_chain(z, 9, w1, w2)
    assert tok.tolist() == toks
    np.testing.assert_allclose(adj, np.array(rows), rtol=1e-12, atol=1e-12)


def test_markov_head_in_the_drafter():
    """The tiny drafter with a rank-32 head: with w2 zeroed the Markov drafts are the plain
    drafts; with the seeded head at least one draft changes (the head is not a no-op)."""
    cfg = CONFIGS["tiny_fp32_markov"]
    W = make_weights(cfg, 1)
    wl = make_workload(cfg, 1, [64])
    taps = workload_taps(wl, 0, 0, 64)
    o = O.Oracle(cfg, W, cache=True)
    ref = o.run_sequence(taps, wl.ctx_positions(0, 0, 64), 77)
    zero = O.Oracle(cfg, DictWeights(W, {"markov_w2": np.zeros((cfg.vocab, cfg.markov_rank), np.float32)}))
    z0, adj0, tok0, _ = zero.drafts_markov(ref["h"], 77)
    assert tok0.tolist() == ref["tokens"].tolist()
    np.testing.assert_allclose(z0, ref["logits"][0], rtol=1e-12)
    _, adj, tok, _ = o.drafts_markov(ref["h"], 77)
    assert tok.tolist() != ref["tokens"].tolist()
    w1 = W.get("markov_w1").astype(np.float64)
    w2 = W.get("markov_w2").astype(np.float64)
    np.testing.assert_allclose(adj[0], ref["logits"][1] + w2 @ w1[77], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- block width, RoPE start


def test_block_width_is_a_narrower_block():
    """A width-b block (the Atlas head's active block width) is exactly the forward of a drafter
    whose block size is b: b rows [bonus, mask x (b-1)], attending to the context and to those b
    rows only.  It is not the first b rows of the full block (whose extra mask rows are keys)."""
    import dataclasses
    cfg, wl, W = tiny()
    o = O.Oracle(cfg, W, cache=True)
    f = o.ctx_features(workload_taps(wl, 0, 0, 64))
    pos = np.arange(64)
    ks, vs = o.ctx_kv(f, pos)
    full = o.forward_block(ks, vs, pos, 5, 64)
    np.testing.assert_array_equal(o.forward_block(ks, vs, pos, 5, 64, width=16), full)
    for b in (2, 7):
        hb = o.forward_block(ks, vs, pos, 5, 64, width=b)
        ob = O.Oracle(dataclasses.replace(cfg, gamma=b), W, cache=True)
        np.testing.assert_allclose(hb, ob.forward_block(ks, vs, pos, 5, 64), rtol=1e-12, atol=1e-12)
        assert hb.shape == (b, cfg.hidden) and np.abs(hb - full[:b]).max() > 1e-3
        z, tok, _ = o.drafts(hb)
        assert z.shape == (b, cfg.vocab) and tok.shape == (b - 1,)


def test_window_is_measured_on_row_indices():
    """The sliding window counts rows of the sequence (context row i at i, block row r at
    ctx_len + r), not RoPE positions: with the block's RoPE start moved 5000 past the context, a
    window covering every row changes nothing, while a window of 20 rows does mask keys."""
    import dataclasses
    cfg0, wl, W = tiny()
    cfg_w = dataclasses.replace(cfg0, sliding_window=80, layer_sliding=(True,))
    o_full, o_w = O.Oracle(cfg0, W, cache=True), O.Oracle(cfg_w, W, cache=True)
    f = o_full.ctx_features(workload_taps(wl, 0, 0, 64))
    pos = np.arange(64)
    ks, vs = o_full.ctx_kv(f, pos)
    a = o_full.forward_block(ks, vs, pos, 5, 64, block_pos0=5064)
    b = o_w.forward_block(ks, vs, pos, 5, 64, block_pos0=5064)
    np.testing.assert_array_equal(a, b)
    o_20 = O.Oracle(dataclasses.replace(cfg0, sliding_window=20, layer_sliding=(True,)), W, cache=True)
    assert np.abs(o_20.forward_block(ks, vs, pos, 5, 64, block_pos0=5064) - a).max() > 1e-3


# ----------------------------------------------------------------------------- FP8 layer weights


def test_fp8_layer_weights_rounding_bound_and_cached_equals_uncached():
    """With FP8 layer weights every projection the block uses is within half an e4m3 step of the
    stored weight (relative 2^-4 for normal codes, absolute 2^-10 * scale below them), the
    context K/V keep the stored weights, and the cached and uncached forms still agree."""
    cfg = CONFIGS["tiny_fp32_fp8w"]
    W = make_weights(cfg, 1)
    wl = make_workload(cfg, 1, [64])
    o = O.Oracle(cfg, W, cache=True)
    for t in O.Oracle.FP8_LAYER:
        w = o.W(f"L0.{t}")
        q = o.Wproj(0, t)
        scale = np.abs(w).max(axis=1, keepdims=True).astype(np.float32) / np.float32(448.0)
        err = np.abs(q - w)
        bound = np.maximum(np.abs(w) * 2.0 ** -4, scale.astype(np.float64) * 2.0 ** -10)
        assert np.all(err <= bound * (1 + 1e-6)), t
        assert np.abs(q - w).max() > 0
    taps = workload_taps(wl, 0, 0, 64)
    pos = wl.ctx_positions(0, 0, 64)
    f = o.ctx_features(taps)
    ks, vs = o.ctx_kv(f, pos)
    k_plain, _ = O.Oracle(CONFIGS["tiny_fp32"], W, cache=True).ctx_kv(f, pos)
    np.testing.assert_array_equal(ks[0], k_plain[0])
    np.testing.assert_allclose(o.forward_block(ks, vs, pos, 77, 64), o.forward_uncached(f, pos, 77),
                               rtol=1e-12, atol=1e-12)


def test_fp8_layer_weights_exact_on_the_e4m3_grid():
    """Weights whose rows are e4m3 values times 2^-k with a +-448 entry quantise losslessly: the
    FP8 forward then equals the full-precision forward; dividing by the scale instead of
    multiplying would not."""
    cfg8, cfg = CONFIGS["tiny_fp32_fp8w"], CONFIGS["tiny_fp32"]
    W = make_weights(cfg, 1)
    rng = np.random.default_rng(5)
    grid = O.e4m3_decode(np.arange(256, dtype=np.uint8))
    grid = grid[np.isfinite(grid)]
    over = {}
    for t in O.Oracle.FP8_LAYER:
        shape = W.get(f"L0.{t}").shape
        k = rng.integers(8, 14, size=(shape[0], 1))
        vals = rng.choice(grid, size=shape)
        vals[:, 0] = 448.0
        over[f"L0.{t}"] = (vals * 2.0 ** -k).astype(np.float32)
    src = DictWeights(W, over)
    o8, o = O.Oracle(cfg8, src, cache=True), O.Oracle(cfg, src, cache=True)
    for t in O.Oracle.FP8_LAYER:
        np.testing.assert_array_equal(o8.Wproj(0, t), o.W(f"L0.{t}"))
    wl = make_workload(cfg, 1, [32])
    taps = workload_taps(wl, 0, 0, 32)
    a = o8.run_sequence(taps, wl.ctx_positions(0, 0, 32), 9)
    b = o.run_sequence(taps, wl.ctx_positions(0, 0, 32), 9)
    np.testing.assert_array_equal(a["h"], b["h"])
