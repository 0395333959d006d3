// Projection-GEMM epilogues shared by the per-projection kernels (gemm_tc.cu) and the
// persistent propose kernel (persist_tc.cu): per-token RMS scales, fused per-head RMSNorm +
// RoPE + paged block-K/V write, residual + next-norm operand, SiLU-gated MLP, lm_head argmax,
// context-K/V writer.  One thread owns one weight row (TMEM lane) and 16 token columns.
#pragma once

#include <cuda_bf16.h>
#include <float.h>

#include "dflash_internal.cuh"
#include "gemm_tc.cuh"

namespace dflash {
namespace {

constexpr int kThreads = 128;

// Barrier over the 128 threads of one epilogue warpgroup (threads 128 g .. 128 g + 127 use
// named barrier 2 + g), so the epilogue also runs inside kernels whose other warps are busy
// elsewhere, and several groups can run epilogues side by side (non-aligned form).
__device__ __forceinline__ void epi_sync() {
  asm volatile("barrier.sync %0, 128;" ::"r"(2 + (int)(threadIdx.x >> 7)) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// RoPE angle of pair j at position pos (from_weights.rs inv_freq table; YaRN divisors
// already folded into inv_freq), as half-turns t = pos * inv_freq_j / pi reduced to [-1, 1],
// then sin/cos(pi t) in fp32.  ip[j] = (hi, lo) splits inv_freq_j / pi into two floats;
// fmaf gives the exact rounding error of pos * hi, and subtracting the nearest even integer
// is exact below 2^24, so t carries ~1e-7 absolute error without float64 arithmetic.
__device__ __forceinline__ void rope_cs(const float2 v, int pos, float* c, float* s) {
  const float p = (float)pos;
  const float a = p * v.x;
  const float e = fmaf(p, v.x, -a);
  const float k = 2.f * rintf(0.5f * a);
  const float t = (a - k) + fmaf(p, v.y, e);
  sincospif(t, s, c);
}

__device__ __forceinline__ int m0_of(int tile_m, int tn) { return tile_m * tn; }

__device__ __forceinline__ void set_status(unsigned* status, unsigned bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// (logit, index) as one unsigned 64-bit key whose unsigned order is `better`'s order: the
// float's bits mapped to an order-preserving unsigned (-0 folded onto +0) in the high word,
// the complement of the index in the low word (ties -> lowest index).
__device__ __forceinline__ unsigned long long argmax_key(float v, int i) {
  const unsigned u = __float_as_uint(v + 0.f);
  const unsigned o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)i);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull));
}

// Shared-memory carve-up of the epilogue (aliases the drained pipeline stages).
struct EpiSmem {
  float xch[kThreads][17];   // one 16-token chunk of the tile, transposed exchange
  float red[4][16];          // per-warp partial reductions for 16 tokens
  float tot[16];             // per-token totals over the tile's 128 rows
  float bv[4][16];
  int bi[4][16];
};

// Sum over the tile's 128 rows of w[row][c] for each of the chunk's 16 tokens, into es.tot.
// Transposed through shared memory: thread (token c = t % 16, group g = t / 16) adds rows
// 16g..16g+15 of token c, then one shuffle and a 4-warp combine.  eps >= 0: es.tot gets the
// RMS scale 1 / sqrt(sum / 128 + eps) instead, computed once per token.
__device__ __forceinline__ void rowsum16(EpiSmem& es, const float (&w)[16], int t, float eps = -1.f) {
#pragma unroll
  for (int c = 0; c < 16; ++c) es.xch[t][c] = w[c];
  epi_sync();
  const int c = t & 15, g = t >> 4;
  float a = 0.f;
#pragma unroll
  for (int r = 0; r < 16; ++r) a += es.xch[g * 16 + r][c];
  a += __shfl_xor_sync(0xffffffffu, a, 16);
  if ((t & 31) < 16) es.red[t >> 5][c] = a;
  epi_sync();
  if (t < 16) {
    const float sum = (es.red[0][t] + es.red[1][t]) + (es.red[2][t] + es.red[3][t]);
    es.tot[t] = eps >= 0.f ? 1.f / sqrtf(sum * (1.f / 128.f) + eps) : sum;
  }
  epi_sync();
}

// Epilogue inputs that do not depend on the accumulator, loaded by epilogue_pre so a caller
// can fetch them while the MMAs are still running.
struct EpiPre {
  float x[16];   // EPI_RESID: residual of the chunk's 16 tokens at this thread's row
  float lnw;     // EPI_RESID: next RMSNorm weight of the row
  float nw;      // EPI_QKV: q_norm / k_norm weight of the row
  float2 ip;     // EPI_QKV: RoPE inv_freq / pi of this thread's pair
  int ctx;       // EPI_QKV: first row index of the chunk's gamma block (its K/V slots)
  int rp0;       // EPI_QKV: RoPE position of the block's row 0
  int pg0, pg1;  // EPI_QKV: page ids of the block's rows (ctx / 16 and the next page)
};

// ctx_known >= 0: the block's start position is already known (saves a dependent load).
template <int EPI>
__device__ __forceinline__ void epilogue_pre(const GemmParams& p, EpiPre& q, int t, int n, int m0, int c0, int tile_n,
                                             int ctx_known = -1) {
  if constexpr (EPI == EPI_RESID) {
    q.lnw = p.ln_next ? __bfloat162float(p.ln_next[n]) : 1.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) q.x[c] = m0 + c0 + c < p.M ? __ldcg(p.x + (int64_t)(m0 + c0 + c) * p.H + n) : 0.f;
  } else if constexpr (EPI == EPI_QKV) {
    const int hh = tile_n;
    const bool is_q = hh < p.nh, is_k = !is_q && hh < p.nh + p.nkv;
    const int mb = m0 + c0;
    const int s = mb / kGamma;
    q.ctx = ctx_known >= 0 ? ctx_known : (mb < p.M ? __ldg(p.ctx_lens + s) : 0);
    q.rp0 = mb < p.M ? rope_start(p.rope_pos0, s, q.ctx) : 0;
    q.nw = (is_q || is_k) ? __bfloat162float((is_q ? p.q_norm : p.k_norm)[t]) : 1.f;
    q.ip = p.inv_pi[t & 63];
    q.pg0 = q.pg1 = -1;
    if (!is_q && mb < p.M && q.ctx >= 0 && q.ctx + kGamma <= p.mpps * kPage) {
      const int32_t* pt = p.page_tables + (int64_t)s * p.mpps + q.ctx / kPage;
      q.pg0 = __ldg(pt);
      q.pg1 = (q.ctx % kPage) ? __ldg(pt + 1) : q.pg0;
    }
  }
}

template <int EPI>
__device__ void epilogue_chunk(const GemmParams& p, EpiSmem& es, const float* rsc, float (&v)[16], int t, int n,
                               int m0, int c0, int tile_n, const EpiPre& q) {
  if constexpr (EPI == EPI_STORE) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int m = m0 + c0 + c;
      if (m < p.M && n < p.N) p.out[(int64_t)m * p.ldo + n] = v[c] * (p.ss_in ? rsc[c0 + c] : 1.f);
    }
  } else if constexpr (EPI == EPI_RESID) {
    float sq[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int m = m0 + c0 + c;
      float xv = 0.f;
      if (m < p.M) {
        const int64_t o = (int64_t)m * p.H + n;
        xv = q.x[c] + v[c];
        p.x[o] = xv;
        p.xb[o] = __float2bfloat16_rn(xv * q.lnw);
      }
      sq[c] = xv * xv;
    }
    rowsum16(es, sq, t);
    if (t < 16) {
      const int m = m0 + c0 + t;
      if (m < p.M) p.ss_out[(int64_t)tile_n * p.Mp + m] = es.tot[t];
    }
  } else if constexpr (EPI == EPI_GATEUP) {
#pragma unroll
    for (int c = 0; c < 16; ++c) es.xch[t][c] = v[c] * rsc[c0 + c];
    epi_sync();
    const int f = tile_n * 64 + (t & 63);
    const int cb = (t >> 6) * 8;
#pragma unroll
    for (int c = cb; c < cb + 8; ++c) {
      const int m = m0 + c0 + c;
      if (m < p.M) {
        const float g = es.xch[t & 63][c], u = es.xch[(t & 63) + 64][c];
        p.act[(int64_t)m * p.F + f] = __float2bfloat16_rn(g / (1.f + __expf(-g)) * u);
      }
    }
    epi_sync();
  } else if constexpr (EPI == EPI_QKV) {
    const int hh = tile_n;
    const bool is_q = hh < p.nh, is_k = !is_q && hh < p.nh + p.nkv;
    // the chunk's 16 tokens are one gamma block at positions ctx .. ctx + 15
    const int mb = m0 + c0;
    const int ctx = q.ctx;
#pragma unroll
    for (int c = 0; c < 16; ++c) v[c] *= rsc[c0 + c];
    if (is_q || is_k) {
      // per-head RMSNorm over the 128 rows of the tile
      float sq[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) sq[c] = v[c] * v[c];
      rowsum16(es, sq, t, p.eps);
#pragma unroll
      for (int c = 0; c < 16; ++c) es.xch[t][c] = v[c] * es.tot[c] * q.nw;
      epi_sync();
      // RoPE: pair (j, j + 64), NeoX rotate-half.  The block's positions are consecutive, so
      // the angle at ctx + c comes from the one at ctx by c rotations through one position's
      // angle (fp32 error ~c * 6e-8, far below the bf16 rounding of the result).
      const int j = t & 63;
      float cs, sn, c1, s1;
      rope_cs(q.ip, q.rp0, &cs, &sn);
      rope_cs(q.ip, 1, &c1, &s1);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float a = es.xch[j][c], b = es.xch[j + 64][c];
        v[c] = (t < 64 ? a * cs - b * sn : b * cs + a * sn) * p.mscale;
        const float cn = cs * c1 - sn * s1;
        sn = fmaf(sn, c1, cs * s1);
        cs = cn;
      }
      epi_sync();
    }
    if (mb < p.M) {
      if (is_q) {
#pragma unroll
        for (int c = 0; c < 16; ++c) p.q[(int64_t)(mb + c) * p.nh * 128 + hh * 128 + t] = __float2bfloat16_rn(v[c]);
      } else if (ctx < 0 || ctx + kGamma > p.mpps * kPage) {
        if (t == 0) set_status(p.status, DFLASH_DEV_BAD_CTX);
      } else {
        // the block's rows fall on at most two pages (ids looked up in epilogue_pre); each
        // thread writes whole 16-byte runs of the page tile layout
        const int head = is_k ? hh - p.nh : hh - p.nh - p.nkv;
        const bool ok0 = q.pg0 >= 0 && q.pg0 < p.g.num_pages, ok1 = q.pg1 >= 0 && q.pg1 < p.g.num_pages;
        if (t == 0 && (!ok0 || ((ctx % kPage) && !ok1))) set_status(p.status, DFLASH_DEV_BAD_PAGE);
        const int64_t base0 = ok0 ? tile_base(p.g, p.layer, q.pg0, is_k ? 0 : 1, head) : -1;
        const int64_t base1 = ok1 ? tile_base(p.g, p.layer, q.pg1, is_k ? 0 : 1, head) : -1;
        if (is_k) {
          // K rows hold 8 consecutive dims per run: gather dims through shared memory
#pragma unroll
          for (int c = 0; c < 16; ++c) es.xch[t][c] = v[c];
          epi_sync();
          const int c = t >> 3, li = ctx + c;
          const int64_t base = (li / kPage == ctx / kPage) ? base0 : base1;
          if (base >= 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int d0 = (2 * (t & 7) + h) * 8;
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(es.xch[d0 + 2 * e][c], es.xch[d0 + 2 * e + 1][c]);
                pk[e] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              *reinterpret_cast<uint4*>(p.pool + base + k_in_tile(li % kPage, d0, 128)) =
                  make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
          epi_sync();
        } else if ((ctx & 7) == 0) {
          // V rows hold 8 consecutive keys per run: this thread's dim, keys 8h .. 8h + 7
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int li = ctx + 8 * h;
            const int64_t base = (li / kPage == ctx / kPage) ? base0 : base1;
            if (base < 0) continue;
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * h + 2 * e], v[8 * h + 2 * e + 1]);
              pk[e] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(p.pool + base + v_in_tile(li % kPage, t, 128)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int li = ctx + c;
            const int64_t base = (li / kPage == ctx / kPage) ? base0 : base1;
            if (base >= 0) p.pool[base + v_in_tile(li % kPage, t, 128)] = __float2bfloat16_rn(v[c]);
          }
        }
      }
    }
  } else if constexpr (EPI == EPI_CTXKV) {
    // one tile = one head of one layer's K or V in the fused context-K/V weight
    // [K_0; V_0; K_1; V_1; ...]; token m is context row first + m at position positions[m]
    const int l = tile_n / (2 * p.nkv), rem = tile_n % (2 * p.nkv);
    const bool is_k = rem < p.nkv;
    const int head = is_k ? rem : rem - p.nkv;
    if (is_k) {
      float sq[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) sq[c] = v[c] * v[c];
      rowsum16(es, sq, t, p.eps);
      const float w = __bfloat162float(p.k_norm[l * 128 + t]);
#pragma unroll
      for (int c = 0; c < 16; ++c) es.xch[t][c] = v[c] * es.tot[c] * w;
      epi_sync();
      const int j = t & 63;
      const float2 ipj = p.inv_pi[j];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int m = m0 + c0 + c;
        const int pos = m < p.M ? p.positions[m] : 0;
        float cs, sn;
        rope_cs(ipj, pos, &cs, &sn);
        const float a = es.xch[j][c], b = es.xch[j + 64][c];
        v[c] = (t < 64 ? a * cs - b * sn : b * cs + a * sn) * p.mscale;
      }
      epi_sync();
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int m = m0 + c0 + c;
      if (m >= p.M) continue;
      const int li = p.row_index ? __ldg(p.row_index + m) : p.first + m;
      const int sq = p.row_seq ? __ldg(p.row_seq + m) : 0;
      if (sq < 0 || sq >= p.nseq || li < 0 || li >= p.mpps * kPage) {  // batched rows: checked on the device
        if (t == 0) set_status(p.status, DFLASH_DEV_BAD_CTX);
        continue;
      }
      const int page = p.page_tables[(int64_t)sq * p.mpps + li / kPage];
      if (page < 0 || page >= p.g.num_pages) {
        if (t == 0) set_status(p.status, DFLASH_DEV_BAD_PAGE);
        continue;
      }
      const int64_t base = tile_base(p.g, l, page, is_k ? 0 : 1, head);
      p.pool[base + (is_k ? k_in_tile(li % kPage, t, 128) : v_in_tile(li % kPage, t, 128))] =
          __float2bfloat16_rn(v[c]);
    }
  } else if constexpr (EPI == EPI_LMHEAD) {
    const bool valid_row = n < p.N;
    const float sc = (p.row_scale && valid_row) ? p.row_scale[n] : 1.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int m = m0 + c0 + c;
      const float z = v[c] * sc * (p.ss_in ? rsc[c0 + c] : 1.f);
      if (p.logits && valid_row && m < p.M) p.logits[(int64_t)m * p.N + n] = __float2bfloat16_rn(z);
      if (p.logits32 && valid_row && m < p.M) p.logits32[(int64_t)m * p.N + n] = z;
      es.xch[t][c] = valid_row ? z : -FLT_MAX;
    }
    epi_sync();
    // thread (token c, group g) scans rows 16g..16g+15 (ties -> lowest row), then combine
    const int c = t & 15, g = t >> 4;
    float b = -FLT_MAX;
    int bi = 0x7fffffff;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float z = es.xch[g * 16 + r][c];
      const int idx = tile_n * 128 + g * 16 + r;
      if (z > b) { b = z; bi = idx; }
    }
    if (b == -FLT_MAX) bi = 0x7fffffff;
    {
      const float ob = __shfl_xor_sync(0xffffffffu, b, 16);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, 16);
      if (better(ob, oi, b, bi)) { b = ob; bi = oi; }
    }
    if ((t & 31) < 16) { es.bv[t >> 5][c] = b; es.bi[t >> 5][c] = bi; }
    epi_sync();
    if (t < 16) {
      float bb = es.bv[0][t];
      int ii = es.bi[0][t];
      for (int w2 = 1; w2 < 4; ++w2)
        if (better(es.bv[w2][t], es.bi[w2][t], bb, ii)) { bb = es.bv[w2][t]; ii = es.bi[w2][t]; }
      const int m = m0 + c0 + t;
      if (m < p.M && ii != 0x7fffffff) atomicMax(p.amax_best + m, argmax_key(bb, ii));
    }
    epi_sync();
  }
}

}  // namespace
}  // namespace dflash
