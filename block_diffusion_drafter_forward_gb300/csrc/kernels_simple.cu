// CUDA-core kernels of the drafter forward, templated on the element type (fp32 or bf16).
// They carry the fp32 configuration end to end (tensor cores have no fp32 kind that
// meets an fp32 tolerance) and are the building blocks the tensor-core path reuses for
// its small steps (embedding gather, argmax, the create-time FP8 quantiser).
//
// Operations follow memra-engine `dflash.rs` (forward_round, ingest_ctx, the draft step)
// and spark_model `dflash_head/from_weights.rs` (paged pool, slot mapping, FP8 block).
#include <cuda_fp8.h>
#include <float.h>

#include "dflash_internal.cuh"

namespace dflash {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the block (blockDim.x a multiple of 32, <= 1024).  All threads get the total.
__device__ float block_sum(float v) {
  __shared__ float part[32];
  __shared__ float total;
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) part[w] = v;
  __syncthreads();
  if (w == 0) {
    float t = lane < (int)(blockDim.x >> 5) ? part[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) total = t;
  }
  __syncthreads();
  const float r = total;
  __syncthreads();
  return r;
}

// RoPE angle of pair j at position pos (from_weights.rs inv_freq table; YaRN divisors
// already folded into inv_freq), as half-turns t = pos * inv_freq_j / pi reduced to [-1, 1],
// then sin/cos(pi t) in fp32.  ip[j] = (hi, lo) splits inv_freq_j / pi into two floats;
// fmaf gives the exact rounding error of pos * hi, and subtracting the nearest even integer
// is exact below 2^24, so t carries ~1e-7 absolute error without float64 arithmetic.
__device__ __forceinline__ void rope_cs(const float2* ip, int j, int pos, float* c, float* s) {
  const float p = (float)pos;
  const float2 v = ip[j];
  const float a = p * v.x;
  const float e = fmaf(p, v.x, -a);
  const float k = 2.f * rintf(0.5f * a);
  const float t = (a - k) + fmaf(p, v.y, e);
  sincospif(t, s, c);
}

__device__ __forceinline__ void flag(unsigned* status, unsigned bit) { atomicOr(status, bit); }

// ------------------------------------------------------------------------ embedding
// x[r] = E[tok_r], tok = bonus for band row 0, mask_token_id for rows 1..gamma-1
// (dflash.rs draft step: block = [last, MASK x (b-1)]).
template <typename T>
__global__ void embed_kernel(const T* __restrict__ E, const int32_t* __restrict__ bonus, int mask, int V,
                             int H, float* __restrict__ x, unsigned* status, const int32_t* __restrict__ widths) {
  const int row = blockIdx.x;
  const int r = row % kGamma, s = row / kGamma;
  int tok = r == 0 ? bonus[s] : mask;
  const bool ok = tok >= 0 && tok < V;
  if (!ok && threadIdx.x == 0) flag(status, DFLASH_DEV_BAD_TOKEN);
  if (r == 0 && threadIdx.x == 0 && width_out_of_range(widths, s)) flag(status, DFLASH_DEV_BAD_WIDTH);
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    x[(int64_t)row * H + i] = ok ? Elem<T>::to_f(E[(int64_t)tok * H + i]) : 0.f;
}

// ------------------------------------------------------------------------ RMSNorm
// out = x * w / sqrt(mean(x^2) + eps)   (vanilla form, from_weights.rs kernel table)
template <typename T, typename TO = T>
__global__ void rmsnorm_kernel(const float* __restrict__ x, const T* __restrict__ w, TO* __restrict__ out,
                               int n, float eps) {
  const float* xr = x + (int64_t)blockIdx.x * n;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) ss += xr[i] * xr[i];
  ss = block_sum(ss);
  const float inv = 1.f / sqrtf(ss / (float)n + eps);
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    out[(int64_t)blockIdx.x * n + i] = Elem<TO>::from_f(xr[i] * inv * Elem<T>::to_f(w[i]));
}

// ------------------------------------------------------------------------ GEMM (CUDA cores)
// Y[m, n] (+)= sum_k X[m, k] W[n, k].  64x64 tile per block, 16-deep k slices, 4x4 per
// thread, fp32 accumulation.
template <typename TX, typename T, bool FP8W>
__global__ void __launch_bounds__(256) gemm_kernel(const TX* __restrict__ X, int ldx, const void* __restrict__ Wv,
                                                   const float* __restrict__ wscale, int M, int N, int K,
                                                   float* __restrict__ Y, int ldy, int accumulate) {
  __shared__ float Xs[16][68];
  __shared__ float Ws[16][68];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 1024; i += 256) {
      const int rr = i >> 4, kk = i & 15;
      const int k = k0 + kk;
      const int m = m0 + rr, n = n0 + rr;
      Xs[kk][rr] = (m < M && k < K) ? Elem<TX>::to_f(X[(int64_t)m * ldx + k]) : 0.f;
      float wv = 0.f;
      if (n < N && k < K) {
        if constexpr (FP8W) {
          const uint8_t c = static_cast<const uint8_t*>(Wv)[(int64_t)n * K + k];
          __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
          wv = __half2float(__half(hr));
        } else {
          wv = Elem<T>::to_f(static_cast<const T*>(Wv)[(int64_t)n * K + k]);
        }
      }
      Ws[kk][rr] = wv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = Xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float v = acc[i][j];
      if constexpr (FP8W) v *= wscale[n];
      float* yp = Y + (int64_t)m * ldy + n;
      *yp = accumulate ? *yp + v : v;
    }
  }
}

// ------------------------------------------------------------------------ q/k/v post-processing
// For block row `row` and fused-QKV head `hh` (q heads, then k heads, then v heads):
// q, k: per-head RMSNorm with q_norm / k_norm, RoPE at position ctx_len + r, * mscale
// (dflash.rs forward_round + rope_rows); q -> q buffer; k, v -> the pool at logical row
// ctx_len + r of the sequence (the transient block K/V).
template <typename T>
__global__ void qkv_post_kernel(const float* __restrict__ y, int ldy, const T* __restrict__ qn_w,
                                const T* __restrict__ kn_w, const float2* __restrict__ inv_pi, float mscale,
                                float eps, int nh, int nkv, int hd, const int32_t* __restrict__ ctx_lens,
                                const int32_t* __restrict__ page_tables, int mpps, PoolGeom g, int layer,
                                T* __restrict__ pool, T* __restrict__ qout, unsigned* status,
                                const int32_t* __restrict__ rope_pos0) {
  extern __shared__ float sm[];
  const int row = blockIdx.x, hh = blockIdx.y, d = threadIdx.x;
  const int s = row / kGamma, r = row % kGamma;
  const int ctx = ctx_lens[s];
  if (ctx < 0 || ctx + kGamma > mpps * kPage) {
    if (d == 0) flag(status, DFLASH_DEV_BAD_CTX);
    return;
  }
  const int pos = rope_start(rope_pos0, s, ctx) + r;  // RoPE position; the K/V slot stays ctx + r
  float v = y[(int64_t)row * ldy + hh * hd + d];
  const bool is_q = hh < nh, is_k = !is_q && hh < nh + nkv;
  if (is_q || is_k) {
    const float ss = block_sum(v * v);
    const float w = Elem<T>::to_f((is_q ? qn_w : kn_w)[d]);
    v = v * (1.f / sqrtf(ss / (float)hd + eps)) * w;
    sm[d] = v;
    __syncthreads();
    const int half = hd >> 1, j = d < half ? d : d - half;
    float c, sn;
    rope_cs(inv_pi, j, pos, &c, &sn);
    const float a = sm[j], b = sm[j + half];
    v = (d < half ? a * c - b * sn : b * c + a * sn) * mscale;
  }
  if (is_q) {
    qout[(int64_t)row * nh * hd + hh * hd + d] = Elem<T>::from_f(v);
    return;
  }
  const int head = is_k ? hh - nh : hh - nh - nkv;
  const int li = ctx + r;
  const int page = page_tables[(int64_t)s * mpps + li / kPage];
  if (page < 0 || page >= g.num_pages) {
    if (d == 0) flag(status, DFLASH_DEV_BAD_PAGE);
    return;
  }
  const int64_t base = tile_base(g, layer, page, is_k ? 0 : 1, head);
  const int64_t off = is_k ? k_in_tile(li % kPage, d, hd) : v_in_tile(li % kPage, d, hd);
  pool[base + off] = Elem<T>::from_f(v);
}

// ------------------------------------------------------------------------ attention (CUDA cores)
// One warp per (block row, q head): online softmax over keys 0..ctx_len+gamma-1 of the
// sequence, all read through the page table.  Non-causal; on sliding layers a key at
// logical position j is masked for query position p iff p - j >= window.
template <typename T>
__global__ void attention_kernel(const T* __restrict__ q, const T* __restrict__ pool, PoolGeom g, int layer,
                                 const int32_t* __restrict__ ctx_lens, const int32_t* __restrict__ page_tables,
                                 int mpps, int max_ctx, int rows, int nh, int nkv, int hd, int window,
                                 T* __restrict__ out, unsigned* status, const int32_t* __restrict__ widths) {
  const int lane = threadIdx.x & 31;
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= rows * nh) return;
  const int row = wid / nh, h = wid % nh;
  const int s = row / kGamma, r = row % kGamma;
  const int kvh = h / (nh / nkv);
  const int ctx = ctx_lens[s];
  if (ctx < 0 || ctx + kGamma > mpps * kPage) return;  // flagged by qkv_post
  if (ctx > max_ctx) {  // the caller's bound on every ctx_len of this call
    if (lane == 0 && r == 0 && h == 0) flag(status, DFLASH_DEV_BAD_CTX);
    return;
  }
  const int nkeys = ctx + block_width(widths, s), pq = ctx + r;  // keys past the block width are masked
  const int per = hd >> 5;  // dims per lane (2 or 4)
  float qv[4], o[4];
  for (int i = 0; i < per; ++i) {
    qv[i] = Elem<T>::to_f(q[(int64_t)row * nh * hd + h * hd + lane + 32 * i]);
    o[i] = 0.f;
  }
  const float scale = 1.f / sqrtf((float)hd);
  float m = -FLT_MAX, l = 0.f;
  const int j0 = window > 0 ? max(0, pq - window + 1) : 0;
  for (int j = j0; j < nkeys; ++j) {
    const int page = page_tables[(int64_t)s * mpps + j / kPage];
    if (page < 0 || page >= g.num_pages) {
      if (lane == 0) flag(status, DFLASH_DEV_BAD_PAGE);
      continue;
    }
    const int64_t kb = tile_base(g, layer, page, 0, kvh), vb = tile_base(g, layer, page, 1, kvh);
    float dot = 0.f;
    for (int i = 0; i < per; ++i) dot += qv[i] * Elem<T>::to_f(pool[kb + k_in_tile(j % kPage, lane + 32 * i, hd)]);
    dot = warp_sum(dot) * scale;
    const float mn = fmaxf(m, dot);
    const float corr = __expf(m - mn), p = __expf(dot - mn);
    l = l * corr + p;
    for (int i = 0; i < per; ++i)
      o[i] = o[i] * corr + p * Elem<T>::to_f(pool[vb + v_in_tile(j % kPage, lane + 32 * i, hd)]);
    m = mn;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  for (int i = 0; i < per; ++i) out[(int64_t)row * nh * hd + h * hd + lane + 32 * i] = Elem<T>::from_f(o[i] * inv);
}

// ------------------------------------------------------------------------ SiLU-gated MLP
// act = silu(gate) * up with y = [gate | up] per row (dflash.rs forward_round: silu_mul).
template <typename T>
__global__ void silu_mul_kernel(const float* __restrict__ y, int ldy, int F, int rows, T* __restrict__ act) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)rows * F) return;
  const int64_t row = i / F, c = i % F;
  const float gt = y[row * ldy + c], up = y[row * ldy + F + c];
  act[i] = Elem<T>::from_f(gt / (1.f + __expf(-gt)) * up);
}

// ------------------------------------------------------------------------ argmax + logits out
// drafts[s, r-1] = argmax_v z[s*gamma + r, v] for r = 1..gamma-1, ties to the lowest v
// (dflash.rs draft step: argmax of lm_head over block rows 1..b-1).
template <typename T>
__global__ void argmax_kernel(const float* __restrict__ z, int V, int32_t* __restrict__ drafts, T* __restrict__ zout,
                              const int32_t* __restrict__ widths) {
  const int row = blockIdx.x;
  const float* zr = z + (int64_t)row * V;
  float best = -FLT_MAX;
  int bi = 0x7fffffff;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float x = zr[v];
    if (zout) zout[(int64_t)row * V + v] = Elem<T>::from_f(x);
    if (x > best || (x == best && v < bi)) { best = x; bi = v; }
  }
  __shared__ float sb[32];
  __shared__ int si[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) { sb[w] = best; si[w] = bi; }
  __syncthreads();
  if (w == 0) {
    best = lane < (int)(blockDim.x >> 5) ? sb[lane] : -FLT_MAX;
    bi = lane < (int)(blockDim.x >> 5) ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
    }
    const int r = row % kGamma;
    if (lane == 0 && r > 0) drafts[(row / kGamma) * (kGamma - 1) + r - 1] = r < block_width(widths, row / kGamma) ? bi : -1;
  }
}

// ------------------------------------------------------------------------ context K/V writer epilogue
// ykv row i = [K_0 | V_0 | K_1 | V_1 | ...] (fused context-K/V weight, from_weights.rs);
// K: k_norm per head, RoPE at positions[i], * mscale; V raw; both stored at logical row
// first + i (dflash.rs ingest_ctx).
template <typename T>
__global__ void ctxkv_post_kernel(const float* __restrict__ ykv, int ldy, const T* __restrict__ kn_all,
                                  const float2* __restrict__ inv_pi, float mscale, float eps, int nkv, int hd,
                                  const int32_t* __restrict__ positions, const int32_t* __restrict__ page_table,
                                  int first, PoolGeom g, T* __restrict__ pool, unsigned* status,
                                  const int32_t* __restrict__ row_seq, const int32_t* __restrict__ row_index,
                                  int nseq, int mpps) {
  extern __shared__ float sm[];
  const int i = blockIdx.x, d = threadIdx.x;
  const int l = blockIdx.y / (2 * nkv), rem = blockIdx.y % (2 * nkv);
  const bool is_k = rem < nkv;
  const int head = is_k ? rem : rem - nkv;
  float v = ykv[(int64_t)i * ldy + (int64_t)blockIdx.y * hd + d];
  if (is_k) {
    const float ss = block_sum(v * v);
    v = v * (1.f / sqrtf(ss / (float)hd + eps)) * Elem<T>::to_f(kn_all[l * hd + d]);
    sm[d] = v;
    __syncthreads();
    const int half = hd >> 1, j = d < half ? d : d - half;
    float c, sn;
    rope_cs(inv_pi, j, positions[i], &c, &sn);
    const float a = sm[j], b = sm[j + half];
    v = (d < half ? a * c - b * sn : b * c + a * sn) * mscale;
  }
  // row i -> row index first + i of the one sequence, or (batched) row_index[i] of row_seq[i]
  const int li = row_index ? row_index[i] : first + i;
  const int sq = row_seq ? row_seq[i] : 0;
  if (sq < 0 || sq >= nseq || li < 0 || li >= mpps * kPage) {
    if (d == 0) flag(status, DFLASH_DEV_BAD_CTX);
    return;
  }
  const int page = page_table[(int64_t)sq * mpps + li / kPage];
  if (page < 0 || page >= g.num_pages) {
    if (d == 0) flag(status, DFLASH_DEV_BAD_PAGE);
    return;
  }
  const int64_t base = tile_base(g, l, page, is_k ? 0 : 1, head);
  pool[base + (is_k ? k_in_tile(li % kPage, d, hd) : v_in_tile(li % kPage, d, hd))] = Elem<T>::from_f(v);
}

// ------------------------------------------------------------------------ FP8 quantiser (create time)
// scale_v = fp32(max_k |w_vk|) / 448 (1 for a zero row); q_vk = e4m3_rne_satfinite(w_vk / scale_v)
// (from_weights.rs FP8 block: per-output-row fp32 scale; IEEE divisions).
template <typename T>
__global__ void quantize_fp8_kernel(const T* __restrict__ w, int cols, uint8_t* __restrict__ codes,
                                    float* __restrict__ scale) {
  const T* wr = w + (int64_t)blockIdx.x * cols;
  float mx = 0.f;
  for (int k = threadIdx.x; k < cols; k += blockDim.x) mx = fmaxf(mx, fabsf(Elem<T>::to_f(wr[k])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __shared__ float part[32];
  __shared__ float sc;
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t = fmaxf(t, part[i]);
    sc = t == 0.f ? 1.f : __fdiv_rn(t, 448.f);
    scale[blockIdx.x] = sc;
  }
  __syncthreads();
  const float s = sc;
  for (int k = threadIdx.x; k < cols; k += blockDim.x)
    codes[(int64_t)blockIdx.x * cols + k] =
        (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(Elem<T>::to_f(wr[k]), s), __NV_SATFINITE, __NV_E4M3);
}

// ------------------------------------------------------------------------ tensor-core path helpers
// Embedding rows for the tensor-core path: fp32 residual x, xb = bf16(x * ln) with ln the
// first layer's input RMSNorm weight (operand of the first projection), and per-128-column
// partial sums of x^2 (ss[g * Mp + row]), from which that projection's epilogue forms
// 1/RMS(x): W (x * ln) / RMS(x) = W RMSNorm(x).
__global__ void embed_tc_kernel(const __nv_bfloat16* __restrict__ E, const int32_t* __restrict__ bonus, int mask,
                                int V, int H, int Mp, const __nv_bfloat16* __restrict__ ln, float* __restrict__ x,
                                __nv_bfloat16* __restrict__ xb, float* __restrict__ ss, unsigned* status,
                                const int32_t* __restrict__ widths) {
  __shared__ float part[4];
  const int row = blockIdx.x, t = threadIdx.x;
  const int r = row % kGamma, s = row / kGamma;
  const int tok = r == 0 ? bonus[s] : mask;
  const bool ok = tok >= 0 && tok < V;
  if (!ok && t == 0) flag(status, DFLASH_DEV_BAD_TOKEN);
  if (r == 0 && t == 0 && width_out_of_range(widths, s)) flag(status, DFLASH_DEV_BAD_WIDTH);
  for (int g = 0; g < H / 128; ++g) {
    const int i = g * 128 + t;
    const __nv_bfloat16 e = ok ? E[(int64_t)tok * H + i] : __float2bfloat16_rn(0.f);
    const float v = __bfloat162float(e);
    x[(int64_t)row * H + i] = v;
    xb[(int64_t)row * H + i] = __float2bfloat16_rn(v * __bfloat162float(ln[i]));
    const float w = warp_sum(v * v);
    if ((t & 31) == 0) part[t >> 5] = w;
    __syncthreads();
    if (t == 0) ss[(int64_t)g * Mp + row] = part[0] + part[1] + part[2] + part[3];
    __syncthreads();
  }
}

// out[p, k] = W_src(p)[k] (* ln[k] when ln is given) in bf16, with W_src(p) the packed row p:
//  mode 0: rows of A (fused q|k|v, already packed), in place;
//  mode 1: gate/up interleaved in blocks of 64 rows (block b = gate rows 64b..64b+63, then
//          up rows 64b..64b+63), so one 128-row GEMM tile holds matching gate and up rows.
__global__ void fold_norm_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B, int mode,
                                 int cols, const __nv_bfloat16* __restrict__ ln, __nv_bfloat16* __restrict__ out) {
  const int p = blockIdx.x;
  const __nv_bfloat16* src;
  if (mode == 0) {
    src = A + (int64_t)p * cols;
  } else {
    const int b = p / 128, w = p % 128;
    src = w < 64 ? A + (int64_t)(b * 64 + w) * cols : B + (int64_t)(b * 64 + w - 64) * cols;
  }
  for (int k = threadIdx.x; k < cols; k += blockDim.x)
    out[(int64_t)p * cols + k] = ln ? __float2bfloat16_rn(__bfloat162float(src[k]) * __bfloat162float(ln[k])) : src[k];
}

// x (fp32) -> [hi | lo] bf16 with hi = bf16(x), lo = bf16(x - hi): a GEMM that multiplies
// every weight tile by both halves into one accumulator then sees x to ~16 mantissa bits.
__global__ void split_hi_lo_kernel(const float* __restrict__ x, int n, __nv_bfloat16* __restrict__ out) {
  const float* xr = x + (int64_t)blockIdx.x * n;
  __nv_bfloat16* o = out + (int64_t)blockIdx.x * 2 * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float v = xr[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    o[i] = hi;
    o[n + i] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
}

}  // namespace

cudaError_t launch_split_hi_lo(const float* x, int rows, int n, void* out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  split_hi_lo_kernel<<<rows, 256, 0, st>>>(x, n, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_embed_tc(const dflash_handle* h, const int32_t* bonus, int nb, cudaStream_t st) {
  const dflash_cfg& c = h->cfg;
  embed_tc_kernel<<<nb * kGamma, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(h->embed), bonus, c.mask_token_id,
                                               c.vocab, c.hidden, h->rows_max,
                                               static_cast<const __nv_bfloat16*>(h->layer[0].ln_in), h->x,
                                               static_cast<__nv_bfloat16*>(h->xb), h->ss_b, h->d_status,
                                               h->cur_widths);
  return cudaGetLastError();
}

cudaError_t launch_fold_norm(const void* A, const void* B, int mode, int rows, int cols, const void* ln, void* out,
                             cudaStream_t st) {
  fold_norm_kernel<<<rows, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B),
                                         mode, cols, static_cast<const __nv_bfloat16*>(ln),
                                         static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ launchers

#define DISPATCH_T(dtype, ...)                                  \
  do {                                                          \
    if ((dtype) == DFLASH_F32) {                                \
      using T = float;                                          \
      __VA_ARGS__;                                              \
    } else {                                                    \
      using T = __nv_bfloat16;                                  \
      __VA_ARGS__;                                              \
    }                                                           \
  } while (0)

cudaError_t launch_embed(const dflash_handle* h, const int32_t* bonus, int nb, float* x, cudaStream_t st) {
  const dflash_cfg& c = h->cfg;
  DISPATCH_T(c.dtype, embed_kernel<T><<<nb * kGamma, 256, 0, st>>>(static_cast<const T*>(h->embed), bonus,
                                                                     c.mask_token_id, c.vocab, c.hidden, x,
                                                                     h->d_status, h->cur_widths));
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_f32in(const dflash_handle* h, const float* x, const void* w, void* out, int rows,
                                 int n, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  DISPATCH_T(h->cfg.dtype, rmsnorm_kernel<T><<<rows, 256, 0, st>>>(x, static_cast<const T*>(w),
                                                                  static_cast<T*>(out), n, h->cfg.rms_eps));
  return cudaGetLastError();
}

cudaError_t launch_gemm(const dflash_handle* h, const void* X, int ldx, const void* W, int M, int N, int K,
                        float* Y, int ldy, bool accumulate, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  DISPATCH_T(h->cfg.dtype, (gemm_kernel<T, T, false><<<grid, 256, 0, st>>>(static_cast<const T*>(X), ldx, W, nullptr,
                                                                           M, N, K, Y, ldy, accumulate ? 1 : 0)));
  return cudaGetLastError();
}

cudaError_t launch_gemm_xf32(const dflash_handle* h, const float* X, int ldx, const void* W, int M, int N, int K,
                             float* Y, int ldy, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  DISPATCH_T(h->cfg.dtype, (gemm_kernel<float, T, false><<<grid, 256, 0, st>>>(X, ldx, W, nullptr, M, N, K, Y, ldy, 0)));
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_f32out(const dflash_handle* h, const float* x, const void* w, float* out, int rows, int n,
                                  cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  DISPATCH_T(h->cfg.dtype, (rmsnorm_kernel<T, float><<<rows, 256, 0, st>>>(x, static_cast<const T*>(w), out, n,
                                                                          h->cfg.rms_eps)));
  return cudaGetLastError();
}

cudaError_t launch_gemm_fp8w(const dflash_handle* h, const void* X, int ldx, const uint8_t* Wq, const float* scale,
                             int M, int N, int K, float* Y, int ldy, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  DISPATCH_T(h->cfg.dtype, (gemm_kernel<T, T, true><<<grid, 256, 0, st>>>(static_cast<const T*>(X), ldx, Wq, scale,
                                                                          M, N, K, Y, ldy, 0)));
  return cudaGetLastError();
}

cudaError_t launch_qkv_post(const dflash_handle* h, int layer, const float* y, const int32_t* ctx_lens,
                            const int32_t* page_tables, int nb, void* q, cudaStream_t st) {
  const dflash_cfg& c = h->cfg;
  const int nheads = c.n_q_heads + 2 * c.n_kv_heads;
  dim3 grid(nb * kGamma, nheads);
  const int ldy = nheads * c.head_dim;
  DISPATCH_T(c.dtype, qkv_post_kernel<T><<<grid, c.head_dim, c.head_dim * sizeof(float), st>>>(
                          y, ldy, static_cast<const T*>(h->layer[layer].q_norm),
                          static_cast<const T*>(h->layer[layer].k_norm), h->rope_inv_pi, h->rope_mscale, c.rms_eps,
                          c.n_q_heads, c.n_kv_heads, c.head_dim, ctx_lens, page_tables, c.max_pages_per_seq,
                          h->geom, layer, static_cast<T*>(h->pool), static_cast<T*>(q), h->d_status,
                          h->cur_rope_pos));
  return cudaGetLastError();
}

cudaError_t launch_attention(const dflash_handle* h, int layer, const void* q, const int32_t* ctx_lens,
                             const int32_t* page_tables, int nb, int max_ctx_len, void* out, cudaStream_t st) {
  const dflash_cfg& c = h->cfg;
  const int rows = nb * kGamma;
  const int warps = rows * c.n_q_heads;
  const int window = c.layer_sliding[layer] ? c.sliding_window : 0;
  DISPATCH_T(c.dtype, attention_kernel<T><<<(warps + 3) / 4, 128, 0, st>>>(
                          static_cast<const T*>(q), static_cast<const T*>(h->pool), h->geom, layer, ctx_lens,
                          page_tables, c.max_pages_per_seq, max_ctx_len, rows, c.n_q_heads, c.n_kv_heads,
                          c.head_dim, window, static_cast<T*>(out), h->d_status, h->cur_widths));
  return cudaGetLastError();
}

cudaError_t launch_silu_mul(const dflash_handle* h, const float* y, int rows, void* act, cudaStream_t st) {
  const int F = h->cfg.n_ff;
  const int64_t n = (int64_t)rows * F;
  DISPATCH_T(h->cfg.dtype, silu_mul_kernel<T><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(y, 2 * F, F, rows,
                                                                                         static_cast<T*>(act)));
  return cudaGetLastError();
}

cudaError_t launch_argmax(const dflash_handle* h, const float* logits32, int nb, int32_t* drafts, void* logits_out,
                          cudaStream_t st) {
  DISPATCH_T(h->cfg.dtype, argmax_kernel<T><<<nb * kGamma, 1024, 0, st>>>(logits32, h->cfg.vocab, drafts,
                                                                         static_cast<T*>(logits_out), h->cur_widths));
  return cudaGetLastError();
}

cudaError_t launch_copy_hidden(const dflash_handle* h, const void* src, int rows, void* dst, cudaStream_t st) {
  return cudaMemcpyAsync(dst, src, (size_t)rows * h->cfg.hidden * h->esz, cudaMemcpyDeviceToDevice, st);
}

cudaError_t launch_ctxkv_post(const dflash_handle* h, const float* ykv, int n, const int32_t* positions,
                              const int32_t* page_table, int first, cudaStream_t st, const int32_t* row_seq,
                              const int32_t* row_index, int nseq) {
  const dflash_cfg& c = h->cfg;
  if (n <= 0) return cudaSuccess;
  dim3 grid(n, c.n_layers * 2 * c.n_kv_heads);
  const int ldy = c.n_layers * 2 * c.n_kv_heads * c.head_dim;
  DISPATCH_T(c.dtype, ctxkv_post_kernel<T><<<grid, c.head_dim, c.head_dim * sizeof(float), st>>>(
                          ykv, ldy, static_cast<const T*>(h->kn_all), h->rope_inv_pi, h->rope_mscale, c.rms_eps,
                          c.n_kv_heads, c.head_dim, positions, page_table, first, h->geom,
                          static_cast<T*>(h->pool), h->d_status, row_seq, row_index, nseq, c.max_pages_per_seq));
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const void* w, int rows, int cols, int dtype, uint8_t* codes, float* scale,
                                cudaStream_t st) {
  DISPATCH_T(dtype, quantize_fp8_kernel<T><<<rows, 256, 0, st>>>(static_cast<const T*>(w), cols, codes, scale));
  return cudaGetLastError();
}

}  // namespace dflash
