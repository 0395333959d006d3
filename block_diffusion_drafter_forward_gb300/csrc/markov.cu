// DSpark semi-autoregressive Markov chain over the draft logits (memra-engine dflash.rs, the
// draft step of generate_spec_dflash, SEMI-AR MARKOV CHAIN block; Atlas dflash_head.rs, DSpark
// head fields markov_w1 [V, rank] and markov_w2 [V, rank]).
//
// For every band s, left to right from its bonus token:
//     chain_0 = bonus_s
//     for k = 0 .. 14:  z[s, k + 1, :] += w2 @ w1[chain_k];  chain_{k+1} = argmax z[s, k + 1, :]
// drafts[s, k] = chain_{k+1}.  The 15 steps are sequential (each bias needs the previous argmax)
// and each reads all of w2 (V x rank), so the kernel is one cooperative launch over every SM:
// CTA c owns vocabulary rows [c V / G, (c + 1) V / G) for every step and every sequence, takes
// its local argmax per sequence, folds it into one 64-bit key per (step, sequence) with
// atomicMax (order-independent, ties to the lowest id), and the CTAs meet at a bounded grid
// barrier before the next step reads the new previous tokens.  w2 (78 MB in bf16 at rank 256)
// stays in L2 after the first step.
#include <cuda_bf16.h>
#include <float.h>

#include <atomic>

#include "dflash_internal.cuh"
#include "launch_util.cuh"
#include "markov.cuh"

namespace dflash {
namespace {

constexpr int kMkThreads = 256;
constexpr long long kMkSpin = 20000000ll;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void store_logit(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_logit(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ unsigned long long mk_key(float v, int i) {
  const unsigned u = __float_as_uint(v + 0.f);
  const unsigned o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)i);
}
__device__ __forceinline__ int mk_index(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull));
}
__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 8 consecutive weights as fp32 (16-byte loads; rows are 16-byte aligned since R % 32 == 0).
__device__ __forceinline__ void load8(const float* p, float (&w)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&w)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[2 * i] = __low2float(h[i]);
    w[2 * i + 1] = __high2float(h[i]);
  }
}

constexpr int kSB = 8;  // sequences per register block

template <typename T>
__global__ void __launch_bounds__(kMkThreads, 1) markov_kernel(const __grid_constant__ MarkovParams p) {
  extern __shared__ float sf[];                 // [nb][R] fp32: w1 rows of the previous tokens
  __shared__ unsigned long long sbest[kMarkovMaxBatch];
  __shared__ int sprev[kMarkovMaxBatch];
  __shared__ int s_abort;
  const T* w1 = static_cast<const T*>(p.w1);
  const T* w2 = static_cast<const T*>(p.w2);
  T* logits = static_cast<T*>(p.logits);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int v0 = (int)((int64_t)c * p.V / G), v1 = (int)((int64_t)(c + 1) * p.V / G);
  const int R = p.R, q4 = lane & 3, seg = R / 4;   // 4 lanes per vocabulary row, R/4 weights each
  if (t == 0) s_abort = 0;
  __syncthreads();

  for (int k = 0; k < kGamma - 1; ++k) {
    if (t < p.nb) {
      int prev;
      if (k + 1 >= block_width(p.widths, t)) {
        prev = -2;                               // past the sequence's block width: idle
      } else {
        if (k == 0) {
          prev = __ldg(p.bonus + t);
        } else {
          const unsigned long long key = ld_acquire64(p.best + (size_t)(k - 1) * p.nb + t);
          prev = key ? mk_index(key) : -1;
        }
        if (prev < 0 || prev >= p.V) {
          if (c == 0) atomicOr(p.status, DFLASH_DEV_BAD_TOKEN);
          prev = -1;                             // its bias is taken as zero
        }
      }
      sprev[t] = prev;
      sbest[t] = 0ull;
    }
    __syncthreads();
    for (int i = t; i < p.nb * R; i += kMkThreads) {
      const int s = i / R, j = i - s * R;
      sf[i] = sprev[s] >= 0 ? to_f(w1[(int64_t)sprev[s] * R + j]) : 0.f;  // (a bad token: zero bias)
    }
    __syncthreads();
    for (int s0 = 0; s0 < p.nb; s0 += kSB) {
      const int ns = min(kSB, p.nb - s0);
      unsigned long long best[kSB];
#pragma unroll
      for (int s = 0; s < kSB; ++s) best[s] = 0ull;
      // rows: 8 per warp pass, 4 lanes each
      for (int vb = v0 + warp * 8; vb < v1; vb += (kMkThreads / 32) * 8) {
        const int v = vb + (lane >> 2);
        const bool ok = v < v1;
        const T* wr = w2 + (int64_t)(ok ? v : v0) * R + q4 * seg;
        float acc[kSB];
#pragma unroll
        for (int s = 0; s < kSB; ++s) acc[s] = 0.f;
        for (int j0 = 0; j0 < seg; j0 += 8) {
          float w[8];
          load8(wr + j0, w);
#pragma unroll
          for (int s = 0; s < kSB; ++s) {
            if (s < ns) {
              const float4* f4 = reinterpret_cast<const float4*>(sf + (s0 + s) * R + q4 * seg + j0);
              const float4 a = f4[0], b = f4[1];
              acc[s] = fmaf(w[0], a.x, fmaf(w[1], a.y, fmaf(w[2], a.z, fmaf(w[3], a.w, acc[s]))));
              acc[s] = fmaf(w[4], b.x, fmaf(w[5], b.y, fmaf(w[6], b.z, fmaf(w[7], b.w, acc[s]))));
            }
          }
        }
#pragma unroll
        for (int s = 0; s < kSB; ++s) {
          float a = acc[s];
          a += __shfl_xor_sync(0xffffffffu, a, 1);
          a += __shfl_xor_sync(0xffffffffu, a, 2);
          if (s < ns && ok && q4 == 0 && sprev[s0 + s] != -2) {
            const int64_t row = (int64_t)((s0 + s) * kGamma + k + 1) * p.V + v;
            const float z = __ldcg(p.z + row) + a;
            if (logits) store_logit(logits + row, z);
            const unsigned long long key = mk_key(z, v);
            if (key > best[s]) best[s] = key;
          }
        }
      }
      // the CTA's best per sequence: warp maximum, then one shared atomic per warp
#pragma unroll
      for (int s = 0; s < kSB; ++s) {
        unsigned long long b = best[s];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long ob = __shfl_xor_sync(0xffffffffu, b, o);
          b = ob > b ? ob : b;
        }
        if (lane == 0 && s < ns && b) atomicMax(&sbest[s0 + s], b);
      }
    }
    __syncthreads();
    if (t < p.nb && sbest[t]) {
      atomicMax(p.best + (size_t)k * p.nb + t, sbest[t]);
      __threadfence();
    }
    // grid barrier (bounded): every CTA's keys of step k are in before step k + 1 reads them
    __syncthreads();
    if (t == 0) {
      __threadfence();
      atomicAdd(p.bar + k, 1u);
      long long spin = 0;
      while (ld_acquire32(p.bar + k) < (unsigned)G) {
        if (++spin > kMkSpin || *reinterpret_cast<volatile int*>(p.gabort)) {
          atomicExch(p.gabort, 1);
          s_abort = 1;
          break;
        }
        __nanosleep(64);
      }
    }
    __syncthreads();
    if (s_abort) break;
  }
  if (t == 0 && s_abort) atomicOr(p.status, DFLASH_DEV_TIMEOUT);
  if (c == 0 && !s_abort) {
    for (int i = t; i < p.nb * (kGamma - 1); i += kMkThreads) {
      const int s = i / (kGamma - 1), k = i - s * (kGamma - 1);
      const unsigned long long key = ld_acquire64(p.best + (size_t)k * p.nb + s);
      p.drafts[i] = k + 1 < block_width(p.widths, s) ? (key ? mk_index(key) : 0) : -1;
    }
  }
}

std::atomic<unsigned long long> g_mk_attr_f32{0}, g_mk_attr_bf16{0};

}  // namespace

size_t markov_smem_bytes(int nb, int R) { return (size_t)nb * R * sizeof(float); }

size_t markov_ctl_bytes(int nb) {
  return (size_t)(kGamma - 1) * nb * sizeof(unsigned long long) + 64 * sizeof(unsigned);
}

void markov_bind_ctl(MarkovParams& p, void* ctl, int nb) {
  p.best = static_cast<unsigned long long*>(ctl);
  unsigned* w = reinterpret_cast<unsigned*>(p.best + (size_t)(kGamma - 1) * nb);
  p.bar = w;
  p.gabort = reinterpret_cast<int*>(w + 32);
}

cudaError_t markov_occupancy(int dtype, int nb, int R, int* per_sm) {
  const int smem = (int)markov_smem_bytes(nb, R);
  if (dtype == DFLASH_F32) {
    if (cudaError_t e = smem_attr_once(markov_kernel<float>, kMarkovMaxSmem, g_mk_attr_f32); e != cudaSuccess)
      return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, markov_kernel<float>, kMkThreads, smem);
  }
  if (cudaError_t e = smem_attr_once(markov_kernel<__nv_bfloat16>, kMarkovMaxSmem, g_mk_attr_bf16); e != cudaSuccess)
    return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, markov_kernel<__nv_bfloat16>, kMkThreads, smem);
}

cudaError_t launch_markov(int dtype, const MarkovParams& p, int G, cudaStream_t st) {
  const int smem = (int)markov_smem_bytes(p.nb, p.R);
  int per_sm = 0;
  if (cudaError_t e = markov_occupancy(dtype, p.nb, p.R, &per_sm); e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kMkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the step barrier needs it
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (dtype == DFLASH_F32) return cudaLaunchKernelEx(&cfg, markov_kernel<float>, p);
  return cudaLaunchKernelEx(&cfg, markov_kernel<__nv_bfloat16>, p);
}

}  // namespace dflash
