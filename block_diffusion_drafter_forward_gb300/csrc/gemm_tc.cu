// Weight-streaming projection GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// with the drafter's per-projection epilogues fused in.
//
// Orientation ("swap AB"): the weight W [N, K] is the A operand, so 128 weight rows fill
// the UMMA M = 128 dimension, and the TN (16..128) token rows of the activation X [M, K]
// are the N dimension.  The accumulator tile D[n, m] sits in TMEM, one weight row per
// TMEM lane.  Tiles are staged by TMA (128-byte swizzle) through an mbarrier ring;
// weights are requested before the programmatic-dependent-launch wait, so a kernel
// streams its weights while its predecessor in the stream is still finishing.
// Split-K: each split writes fp32 partials, the last split of a tile (atomic counter)
// sums them in split order (deterministic) and runs the epilogue.  Wide token tiles run the
// epilogue's 16-token chunks on 2 or 4 warpgroups side by side.
//
// Epilogues (memra-engine `dflash.rs` forward_round; spark_model `dflash_head` pages):
//   EPI_STORE : out[m, n] = r_m * D                       (plain projection, fp32 out)
//   EPI_QKV   : one tile = one head of the fused q|k|v projection.  r_m * D (the
//               operand is x * ln_in in bf16, r_m = 1/RMS(x_m), so r_m D = W RMSNorm(x));
//               q/k: per-head RMSNorm (q_norm/k_norm), RoPE at ctx_len + r, * mscale;
//               q -> q buffer, k/v -> paged pool rows ctx_len..ctx_len+15 (block K/V).
//   EPI_RESID : x[m, n] += D (o_proj / down_proj residual), bf16(x * ln_next) as the next
//               projection's operand, per-tile partial sums of x^2 for the next RMSNorm.
//   EPI_GATEUP: tile = 64 gate rows + 64 up rows; act = silu(r_m g) * (r_m u).
//   EPI_LMHEAD: logits (optional, bf16), per-row fp32 scale for the FP8 head, each tile's
//               per-token best (logit, index) folded in with a 64-bit atomicMax; the last
//               tile turns them into drafts.
//   With e4m3 layer weights (FP8A, from_weights.rs Phase G) the QKV / RESID / GATEUP tiles take
//   D times the weight row's fp32 scale before their epilogue.
//   EPI_CTXKV : context-K/V writer (dflash.rs ingest_ctx): tile = one head of one layer's
//               K or V; K gets k_norm, RoPE at the row's position and mscale; both are
//               scattered to the row's paged slot.  The fp32 operand comes as bf16 hi + lo
//               (see below).
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <float.h>

#include <mutex>

#include "dflash_internal.cuh"
#include "gemm_epi.cuh"
#include "gemm_tc.cuh"
#include "launch_util.cuh"
#include "tc_common.cuh"

namespace dflash {
namespace {

using namespace tc;

// EPI_CTXKV (the context-K/V writer) takes its fp32 activations as a bf16 pair: X holds
// [hi | lo] along K (ldx = 2K) and every weight tile is multiplied by both halves into the
// same accumulator, so the weight is read once while the product keeps the fp32 operand.
// FP8A: the weight arrives as e4m3 codes (TMA, 64-byte rows) and warps 2-3 widen each
// stage to the bf16 128-byte-swizzled A tile before the MMA reads it (the per-row scale is
// applied in the epilogue), so the activations stay bf16 (weight-only FP8).
// WG epilogue warpgroups: wide token tiles hand their 16-token chunks round-robin to WG
// groups of 4 warps, so the latency-bound per-chunk epilogues run side by side (warps
// 4k..4k+3 read the same TMEM lanes as warps 0-3).  With WG <= 2 two CTAs fit on an SM.
template <int EPI, int TN, int STAGES, bool FP8A, int WG>
__global__ void __launch_bounds__(kThreads * WG, WG <= 2 ? 2 : 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const GemmParams p) {
  constexpr int A_BYTES = 128 * 64 * 2;
  constexpr int B_BYTES = TN * 64 * 2;
  constexpr int A8_BYTES = FP8A ? 128 * 64 : 0;
  constexpr bool HILO = EPI == EPI_CTXKV;
  constexpr int NB = HILO ? 2 : 1;  // activation tiles per stage
  constexpr int STAGE_BYTES = A_BYTES + NB * B_BYTES + A8_BYTES;
  constexpr uint32_t LOAD_BYTES = (FP8A ? A8_BYTES : A_BYTES) + NB * B_BYTES;
  constexpr int W_OFF = FP8A ? A_BYTES + B_BYTES : 0;  // where the TMA puts the weight tile
  constexpr uint32_t TMEM_COLS = TN < 32 ? 32 : TN;
  static_assert(WG * sizeof(EpiSmem) <= STAGES * STAGE_BYTES, "epilogue scratch must fit in the stages");
  static_assert(sizeof(EpiSmem) % 16 == 0, "epilogue scratch alignment");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);  // barriers: 1 KB, then EpiSmem
  uint64_t* empty = full + STAGES;
  uint64_t* conv = empty + STAGES;   // FP8A: widened A tile ready (64 arrivals)
  uint64_t* accf = conv + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] timed out, [1] last split

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int tile_m = blockIdx.x, tile_n = blockIdx.y, split = blockIdx.z;
  const int kb0 = (int)((int64_t)split * p.nkb / p.nsplit);
  const int kb1 = (int)((int64_t)(split + 1) * p.nkb / p.nsplit);
  const int nloc = kb1 - kb0;

  if (t == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&conv[s], 64);
    }
    mbar_init(accf, 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX);
  }
  if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      const int pre = nloc < STAGES ? nloc : STAGES;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], LOAD_BYTES);
        tma_load_2d(smem + i * STAGE_BYTES + W_OFF, &tmW, &full[i], (kb0 + i) * 64, tile_n * 128, pol_w);
      }
      pdl_wait();  // everything the previous kernel wrote is visible from here on
      for (int i = 0; i < pre; ++i) {
        tma_load_2d(smem + i * STAGE_BYTES + A_BYTES, &tmX, &full[i], (kb0 + i) * 64, tile_m * TN, pol_x);
        if constexpr (HILO)
          tma_load_2d(smem + i * STAGE_BYTES + A_BYTES + B_BYTES, &tmX, &full[i], p.K + (kb0 + i) * 64, tile_m * TN,
                      pol_x);
      }
      for (int i = pre; i < nloc; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(&empty[s], ((i / STAGES) - 1) & 1)) {
          flags[0] = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], LOAD_BYTES);
        tma_load_2d(smem + s * STAGE_BYTES + W_OFF, &tmW, &full[s], (kb0 + i) * 64, tile_n * 128, pol_w);
        tma_load_2d(smem + s * STAGE_BYTES + A_BYTES, &tmX, &full[s], (kb0 + i) * 64, tile_m * TN, pol_x);
        if constexpr (HILO)
          tma_load_2d(smem + s * STAGE_BYTES + A_BYTES + B_BYTES, &tmX, &full[s], p.K + (kb0 + i) * 64, tile_m * TN,
                      pol_x);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer (single thread)
      constexpr uint32_t idesc = idesc_bf16(128, TN);
      for (int i = 0; i < nloc; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(FP8A ? &conv[s] : &full[s], (i / STAGES) & 1)) {
          flags[0] = 1;
          break;
        }
        tc_fence_after();
        const uint64_t ad = desc_sw128(smem + s * STAGE_BYTES);
        const uint64_t bd = desc_sw128(smem + s * STAGE_BYTES + A_BYTES);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (i > 0 || k > 0) ? 1u : 0u);
        if constexpr (HILO) {
          const uint64_t bl = desc_sw128(smem + s * STAGE_BYTES + A_BYTES + B_BYTES);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_bf16(tmem, ad + 2 * k, bl + 2 * k, idesc, 1u);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(accf);
    }
    __syncwarp();
  } else if (FP8A && warp < 4) {
    // ---------------- e4m3 -> bf16 widening (warps 2-3): thread ct owns rows ct, ct + 64
    const int ct = t - 64;
    for (int i = 0; i < nloc; ++i) {
      const int s = i % STAGES;
      if (!mbar_wait(&full[s], (i / STAGES) & 1)) {
        flags[0] = 1;
        mbar_arrive(&conv[s]);
        break;
      }
      const uint8_t* a8 = smem + s * STAGE_BYTES + W_OFF;
      uint8_t* a = smem + s * STAGE_BYTES;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = ct + rr * 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = *reinterpret_cast<const uint4*>(a8 + row * 64 + q * 16);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(
                  (__nv_fp8x2_storage_t)((w[e] >> (16 * hf)) & 0xFFFFu), __NV_E4M3);
              const __half2 hh = *reinterpret_cast<const __half2*>(&h2);
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(__low2float(hh), __high2float(hh));
              o[e * 2 + hf] = *reinterpret_cast<const uint32_t*>(&b2);
            }
          }
          // 16 codes -> two 16-byte chunks (8 bf16 each) of the 128-byte swizzled row
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int chunk = q * 2 + cc;
            *reinterpret_cast<uint4*>(a + row * 128 + ((chunk ^ (row & 7)) * 16)) =
                make_uint4(o[cc * 4 + 0], o[cc * 4 + 1], o[cc * 4 + 2], o[cc * 4 + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&conv[s]);
    }
    __syncwarp();
  }

  // ---------------- epilogue: every warpgroup (et = row of the tile, wg = its group)
  pdl_wait();
  const int et = t & (kThreads - 1), wg = t / kThreads;
  // the exchange scratch aliases the drained stages; the row scales (needed while the
  // stages are still filling) sit after the barriers
  EpiSmem& es = *reinterpret_cast<EpiSmem*>(smem + wg * sizeof(EpiSmem));
  float* const rsc = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256);
  if (p.ss_in && warp >= 2 && warp < 4) {
    // input row scales 1/RMS(x_m) from the producer's per-128-column partials, computed by
    // the warps that are idle during the mainloop
    for (int c = t - 64; c < TN; c += 64) {
      const int m = m0_of(tile_m, TN) + c;
      float r = 1.f;
      if (m < p.M) {
        float part[8];
        float ssum = 0.f;
        for (int q0 = 0; q0 < p.ss_parts; q0 += 8) {
#pragma unroll
          for (int u = 0; u < 8; ++u) part[u] = q0 + u < p.ss_parts ? __ldcg(p.ss_in + (int64_t)(q0 + u) * p.Mp + m) : 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u) ssum += part[u];
        }
        r = 1.f / sqrtf(ssum / (float)p.ss_n + p.eps);
      }
      rsc[c] = r;
    }
  }
  const bool ok = mbar_wait(accf, 0);
  tc_fence_after();
  __syncthreads();
  if (!ok || flags[0]) {
    // a wait gave up: record it, give copies still in flight time to land, unwind
    if (t == 0) set_status(p.status, DFLASH_DEV_TIMEOUT);
    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
  } else {
    const int m0 = tile_m * TN;
    const int n = tile_n * 128 + et;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int64_t tile_lin = (int64_t)tile_n * gridDim.x + tile_m;
    bool last = true;
    if (p.nsplit > 1) {
      float* mine = p.ws + ((tile_lin * p.nsplit + split) * kThreads + et) * TN;
#pragma unroll 1
      for (int c0 = wg * 16; c0 < TN; c0 += 16 * WG) {
        float v[16];
        tmem_ld16(lane_addr + c0, v);
#pragma unroll
        for (int c = 0; c < 16; c += 4)
          __stcg(reinterpret_cast<float4*>(mine + c0 + c), make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]));
      }
      __threadfence();
      __syncthreads();
      if (t == 0) flags[1] = atomicAdd(&p.counters[tile_lin], 1u) == (unsigned)(p.nsplit - 1);
      __syncthreads();
      last = flags[1] != 0;
      if (last) __threadfence();
    }
    if (last) {
#pragma unroll 1
      for (int c0 = wg * 16; c0 < TN; c0 += 16 * WG) {
        EpiPre pre;  // inputs first, so their loads overlap the partials' loads
        epilogue_pre<EPI>(p, pre, et, n, m0, c0, tile_n);
        float v[16];
        if (p.nsplit > 1) {
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] = 0.f;
          for (int s0 = 0; s0 < p.nsplit; s0 += 4) {
            float4 q4[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float* src = p.ws + ((tile_lin * p.nsplit + (s0 + u)) * kThreads + et) * TN + c0;
#pragma unroll
              for (int c = 0; c < 4; ++c)
                q4[u][c] = s0 + u < p.nsplit ? __ldcg(reinterpret_cast<const float4*>(src) + c)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                v[4 * c] += q4[u][c].x;
                v[4 * c + 1] += q4[u][c].y;
                v[4 * c + 2] += q4[u][c].z;
                v[4 * c + 3] += q4[u][c].w;
              }
            }
          }
        } else {
          tmem_ld16(lane_addr + c0, v);
        }
        if constexpr (FP8A && EPI != EPI_LMHEAD) {
          // e4m3 layer weight: this row's fp32 scale (the lm_head applies its own in the epilogue)
          const float sc = __ldg(p.row_scale + n);
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] *= sc;
        }
        epilogue_chunk<EPI>(p, es, rsc, v, et, n, m0, c0, tile_n, pre);
      }
      if (p.nsplit > 1 && t == 0) p.counters[tile_lin] = 0;
      if constexpr (EPI == EPI_LMHEAD) {
        // the last vocabulary tile of this token tile reduces the per-tile argmaxes
        __threadfence();
        __syncthreads();
        if (t == 0) flags[1] = atomicAdd(&p.amax_counter[tile_m], 1u) == (unsigned)(gridDim.y - 1);
        __syncthreads();
        if (flags[1]) {
          // every vocabulary tile of these tokens has folded its best into amax_best
          __threadfence();
          for (int c = t; c < TN; c += kThreads * WG) {
            const int m = m0 + c;
            if (m < p.M) {
              const unsigned long long k = atomicExch(p.amax_best + m, 0ull);  // read and re-arm
              const int r = m % kGamma;
              if (r > 0)
                p.drafts[(m / kGamma) * (kGamma - 1) + r - 1] =
                    r < block_width(p.widths, m / kGamma) ? argmax_key_index(k) : -1;
            }
          }
          if (t == 0) p.amax_counter[tile_m] = 0;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

template <int EPI, int TN, int STAGES, bool FP8A, int WG>
cudaError_t launch_t(const CUtensorMap& tw, const CUtensorMap& tx, const GemmParams& p, dim3 grid,
                     cudaStream_t st, bool pdl) {
  constexpr int smem =
      STAGES * (128 * 64 * 2 + (EPI == EPI_CTXKV ? 2 : 1) * TN * 64 * 2 + (FP8A ? 128 * 64 : 0)) + 1024 + 256 + 1024;
  auto kern = gemm_tc_kernel<EPI, TN, STAGES, FP8A, WG>;
  static std::atomic<unsigned long long> attr_set{0};
  cudaError_t ea = smem_attr_once(kern, smem, attr_set);
  if (ea != cudaSuccess) return ea;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads * WG);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tw, tx, p);
}

template <int EPI, int TN>
cudaError_t launch_tn(const CUtensorMap& tw, const CUtensorMap& tx, const GemmParams& p, dim3 grid,
                      cudaStream_t st, bool pdl, bool fp8a) {
  // stages: keep two CTAs per SM possible (grids of a little more than one CTA per SM then
  // overlap instead of running a second, nearly empty wave).  Wide tiles with split-K
  // partials to reduce take one SM each with 4 epilogue warpgroups instead.
  constexpr int STAGES = TN <= 32 ? 6 : (TN <= 64 ? 4 : 3);
  constexpr int WG = TN >= 64 ? 2 : 1;
  if constexpr (EPI == EPI_LMHEAD) {
    if (fp8a) return launch_t<EPI, TN, STAGES - 1, true, WG>(tw, tx, p, grid, st, pdl);
  }
  if constexpr (EPI == EPI_QKV || EPI == EPI_RESID || EPI == EPI_GATEUP) {  // FP8 layer weights
    if (fp8a) {
      if constexpr (TN >= 64) {
        if (p.nsplit > 1) return launch_t<EPI, TN, TN >= 128 ? 3 : 6, true, 4>(tw, tx, p, grid, st, pdl);
      }
      return launch_t<EPI, TN, STAGES - 1, true, WG>(tw, tx, p, grid, st, pdl);
    }
  }
  if constexpr (EPI == EPI_CTXKV) {  // two activation tiles per stage
    if constexpr (TN >= 128) {  // compute-heavy: two CTAs per SM rather than a deep ring
      if (p.nsplit > 1) return launch_t<EPI, TN, 4, false, 4>(tw, tx, p, grid, st, pdl);
      return launch_t<EPI, TN, 2, false, 2>(tw, tx, p, grid, st, pdl);
    }
    if constexpr (TN == 64) return launch_t<EPI, TN, 3, false, 2>(tw, tx, p, grid, st, pdl);
    return launch_t<EPI, TN, 5, false, 1>(tw, tx, p, grid, st, pdl);
  }
  if constexpr (TN >= 64) {  // split tiles: one CTA per SM, 4 warpgroups, a deep ring
    if (p.nsplit > 1) return launch_t<EPI, TN, TN >= 128 ? 4 : 8, false, 4>(tw, tx, p, grid, st, pdl);
  }
  return launch_t<EPI, TN, STAGES, false, WG>(tw, tx, p, grid, st, pdl);
}

template <int EPI>
cudaError_t launch_epi(int TN, const CUtensorMap& tw, const CUtensorMap& tx, const GemmParams& p, dim3 grid,
                       cudaStream_t st, bool pdl, bool fp8a) {
  switch (TN) {
    case 16: return launch_tn<EPI, 16>(tw, tx, p, grid, st, pdl, fp8a);
    case 32: return launch_tn<EPI, 32>(tw, tx, p, grid, st, pdl, fp8a);
    case 64: return launch_tn<EPI, 64>(tw, tx, p, grid, st, pdl, fp8a);
    case 128: return launch_tn<EPI, 128>(tw, tx, p, grid, st, pdl, fp8a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld_elems,
                    int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld_elems * 2)};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int pick_tn(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  return 128;  // larger batches: several 128-token tiles, consecutive in the grid (weight tile reuse in L2)
}

int pick_splits(int tiles, int nkb, int num_sms, int tn) {
  // about one CTA per SM; wide tiles that split run one CTA per SM (4 epilogue warpgroups),
  // so they round down rather than start a second, mostly empty wave
  int s = tn >= 64 ? num_sms / tiles : (num_sms + tiles - 1) / tiles;
  if (s > nkb) s = nkb;
  if (s > kMaxSplits) s = kMaxSplits;
  return s < 1 ? 1 : s;
}

bool make_tmap_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_gemm_tc(int epi, const void* W, int N, int K, const void* X, int ldx, int M, GemmParams p,
                           int nsplit, cudaStream_t st, bool pdl, bool w_fp8) {
  const int TN = pick_tn(M);
  CUtensorMap tw, tx;
  if (w_fp8 && (epi == EPI_STORE || epi == EPI_CTXKV)) return cudaErrorInvalidValue;
  if (w_fp8 ? !make_tmap_u8(&tw, W, N, K) : !make_tmap_bf16(&tw, W, N, K, K, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tx, X, M, epi == EPI_CTXKV ? 2 * (int64_t)K : K, ldx, TN)) return cudaErrorInvalidValue;
  p.N = N;
  p.K = K;
  p.M = M;
  p.nkb = K / 64;
  p.nsplit = nsplit;
  dim3 grid((M + TN - 1) / TN, (N + 127) / 128, nsplit);
  switch (epi) {
    case EPI_STORE: return launch_epi<EPI_STORE>(TN, tw, tx, p, grid, st, pdl, false);
    case EPI_QKV: return launch_epi<EPI_QKV>(TN, tw, tx, p, grid, st, pdl, w_fp8);
    case EPI_RESID: return launch_epi<EPI_RESID>(TN, tw, tx, p, grid, st, pdl, w_fp8);
    case EPI_GATEUP: return launch_epi<EPI_GATEUP>(TN, tw, tx, p, grid, st, pdl, w_fp8);
    case EPI_LMHEAD: return launch_epi<EPI_LMHEAD>(TN, tw, tx, p, grid, st, pdl, w_fp8);
    case EPI_CTXKV: return launch_epi<EPI_CTXKV>(TN, tw, tx, p, grid, st, pdl, false);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dflash
