// Host interface of the tensor-core projection GEMM (gemm_tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash_internal.cuh"

namespace dflash {

enum GemmEpi { EPI_STORE = 0, EPI_QKV = 1, EPI_RESID = 2, EPI_GATEUP = 3, EPI_LMHEAD = 4, EPI_CTXKV = 5 };
constexpr int kMaxSplits = 16;

// Everything an epilogue may need; fields an epilogue does not use stay zero.
struct GemmParams {
  int N = 0, K = 0, M = 0, nkb = 0, nsplit = 1;
  float* ws = nullptr;              // split-K partials
  unsigned* counters = nullptr;     // split-K tile counters (zero between launches)
  unsigned* status = nullptr;       // device status word
  // input row scale r_m = 1/sqrt(sum_q ss_in[q*Mp + m] / ss_n + eps) (nullptr: none)
  const float* ss_in = nullptr;
  int ss_parts = 0, ss_n = 1, Mp = 0;
  float eps = 1e-6f;
  // EPI_STORE
  float* out = nullptr;
  int ldo = 0;
  // EPI_QKV
  __nv_bfloat16* q = nullptr;
  const __nv_bfloat16* q_norm = nullptr;
  const __nv_bfloat16* k_norm = nullptr;
  const float2* inv_pi = nullptr;        // RoPE inv_freq / pi as (hi, lo) floats
  float mscale = 1.f;
  int nh = 0, nkv = 0, mpps = 0, layer = 0;
  const int32_t* ctx_lens = nullptr;
  const int32_t* page_tables = nullptr;
  const int32_t* rope_pos0 = nullptr;    // [nb] RoPE start of each block (null: ctx_lens)
  const int32_t* widths = nullptr;       // [nb] active block widths (null: gamma); lm_head drafts
  PoolGeom g{};
  __nv_bfloat16* pool = nullptr;
  // EPI_CTXKV (k_norm: every layer's k_norm [L, 128]).  Row m goes to row index first + m of the
  // one sequence whose table is page_tables, or, with row_seq / row_index (the batched writer),
  // to row index row_index[m] of sequence row_seq[m] (table row row_seq[m] of page_tables [nseq,
  // mpps]).
  const int32_t* positions = nullptr;
  int first = 0;
  const int32_t* row_seq = nullptr;
  const int32_t* row_index = nullptr;
  int nseq = 1;
  // EPI_RESID
  float* x = nullptr;
  __nv_bfloat16* xb = nullptr;
  float* ss_out = nullptr;
  const __nv_bfloat16* ln_next = nullptr;  // next RMSNorm weight: xb = bf16(x * ln_next)
  int H = 0;
  // EPI_GATEUP
  __nv_bfloat16* act = nullptr;
  int F = 0;
  // EPI_LMHEAD
  __nv_bfloat16* logits = nullptr;
  float* logits32 = nullptr;              // fp32 logits [M, N] as well (the Markov head reads them)
  const float* row_scale = nullptr;
  // per token row: max over vocabulary tiles of (orderable logit << 32 | ~index), combined
  // with 64-bit atomicMax (order-independent, so deterministic); zero between launches
  unsigned long long* amax_best = nullptr;
  unsigned* amax_counter = nullptr;
  int32_t* drafts = nullptr;
};

int pick_tn(int M);
// Split-K ways for `tiles` output tiles of `nkb` k-blocks with tn-token tiles.
int pick_splits(int tiles, int nkb, int num_sms, int tn);
bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld_elems, int box_rows);
// D = W [N, K] x X [M, K]^T with the epilogue `epi`; nsplit K-splits (1 for EPI_LMHEAD).
// w_fp8: W holds e4m3 codes and p.row_scale the per-row scales (EPI_LMHEAD, and the layer
// projections EPI_QKV / EPI_RESID / EPI_GATEUP of the FP8 drafter lane).
cudaError_t launch_gemm_tc(int epi, const void* W, int N, int K, const void* X, int ldx, int M, GemmParams p,
                           int nsplit, cudaStream_t st, bool pdl, bool w_fp8 = false);

}  // namespace dflash
