// Host interface of the stream-K projection GEMM (gemm_tc.cu).
#pragma once

#include "gemm_tc.cuh"

namespace dflash {
// Stream-K projection GEMM (bf16 weights, QKV / RESID / GATEUP epilogues, 128-token tiles):
// gemm_sk_grid(num_sms) CTAs, two per SM, each an equal share of the tiles x k-blocks.  Split
// tiles keep fp32 partials in p.ws slots (tile, rank): tiles * gemm_sk_max_contrib(...) *
// 128 * 128 floats, counted in p.counters[tile].  gemm_sk_eligible: the shapes it takes.
int gemm_sk_grid(int num_sms);
int gemm_sk_max_contrib(int tiles, int nkb, int G);
bool gemm_sk_eligible(int epi, int M, int N, int K, bool w_fp8, int num_sms);
cudaError_t launch_gemm_sk(int epi, const void* W, int N, int K, const void* X, int ldx, int M, GemmParams p,
                           int num_sms, cudaStream_t st, bool pdl);

}  // namespace dflash
