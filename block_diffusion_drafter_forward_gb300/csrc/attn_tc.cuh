// Host interface of the tensor-core paged block attention (attn_tc.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash_internal.cuh"

namespace dflash {

struct AttnParams {
  const __nv_bfloat16* q = nullptr;      // [nb*16, nh*128] queries (q_norm + RoPE applied)
  const __nv_bfloat16* pool = nullptr;   // paged K/V pool
  PoolGeom g{};
  int layer = 0;
  const int32_t* ctx_lens = nullptr;     // [nb]
  const int32_t* widths = nullptr;       // [nb] active block widths (null: gamma)
  const int32_t* page_tables = nullptr;  // [nb, mpps]
  int mpps = 0, nh = 0, nkv = 0, window = 0, max_ctx = 0;
  int nb = 0;                            // sequences (set by launch_attn_tc)
  int chunks_per_split = 1;              // compact kernel: key chunks per split
  float* o_part = nullptr;               // [slots, 128, 128] split partials
  float* ml_part = nullptr;              // [slots, 128, 2] running max / sum
  __nv_bfloat16* out = nullptr;          // [nb*16, nh*128]
  unsigned* status = nullptr;
};

// Split-partial slots that cover any launch with at most max_units (sequence, kv head) units.
int64_t attn_tc_partial_slots(int num_sms, int max_units);
cudaError_t launch_attn_tc(AttnParams p, int nb, int max_ctx_len, int num_sms, cudaStream_t st);

}  // namespace dflash
