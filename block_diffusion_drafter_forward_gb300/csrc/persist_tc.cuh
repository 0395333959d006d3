// Host interface of the persistent single-launch propose kernel (persist_tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash_internal.cuh"

namespace dflash {

// Layers the persistent kernel takes (its per-layer table travels in the kernel parameters).
constexpr int kPersistMaxL = 32;

struct PersistLayer {
  const __nv_bfloat16* q_norm;
  const __nv_bfloat16* k_norm;
  const __nv_bfloat16* ln_in;
  const __nv_bfloat16* ln_post;
  int window;        // 0: full attention
};

struct PersistParams {
  int L, M, H, F, nh, nkv, V, mpps, mask, max_ctx, G;
  float eps, mscale;
  int attn_cps[2];      // attention: 64-key chunks per work item (full layers, windowed layers)
  int attn_splits[2];   // attention: work items per (sequence, kv head)
  const int32_t* bonus;
  const int32_t* ctx_lens;
  const int32_t* page_tables;
  const int32_t* rope_pos0;   // [nb] RoPE start of each block, or null (ctx_lens)
  const int32_t* widths;      // [nb] active block widths, or null (gamma)
  const __nv_bfloat16* embed;
  const __nv_bfloat16* norm;
  const float2* inv_pi;
  PersistLayer layers[kPersistMaxL]; // per layer (in the kernel's parameter space)
  const CUtensorMap* maps;          // [4L + 1] weights (qkv, o, gate/up, down per layer; lm_head),
                                    // then [4] activations (xb, attn, act, xb2), device, 64-B aligned
  float* x;
  __nv_bfloat16* xb;    // bf16(x * ln_in) / bf16(x * norm): operand of QKV and the lm_head
  __nv_bfloat16* xb2;   // bf16(x1 * ln_post): operand of gate/up (its own buffer, so down can
                        // write xb while a slower CTA's gate/up still reads this one)
  float* ss_a;
  float* ss_b;
  __nv_bfloat16* q;
  __nv_bfloat16* attn;
  __nv_bfloat16* act;
  __nv_bfloat16* pool;
  PoolGeom g;
  float* ws;            // split-K partials, two halves of ws_half floats used by alternate phases
  size_t ws_half;
  unsigned* counters;   // split-K tile counters, two halves of max_tiles (alternate phases)
  int max_tiles;
  unsigned long long* amax_best;    // [16] packed running argmax per token (control buffer)
  unsigned* amax_counter;
  float* o_part;
  float* ml_part;
  int32_t* drafts;
  __nv_bfloat16* logits;
  __nv_bfloat16* final_hidden;
  // One control buffer, zeroed before each launch (persist_ctl_words words):
  unsigned* bar;                    // [3 + 6L] phase arrival counters
  int* gabort;                      // grid-wide "a wait gave up" flag
  unsigned* ready;                  // [phases][ready_stride] projection tile finished (0/1)
  int ready_stride;
  unsigned* done;                   // [phases] projection tiles finished
  unsigned* head_done;              // [L][64] attention output rows of a unit written (32 = all)
  unsigned* status;
  // Phase timeline (builds with DFLASH_PHASE_TRACE=1 only; else unused and null):
  // [G][phases][kTraceSlots] %globaltimer stamps, see persist_tc.cu.
  unsigned long long* trace;
};

#ifndef DFLASH_PHASE_TRACE
#define DFLASH_PHASE_TRACE 0
#endif
constexpr int kTraceSlots = 13;

// Tokens (M = 16 * nb) the persistent kernel handles: one sequence (bf16 lm_head only); larger
// batches and the FP8 lm_head use the per-projection kernels.
constexpr int kPersistMaxM = 16;

// Shared memory and split-K workspace the persistent kernel needs; the largest hidden size.
int persist_smem_bytes();
int persist_max_hidden();
size_t persist_ws_floats(int H, int F, int nh, int nkv, int V, int num_sms);
// Control words: phase counters, abort flag, lm_head tile counter, split-K tile counters (two
// halves), per-phase tile-ready flags and counts, per-layer attention-unit counters.
size_t persist_ctl_words(int L, int H, int F, int nh, int nkv, int V);
// Point p.bar / p.gabort / p.amax_counter / p.counters / p.ready / p.done / p.head_done into
// `ctl` (p.L, p.H, p.F, p.nh, p.nkv, p.V set).
void persist_bind_ctl(PersistParams& p, unsigned* ctl);
// Attention work split for `units` (sequence, kv head) pairs over G CTAs.
void persist_attn_split(int units, int max_ctx, int window, int G, int* cps, int* splits);
// Resident CTAs of the persistent kernel per SM (1 when it can run).
cudaError_t persist_occupancy(int* per_sm);
// Launch (cooperative, one CTA per SM).  The control buffer must be zero (memset it on `st`).
cudaError_t launch_persist(const PersistParams& p, cudaStream_t st);

}  // namespace dflash
