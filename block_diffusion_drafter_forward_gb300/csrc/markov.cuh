// Host interface of the DSpark Markov-chain kernel (markov.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dflash {

// Sequences and rank the Markov kernel takes (its per-sequence state lives in shared memory).
constexpr int kMarkovMaxBatch = 64;
constexpr int kMarkovMaxRank = 1024;
constexpr int kMarkovMaxSmem = 160 * 1024;

struct MarkovParams {
  const float* z;               // [nb * 16, V] fp32 logits of the block rows (rows 1..15 read)
  const void* w1;               // [V, R] previous-token table (cfg.dtype)
  const void* w2;               // [V, R] projection to the vocabulary (cfg.dtype)
  int V, R, nb;
  const int32_t* bonus;         // [nb] chain starts
  const int32_t* widths;        // [nb] active block widths (null: gamma): b - 1 steps each
  int32_t* drafts;              // [nb, 15] out
  void* logits;                 // [nb * 16, V] cfg.dtype out or null: rows 1..15 adjusted
  unsigned long long* best;     // [15][nb] per-step argmax keys (control buffer, zeroed)
  unsigned* bar;                // [15] step barriers (control buffer, zeroed)
  int* gabort;                  // a barrier wait gave up (control buffer, zeroed)
  unsigned* status;             // device status word
};

size_t markov_smem_bytes(int nb, int R);
// Control buffer (memset to zero before every launch) and its binding into the parameters.
size_t markov_ctl_bytes(int nb);
void markov_bind_ctl(MarkovParams& p, void* ctl, int nb);
cudaError_t markov_occupancy(int dtype, int nb, int R, int* per_sm);
// Cooperative launch over G CTAs (one per SM).
cudaError_t launch_markov(int dtype, const MarkovParams& p, int G, cudaStream_t st);

}  // namespace dflash
