// The whole bf16 gamma-block forward for one small batch (16 tokens) in ONE persistent
// kernel: one CTA per SM, resident for the entire forward (cooperative launch).
//
// Why: at batch 1 each projection streams 17-50 MB of weights (2.5-7.4 us at HBM speed), but
// as separate kernels every projection also pays grid completion, launch and activation-load
// latency on the dependency chain.  Here the phases of the forward
//     embed | per layer: QKV, attention, split combine, o_proj, gate/up, down | lm_head
// run back to back inside one launch and the weight-tile producer runs ahead of them: weights
// depend on nothing, so the next projection's weights stream while the current phase finishes.
// Between consecutive projections there is no grid-wide barrier: k-block kb of a projection's
// operand comes from one tile of the projection before it (down -> QKV and lm_head, o_proj ->
// gate/up: the 128-column tile kb / 2; gate/up -> down: tile kb) or from one attention unit
// (combine -> o_proj), so the activation producer waits for that tile's ready flag only, and
// the MMAs of a projection run while the previous projection's slowest split-K finishers are
// still reducing.  Epilogues that need whole rows (1/RMS of their operand) wait for the count of
// the previous projection's finished tiles instead.  Two buffers are doubled for this: the bf16
// operand written by o_proj (read by gate/up) is not the one written by down (read by QKV and
// lm_head), and alternate phases use alternate halves of the split-K partials and counters.
// Embed -> QKV(0), QKV -> attention and attention -> combine keep grid-wide arrival counters.  The final RMSNorm is
// folded into the last down projection's epilogue (operand bf16(x * norm), per-token 1/RMS
// applied to the logits) the same way every other norm of the forward is.
//
// Roles (224 threads):
//   warp 4 lane 0: weight TMA producer (runs ahead, bounded by the smem ring)
//   warp 5 lane 0: tcgen05.mma issuer (double-buffered TMEM accumulators)
//   warp 6 lane 0: activation TMA producer (waits for the phase the activation comes from)
//   warps 0-3:     epilogues (gemm_epi.cuh), block attention, split combine, embedding
// Every projection is split evenly over the CTAs by k-blocks (stream-K): CTA c owns k-blocks
// [c T/G, (c+1) T/G) of the T = tiles x k-blocks of the projection.  A tile covered by several
// CTAs is finished by the one holding its first k-blocks (for that CTA it is always its last
// segment, so every CTA writes its partials before it reduces anything): the others store
// fp32 partials and count them in; it adds them to its own in CTA order (deterministic).
// The arithmetic of every phase is the same as the per-projection kernels'.
#include <cudaTypedefs.h>
#include <float.h>

#include <algorithm>
#include <atomic>

#include "dflash_internal.cuh"
#include "gemm_epi.cuh"
#include "gemm_tc.cuh"
#include "launch_util.cuh"
#include "persist_tc.cuh"
#include "tc_common.cuh"

namespace dflash {
namespace {

using namespace tc;

constexpr int TN = 16;                        // tokens: one accumulator chunk
constexpr int kS = 6;                         // ring stages
constexpr int kAB = 128 * 64 * 2;             // weight tile (bf16, 128 rows x 64 k)
constexpr int kBB = TN * 64 * 2;              // activation tile
constexpr int kStage = kAB + kBB;
constexpr int kRing = kS * kStage;
// attention region: the epilogue scratch, then Q and two K/V stages; Q and the K/V stages
// double as the landing buffer of split-K partials during projection phases
constexpr int kAKC = 64, kAPages = 4, kATile = 4096;
constexpr int kAP = 128 * kAKC * 2, kAQ = 128 * 128 * 2, kAKVStage = 2 * kAPages * kATile;
constexpr int kAttn = kAP + kAQ + 2 * kAKVStage;
constexpr int kPartBytes = 128 * TN * 4;                     // one contributor's partial tile
constexpr int kRedMax = (kAQ + 2 * kAKVStage) / kPartBytes;  // partials that fit at once
constexpr int kBarOff = kRing + kAttn;

constexpr int kSmemP = kBarOff + 512 + 256 + 1024;
constexpr uint32_t kAccCols = 32;             // per accumulator buffer (16 used)
constexpr uint32_t kTS = 128, kTO = 256;      // attention S/P and O columns (128 each)
constexpr uint32_t kTmemCols = 512;
constexpr long long kGridSpin = 20000000ll;   // polls of a phase counter before giving up
constexpr int kEThreads = 128;
constexpr int kBlockThreads = 224;
constexpr int kMaxHGroups = 48;               // H / 128 the final-hidden pass holds in registers

static_assert(sizeof(EpiSmem) <= kAP, "epilogue scratch overflows its area");

struct Bars {
  uint64_t full[kS], empty[kS];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t kv_full[2], s_done, o_done, red_full;
  uint32_t tmem;
  volatile int abort;
  int flag;
  int ctx0;  // context length of the (single) sequence
};
static_assert(sizeof(Bars) <= 512, "barrier block overflows its slot");

enum { PH_EMBED, PH_GEMM, PH_ATTN, PH_COMB };

__device__ __forceinline__ int phase_kind(int ph, int L) {
  if (ph == 0) return PH_EMBED;
  if (ph == 1 + 6 * L) return PH_GEMM;
  const int k = (ph - 1) % 6;
  return k == 1 ? PH_ATTN : (k == 2 ? PH_COMB : PH_GEMM);
}

struct GPh {
  int epi, wmap, xmap, N, K, layer, kind;  // kind: 0 qkv, 3 o, 4 gate/up, 5 down, 6 lm_head
};

__device__ __forceinline__ GPh gemm_of(int ph, const PersistParams& p) {
  GPh g;
  const int qkvd = (p.nh + 2 * p.nkv) * 128, qd = p.nh * 128;
  if (ph == 1 + 6 * p.L) {
    g.epi = EPI_LMHEAD; g.wmap = 4 * p.L; g.xmap = 0; g.N = p.V; g.K = p.H; g.layer = p.L - 1; g.kind = 6;
    return g;
  }
  const int l = (ph - 1) / 6, k = (ph - 1) % 6;
  g.layer = l;
  g.kind = k;
  if (k == 0) { g.epi = EPI_QKV; g.wmap = 4 * l; g.xmap = 0; g.N = qkvd; g.K = p.H; }
  else if (k == 3) { g.epi = EPI_RESID; g.wmap = 4 * l + 1; g.xmap = 1; g.N = p.H; g.K = qd; }
  else if (k == 4) { g.epi = EPI_GATEUP; g.wmap = 4 * l + 2; g.xmap = 3; g.N = 2 * p.F; g.K = p.H; }
  else { g.epi = EPI_RESID; g.wmap = 4 * l + 3; g.xmap = 2; g.N = p.H; g.K = p.F; }
  return g;
}

// ---------------------------------------------------------------- stream-K segments
struct Seg {
  int tile, kb0, nkb, rank, ncontrib;
};

// Owner CTA of global k-block k when `total` k-blocks are split over G CTAs with CTA c
// starting at floor(c * total / G).
__device__ __forceinline__ int owner_of(int64_t k, int64_t total, int G) {
  return (int)(((k + 1) * G + total - 1) / total) - 1;
}

struct SegIter {
  int64_t k, hi, total;
  int nkb, G, c;
  __device__ SegIter(int tiles, int nkb_, int G_, int c_) : nkb(nkb_), G(G_), c(c_) {
    total = (int64_t)tiles * nkb_;
    k = (int64_t)c_ * total / G_;
    hi = (int64_t)(c_ + 1) * total / G_;
  }
  __device__ bool next(Seg& s) {
    if (k >= hi) return false;
    const int tile = (int)(k / nkb);
    const int64_t tb = (int64_t)tile * nkb, te = tb + nkb;
    const int64_t end = hi < te ? hi : te;
    const int first = owner_of(tb, total, G), last = owner_of(te - 1, total, G);
    s.tile = tile;
    s.kb0 = (int)(k - tb);
    s.nkb = (int)(end - k);
    s.rank = c - first;
    s.ncontrib = last - first + 1;
    k = end;
    return true;
  }
};

// Most CTAs that can share one tile: each CTA covers at least floor(T / G) k-blocks.
__host__ __device__ __forceinline__ int max_contrib(int tiles, int nkb, int G) {
  const int64_t total = (int64_t)tiles * nkb;
  const int64_t per = total / G;
  return (int)(per > 0 ? (nkb + per - 1) / per + 1 : G);
}

// ---------------------------------------------------------------- grid-wide phase counters
__device__ __forceinline__ unsigned ld_acquire(const unsigned* ptr) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// Phase timeline (DFLASH_PHASE_TRACE builds): %globaltimer into slot `slot` of (CTA, phase).
//   0 epilogue warps past the phase barrier      1 activation producer past the barrier
//   2 first weight copy of the phase issued        3 last MMA of the phase committed
//   4 first accumulator (or attention Q) ready     5 split-K partials counted (finisher)
//   6 split-K partials landed / last attention item done
//   7 phase arrival                                8 epilogue warps done (before the arrival)
//   9 a contributor's partial counted in
//  10 finisher: partials added / attention: first S ready / combine: partials landed
//  11 finisher: epilogue body done / attention: last P V done
//  12 finisher: outputs fenced, before the release / attention: output stored
__device__ __forceinline__ void trace_stamp(const PersistParams& p, int ph, int slot) {
#if DFLASH_PHASE_TRACE
  if (p.trace) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p.trace[((size_t)blockIdx.x * (2 + 6 * p.L) + ph) * kTraceSlots + slot] = t;
  }
#else
  (void)p; (void)ph; (void)slot;
#endif
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Wait until every CTA arrived on counter `ctr`.  Gives up (and raises the grid abort flag) after
// kGridSpin polls, or early when another CTA gave up.
__device__ bool grid_wait(const unsigned* ctr, unsigned target, volatile int* labort, int* gabort) {
  for (long long i = 0; i < kGridSpin; ++i) {
    if (ld_acquire(ctr) >= target) {
      fence_proxy_async_global();
      return true;
    }
    if ((i & 127) == 127 && (*labort || *reinterpret_cast<volatile int*>(gabort))) return false;
  }
  *labort = 1;
  atomicExch(gabort, 1);
  return false;
}

// Release of everything the CTA wrote (its threads met at a barrier first) at GPU scope, then the
// arrival: a cumulative acq_rel fence and a relaxed reduction (lighter than a full SC fence).
__device__ __forceinline__ void release_add(unsigned* ctr) {
  asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
}

__device__ __forceinline__ void grid_arrive(unsigned* ctr) {
  fence_proxy_async_global();
  release_add(ctr);
}

// Same release, two counters (a projection tile finished: its flag and its phase's count).
__device__ __forceinline__ void release_add2(unsigned* a, unsigned* b) {
  asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.u32 [%0], 1;\n\t"
               "red.relaxed.gpu.global.add.u32 [%1], 1;" ::"l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void release_addn(unsigned* a, unsigned n) {
  asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(n) : "memory");
}

// Wait until *ctr >= target (acquire), bounded like grid_wait.
__device__ bool count_wait(const unsigned* ctr, unsigned target, volatile int* labort, int* gabort) {
  for (long long i = 0; i < kGridSpin; ++i) {
    if (ld_acquire(ctr) >= target) {
      fence_proxy_async_global();
      return true;
    }
    if ((i & 127) == 127 && (*labort || *reinterpret_cast<volatile int*>(gabort))) return false;
  }
  *labort = 1;
  atomicExch(gabort, 1);
  return false;
}

// Fine-grained dependencies between consecutive projections: k-block kb of a projection's
// operand is produced by one tile of the phase before it (128-column tiles give two k-blocks;
// a gate/up tile gives the 64 act columns of one down k-block), and o_proj's by the attention
// unit of the head it belongs to.  QKV of layer 0 follows the embedding with a grid barrier.
__device__ __forceinline__ bool fine_deps(const GPh& g) { return !(g.kind == 0 && g.layer == 0); }
// index of the producer tile (attention unit for o_proj) of operand k-block kb
__device__ __forceinline__ int dep_index(const PersistParams& p, const GPh& g, int kb) {
  if (g.kind == 3) return (kb / 2) / (p.nh / p.nkv);
  return g.kind == 5 ? kb : kb / 2;
}
__device__ __forceinline__ const unsigned* dep_ptr(const PersistParams& p, const GPh& g, int ph, int d) {
  return g.kind == 3 ? p.head_done + g.layer * 64 + d : p.ready + (size_t)(ph - 1) * p.ready_stride + d;
}

__device__ __forceinline__ bool wait_ab(uint64_t* bar, uint32_t parity, volatile int* abort, int* gabort) {
  if (*abort) return false;
  for (long long i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023) == 1023 && (*abort || *reinterpret_cast<volatile int*>(gabort))) {
      *abort = 1;
      return false;
    }
  }
  *abort = 1;
  atomicExch(gabort, 1);
  return false;
}

// ---------------------------------------------------------------- embedding (warps 0-3)
// One warp per (token row, 128-column group): x = E[token], xb = bf16(x * ln_in_0) and the
// group's sum of x^2 into ss_b.  No block-wide barrier.
__device__ void embed_phase(const PersistParams& p, int c, int warp, int lane) {
  const int ngr = p.H / 128;
  const int items = p.M * ngr;
  const __nv_bfloat16* ln = p.layers[0].ln_in;
  for (int i = c * 4 + warp; i < items; i += p.G * 4) {
    const int row = i / ngr, gi = i % ngr;
    const int r = row % kGamma, s = row / kGamma;
    const int tok = r == 0 ? __ldg(p.bonus + s) : p.mask;
    const bool ok = tok >= 0 && tok < p.V;
    if (!ok && gi == 0 && lane == 0) atomicOr(p.status, DFLASH_DEV_BAD_TOKEN);
    if (r == 0 && gi == 0 && lane == 0 && width_out_of_range(p.widths, s)) atomicOr(p.status, DFLASH_DEV_BAD_WIDTH);
    const int col = gi * 128 + lane * 4;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
      const uint2 e = __ldg(reinterpret_cast<const uint2*>(p.embed + (int64_t)tok * p.H + col));
      const __nv_bfloat162 e0 = *reinterpret_cast<const __nv_bfloat162*>(&e.x);
      const __nv_bfloat162 e1 = *reinterpret_cast<const __nv_bfloat162*>(&e.y);
      v[0] = __low2float(e0); v[1] = __high2float(e0); v[2] = __low2float(e1); v[3] = __high2float(e1);
    }
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(ln + col));
    const __nv_bfloat162 w0 = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
    const __nv_bfloat162 w1 = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
    *reinterpret_cast<float4*>(p.x + (int64_t)row * p.H + col) = make_float4(v[0], v[1], v[2], v[3]);
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(v[0] * __low2float(w0), v[1] * __high2float(w0));
    const __nv_bfloat162 b1 = __floats2bfloat162_rn(v[2] * __low2float(w1), v[3] * __high2float(w1));
    *reinterpret_cast<uint2*>(p.xb + (int64_t)row * p.H + col) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
    const float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
    if (lane == 0) p.ss_b[(int64_t)gi * p.M + row] = ss;
  }
}

// Per-token input scale 1/RMS(x_m) from the per-128-column partial sums.
__device__ __forceinline__ float row_rscale(const PersistParams& p, const float* ss_in, int m) {
  const int parts = p.H / 128;
  float ssum = 0.f;
  for (int q0 = 0; q0 < parts; q0 += 8) {
    float part[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) part[u] = q0 + u < parts ? __ldcg(ss_in + (int64_t)(q0 + u) * p.M + m) : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) ssum += part[u];
  }
  return 1.f / sqrtf(ssum / (float)p.H + p.eps);
}

// Final hidden state of token `row`: RMSNorm(x) * norm in bf16 (rs = 1/RMS(x_row)).
__device__ void final_hidden_row(const PersistParams& p, int row, float rs, int t) {
  const int ngr = p.H / 128;
  float xv[kMaxHGroups];
#pragma unroll
  for (int k = 0; k < kMaxHGroups; ++k) xv[k] = k < ngr ? __ldcg(p.x + (int64_t)row * p.H + k * 128 + t) : 0.f;
#pragma unroll
  for (int k = 0; k < kMaxHGroups; ++k)
    if (k < ngr)
      p.final_hidden[(int64_t)row * p.H + k * 128 + t] =
          __float2bfloat16_rn(xv[k] * rs * __bfloat162float(p.norm[k * 128 + t]));
}

// ---------------------------------------------------------------- attention (warps 0-3)
struct AttnUse {
  int kv[2], s, o;
};

// Geometry of one attention work item (unit = sequence x kv head, split of its key chunks).
struct AItem {
  int s, g, ctx, k0, nch, c_begin, c_end, nsplit, splits, window;
  bool bad;  // context length out of range (reported once per unit)
  bool run;  // false: nothing to do (bad context, or a split beyond the sequence's chunks)
};

__device__ __forceinline__ int chunk_range_p(int window, int ctx, int* first_key) {
  const int nkeys = ctx + kGamma;
  int k0 = 0;
  if (window > 0) {
    k0 = ctx - window + 1;
    if (k0 < 0) k0 = 0;
    k0 &= ~(kPage - 1);
  }
  *first_key = k0;
  return (nkeys - k0 + kAKC - 1) / kAKC;
}

__device__ AItem attn_geom(const PersistParams& p, int layer, int unit, int split, int ctx0) {
  AItem a;
  a.window = p.layers[layer].window;
  a.s = unit / p.nkv;
  a.g = unit % p.nkv;
  a.ctx = ctx0;
  const int wi = a.window > 0;
  const int cps = p.attn_cps[wi];
  a.splits = p.attn_splits[wi];
  a.run = false;
  a.bad = false;
  a.nch = a.k0 = a.nsplit = a.c_begin = a.c_end = 0;
  if (a.ctx < 0 || a.ctx > p.max_ctx || a.ctx + kGamma > p.mpps * kPage) {
    a.bad = true;
    return a;
  }
  a.nch = chunk_range_p(a.window, a.ctx, &a.k0);
  a.nsplit = (a.nch + cps - 1) / cps;
  if (a.nsplit > a.splits) {  // cannot happen for ctx <= max_ctx; never drop keys silently
    a.bad = true;
    return a;
  }
  if (split >= a.nsplit) return a;
  a.c_begin = split * cps;
  a.c_end = min(a.nch, a.c_begin + cps);
  a.run = true;
  return a;
}

// K and V pages of key chunk c into K/V stage st (one thread).
__device__ void attn_load_chunk(const PersistParams& p, int layer, const AItem& a, int c, int st, uint8_t* sKV,
                                Bars& B) {
  uint8_t* dK = sKV + st * kAKVStage;
  uint8_t* dV = dK + kAPages * kATile;
  const int32_t* pt = p.page_tables + (int64_t)a.s * p.mpps;
  const int npages_seq = (a.ctx + kGamma + kPage - 1) / kPage;
  mbar_arrive_expect_tx(&B.kv_full[st], 2 * kAPages * kATile);
  const int pg0 = (a.k0 + c * kAKC) / kPage;
  int pages[kAPages];
#pragma unroll
  for (int i = 0; i < kAPages; ++i) pages[i] = __ldg(pt + (pg0 + i < npages_seq ? pg0 + i : 0));
#pragma unroll
  for (int i = 0; i < kAPages; ++i) {
    int page = pages[i];
    if (page < 0 || page >= p.g.num_pages) {
      atomicOr(p.status, DFLASH_DEV_BAD_PAGE);
      page = 0;
    }
    bulk_load(dK + i * kATile, p.pool + tile_base(p.g, layer, page, 0, a.g), kATile, &B.kv_full[st]);
    bulk_load(dV + i * kATile, p.pool + tile_base(p.g, layer, page, 1, a.g), kATile, &B.kv_full[st]);
  }
}

// Chunk c holds context keys only (pages written before this forward), so it may be copied
// before this forward's QKV phase has finished.
__device__ __forceinline__ bool chunk_is_context(const AItem& a, int c) {
  return a.k0 + (c + 1) * kAKC <= (a.ctx / kPage) * kPage;
}

// Before the QKV phase completes: copy the first two chunks of this CTA's first item if they
// hold context keys only.  Returns the stages loaded (bit st).  One thread.
__device__ int attn_prefetch(const PersistParams& p, int layer, int unit, int split, uint8_t* sKV, Bars& B) {
  const AItem a = attn_geom(p, layer, unit, split, B.ctx0);
  if (!a.run) return 0;
  fence_proxy_async_smem();
  int pre = 0;
  for (int i = 0; i < 2; ++i) {
    const int c = a.c_begin + i;
    if (c < a.c_end && chunk_is_context(a, c)) {
      attn_load_chunk(p, layer, a, c, i, sKV, B);
      pre |= 1 << i;
    }
  }
  return pre;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One attention work item on warps 0-3: the 8 query heads x 16 rows of one kv head against
// key chunks [c_begin, c_end), taken two chunks (128 keys) at a time: S = Q K^T for both
// chunks on the tensor cores, one max pass and one exp pass over the 128 scores, P (bf16) back
// into the S columns of TMEM, O += P V with P read from TMEM.  O stays in TMEM (rescaled
// there when a row's running max grows) and is read once at the end.  Warp 0 waits for the
// K/V copies and issues the MMAs (lane 0) with the warp converged.  The loops are kept
// rolled: straight-line code this large would run from a cold instruction cache every time.
__device__ void attn_item(const PersistParams& p, int layer, int unit, int split, int pre, uint8_t* sA, Bars& B,
                          AttnUse& use, int t) {
  const int warp = t >> 5, lane = t & 31;
  const AItem a = attn_geom(p, layer, unit, split, B.ctx0);
  if (!a.run) {
    if (a.bad && split == 0 && t == 0) atomicOr(p.status, DFLASH_DEV_BAD_CTX);
    return;
  }
  const int group = p.nh / p.nkv;
  const int nkeys = a.ctx + block_width(p.widths, a.s);  // keys past the active block width are masked
  uint8_t* sQ = sA + kAP;
  uint8_t* sKV = sQ + kAQ;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = B.tmem + kTS + lane_off, tO = B.tmem + kTO + lane_off;
  volatile int* ab = &B.abort;

  if (warp == 0) {
    if (lane == 0) {
      fence_proxy_async_smem();
      if (!(pre & 1)) attn_load_chunk(p, layer, a, a.c_begin, 0, sKV, B);
      if (a.c_begin + 1 < a.c_end && !(pre & 2)) attn_load_chunk(p, layer, a, a.c_begin + 1, 1, sKV, B);
    }
    __syncwarp();
  }
  // the unit's queries: 16-byte copies, 32 consecutive ones reading 512 contiguous bytes
#pragma unroll
  for (int k = 0; k < 16; ++k) stage_q_piece(sQ, p.q, a.s, a.g, p.nh, k * kEThreads + t);
  cp_async_wait_all();
  fence_proxy_async_smem();
  epi_sync();
  const int tph = 2 + 6 * layer;  // this attention phase (trace stamps)
  const bool stamp = t == 0 && unit * a.splits + split == (int)blockIdx.x;  // the CTA's first item
  if (stamp) trace_stamp(p, tph, 4);

  const int pos_q = a.ctx + (t & 15);
  const float scale_log2 = 1.4426950408889634f / sqrtf(128.f);
  float m_run = -FLT_MAX, l_run = 0.f;
  constexpr uint32_t idesc_s = idesc_bf16(128, kAKC);
  constexpr uint32_t idesc_o = idesc_bf16(128, 128);

#pragma unroll 1
  for (int sc = a.c_begin; sc < a.c_end; sc += 2) {
    const int nchk = min(2, a.c_end - sc);
    if (warp == 0) {
#pragma unroll 1
      for (int i = 0; i < nchk; ++i) {
        wait_ab(&B.kv_full[i], use.kv[i] & 1, ab, p.gabort);
        tc_fence_after();
        if (lane == 0 && !*ab) {
          uint8_t* sK = sKV + i * kAKVStage;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_bf16(B.tmem + kTS + i * kAKC, desc_noswz(sQ + k * 256, 128, 2048), desc_noswz(sK + k * 256, 128, 2048),
                     idesc_s, k > 0 ? 1u : 0u);
        }
        __syncwarp();
      }
      if (lane == 0) mma_commit(&B.s_done);
      __syncwarp();
    }
    use.kv[0]++;
    if (nchk > 1) use.kv[1]++;
    wait_ab(&B.s_done, use.s & 1, ab, p.gabort);
    use.s++;
    tc_fence_after();
    if (stamp && sc == a.c_begin) trace_stamp(p, tph, 10);

    // every key of the super-chunk visible to every row: no masking
    const int kb = a.k0 + sc * kAKC, nk = nchk * kAKC;
    const bool full = kb + nk <= nkeys && (a.window <= 0 || a.ctx + kGamma - 1 - kb < a.window);
    float mc = -FLT_MAX;
#pragma unroll 1
    for (int q4 = 0; q4 < 2 * nchk; ++q4) {
      float v[32];
      tmem_ld32(tS + q4 * 32, v);
      if (full) {
#pragma unroll
        for (int j = 0; j < 32; ++j) mc = fmaxf(mc, v[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int key = kb + q4 * 32 + j;
          if (key < nkeys && (a.window <= 0 || pos_q - key < a.window)) mc = fmaxf(mc, v[j]);
        }
      }
    }
    // max(s) * c == max(s * c) for c > 0 (rounding is monotonic)
    const float m_new = fmaxf(m_run, mc == -FLT_MAX ? -FLT_MAX : mc * scale_log2);
    const float alpha = m_run == -FLT_MAX ? 1.f : ex2(m_run - m_new);
    if (sc > a.c_begin && __any_sync(0xffffffffu, alpha != 1.f)) {
      // O (complete: the previous P V was waited for) times alpha, in TMEM
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        float v[32];
        tmem_ld32(tO + q4 * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= alpha;
        tmem_st32(tO + q4 * 32, v);
      }
    }
    // P = exp2(s * c - m) as bf16 pairs; keys 64 h .. 64 h + 63 go to columns 32 h .. 32 h + 31,
    // over scores already read
    float lsum = 0.f;
#pragma unroll 1
    for (int h = 0; h < nchk; ++h) {
      uint32_t pk[32];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float v[32];
        tmem_ld32(tS + (2 * h + q) * 32, v);
        if (full) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(ex2(fmaf(v[2 * e], scale_log2, -m_new)),
                                                            ex2(fmaf(v[2 * e + 1], scale_log2, -m_new)));
            lsum += __low2float(h2) + __high2float(h2);
            pk[q * 16 + e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float pr[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int key = kb + (2 * h + q) * 32 + 2 * e + u;
              const bool vis = key < nkeys && (a.window <= 0 || pos_q - key < a.window);
              pr[u] = vis ? ex2(fmaf(v[2 * e + u], scale_log2, -m_new)) : 0.f;
            }
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(pr[0], pr[1]);
            lsum += __low2float(h2) + __high2float(h2);
            pk[q * 16 + e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
        }
      }
      tmem_st32u(tS + h * 32, pk);
    }
    l_run = l_run * alpha + lsum;
    m_run = m_new;
    tc_fence_before();
    epi_sync();
    if (warp == 0) {
      if (lane == 0) {
        tc_fence_after();
        if (!*ab) {
#pragma unroll 1
          for (int kk = 0; kk < 4 * nchk; ++kk)
            mma_bf16_tmem_a(B.tmem + kTO, B.tmem + kTS + kk * 8,
                            desc_noswz(sKV + (kk >> 2) * kAKVStage + kAPages * kATile + (kk & 3) * kATile, 128, 256),
                            idesc_o, (sc > a.c_begin || kk > 0) ? 1u : 0u);
        }
        mma_commit(&B.o_done);
      }
      __syncwarp();
    }
    wait_ab(&B.o_done, use.o & 1, ab, p.gabort);
    use.o++;
    tc_fence_after();
    if (sc + 2 < a.c_end && warp == 0) {
      // the MMAs that read both stages are complete: refill them
      if (lane == 0 && !*ab) {
        attn_load_chunk(p, layer, a, sc + 2, 0, sKV, B);
        if (sc + 3 < a.c_end) attn_load_chunk(p, layer, a, sc + 3, 1, sKV, B);
      }
      __syncwarp();
    }
  }
  if (stamp) trace_stamp(p, tph, 11);
  // O out of TMEM: normalised bf16 rows, or the split's fp32 partial (O, m, l)
  const int hh = t >> 4;
  __nv_bfloat16* dst = p.attn + ((int64_t)(a.s * kGamma + (t & 15)) * p.nh + a.g * group + hh) * 128;
  const int64_t slot = (int64_t)unit * a.splits + split;
  const float inv = a.nsplit == 1 ? (l_run > 0.f ? 1.f / l_run : 0.f) : 1.f;
#pragma unroll 1
  for (int q4 = 0; q4 < 4; ++q4) {
    float v[32];
    tmem_ld32(tO + q4 * 32, v);
    if (a.nsplit == 1) {
#pragma unroll
      for (int d8 = 0; d8 < 4; ++d8) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[d8 * 8 + 2 * e] * inv, v[d8 * 8 + 2 * e + 1] * inv);
          pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        reinterpret_cast<uint4*>(dst + q4 * 32)[d8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        __stcg(o_part_at(p.o_part, slot, t, q4 * 8 + (i >> 2)), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
    }
  }
  if (a.nsplit > 1) __stcg(reinterpret_cast<float2*>(p.ml_part + (slot * 128 + t) * 2), make_float2(m_run, l_run));
  if (stamp) trace_stamp(p, tph, 12);
  tc_fence_before();  // TMEM reads done before the next item's MMAs overwrite S and O
}

// Merge the split partials of rows 4 rb .. 4 rb + 3 of one unit (a warp per row, a lane per
// 4 dims).  Every split's 4 rows of O (2 KB) and (m, l) (32 B) arrive in shared memory in one
// round trip, as 16-byte asynchronous copies spread over the 128 threads (one thread issuing a
// bulk copy per split serialises on the issue); the merge then takes the rows' global max first
// and sums the splits in order.
constexpr int kCmbBytes = kAQ + 2 * kAKVStage;  // landing buffer: the attention Q + K/V area

__device__ void combine_item(const PersistParams& p, int layer, int unit, int rb, int t, int ctx0, uint8_t* sBuf,
                             Bars& B, int& red_use) {
  const AItem a = attn_geom(p, layer, unit, 0, ctx0);
  if (!a.run || a.nsplit <= 1) return;
  // thread t: row r0 + t % 4, dims 4 (t / 4) .. (the order of the 4 rows' 2 KB in o_part)
  const int r0 = rb * 4, rr = t & 3, row = r0 + rr, db = t >> 2, d0 = db * 4;
  const int64_t base = (int64_t)unit * a.splits;
  const int ns = a.nsplit;
  float M = -FLT_MAX, L = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (ns * (2048 + 32) <= kCmbBytes) {
    for (int i = t; i < ns * 128; i += kEThreads) {
      // the 4 rows of split q: 2 KB contiguous, copied as they lie
      const int q = i >> 7, off = i & 127;
      cp_async16(sBuf + q * 2048 + off * 16, o_part_at(p.o_part, base + q, r0, 0) + off);
    }
    for (int i = t; i < ns * 2; i += kEThreads) {
      const int q = i >> 1, half = i & 1;
      cp_async16(sBuf + ns * 2048 + q * 32 + half * 16, p.ml_part + ((base + q) * 128 + r0) * 2 + half * 4);
    }
    cp_async_wait_all();
    epi_sync();
    const float4* so = reinterpret_cast<const float4*>(sBuf);
    const float2* sml = reinterpret_cast<const float2*>(sBuf + ns * 2048);
    for (int q = 0; q < ns; ++q) M = fmaxf(M, sml[q * 4 + rr].x);
#pragma unroll 4
    for (int q = 0; q < ns; ++q) {
      const float2 ml = sml[q * 4 + rr];
      const float w = ml.x == -FLT_MAX ? 0.f : exp2f(ml.x - M);
      const float4 ov = so[q * 128 + t];
      a0 += ov.x * w; a1 += ov.y * w; a2 += ov.z * w; a3 += ov.w * w;
      L += ml.y * w;
    }
  } else {
    for (int q0 = 0; q0 < ns; q0 += 8) {
      float2 ml[8];
      float4 ov[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int q = q0 + u < ns ? q0 + u : q0;
        ml[u] = __ldcg(reinterpret_cast<const float2*>(p.ml_part + ((base + q) * 128 + row) * 2));
        ov[u] = __ldcg(o_part_at(p.o_part, base + q, row, db));
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (q0 + u >= ns) break;
        if (ml[u].x > M) {
          const float sc = M == -FLT_MAX ? 0.f : exp2f(M - ml[u].x);
          a0 *= sc; a1 *= sc; a2 *= sc; a3 *= sc; L *= sc;
          M = ml[u].x;
        }
        const float w = ml[u].x == -FLT_MAX ? 0.f : exp2f(ml[u].x - M);
        a0 += ov[u].x * w; a1 += ov[u].y * w; a2 += ov[u].z * w; a3 += ov[u].w * w;
        L += ml[u].y * w;
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(a0 * inv, a1 * inv);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(a2 * inv, a3 * inv);
  const int hh = row >> 4, r = row & 15;
  __nv_bfloat16* dst = p.attn + ((int64_t)(a.s * kGamma + r) * p.nh + a.g * (p.nh / p.nkv) + hh) * 128 + d0;
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kBlockThreads, 1) persist_kernel(const __grid_constant__ PersistParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* sA = smem + kRing;
  auto stage = [&](int s) { return ring + s * kStage; };
  uint8_t* sRed = sA + kAP;  // split-K partial landing buffer (the attention Q + K/V area)
  Bars& B = *reinterpret_cast<Bars*>(smem + kBarOff);
  float* rsc = reinterpret_cast<float*>(smem + kBarOff + 512);
  EpiSmem& es = *reinterpret_cast<EpiSmem*>(sA);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = p.G, c = blockIdx.x;
  const int P = 2 + 6 * p.L;

  if (t == 0) {
    for (int i = 0; i < kS; ++i) {
      mbar_init(&B.full[i], 1);
      mbar_init(&B.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.acc_full[i], 1);
      mbar_init(&B.acc_empty[i], 1);
      mbar_init(&B.kv_full[i], 1);
    }
    mbar_init(&B.s_done, 1);
    mbar_init(&B.o_done, 1);
    mbar_init(&B.red_full, 1);
    B.abort = 0;
    B.flag = 0;
    B.ctx0 = __ldg(p.ctx_lens);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&B.tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  volatile int* ab = &B.abort;

  if (warp == 4) {
    if (lane == 0) {
      // ---------------- weight producer: runs ahead over every projection of the forward
      const uint64_t pol = policy_evict_first();
      int j = 0;
      for (int ph = 0; ph < P && !*ab; ++ph) {
        if (phase_kind(ph, p.L) != PH_GEMM) continue;
        const GPh gp = gemm_of(ph, p);
        const CUtensorMap* wm = p.maps + gp.wmap;
        SegIter it((gp.N + 127) / 128, gp.K / 64, G, c);
        Seg sg;
        bool first_w = true;
        while (it.next(sg) && !*ab) {
          for (int kk = 0; kk < sg.nkb; ++kk, ++j) {
            const int s = j % kS, u = j / kS;
            if (u > 0 && !wait_ab(&B.empty[s], (u - 1) & 1, ab, p.gabort)) break;
            // arm the stage for the weight and the activation tile (the activation producer
            // adds its copy to the same phase, before or after this arrive)
            mbar_arrive_expect_tx(&B.full[s], kStage);
            tma_load_2d(stage(s), wm, &B.full[s], (sg.kb0 + kk) * 64, sg.tile * 128, pol);
            if (first_w) { trace_stamp(p, ph, 2); first_w = false; }
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    // ---------------- activation producer: the whole warp.  For a segment of k-blocks its
    // lanes poll the ready flags of the producer tiles together (one round trip per poll, lane i
    // the i-th flag not yet seen set); lane 0 copies each k-block's X tile as soon as its own
    // producer tile is done, so the MMAs start on the earliest tiles.
    const uint64_t pol = policy_evict_last();
    int j = 0;
    bool stop = false;
    for (int ph = 0; ph < P && !stop; ++ph) {
      if (phase_kind(ph, p.L) != PH_GEMM) continue;
      const GPh gp = gemm_of(ph, p);
      const CUtensorMap* xm = p.maps + 4 * p.L + 1 + gp.xmap;
      const unsigned target = gp.kind == 3 ? 32u : 1u;
      SegIter it((gp.N + 127) / 128, gp.K / 64, G, c);
      Seg sg;
      bool waited = false;
      const bool fine = fine_deps(gp);
      while (!stop && it.next(sg)) {
        if (!waited && !fine) {
          if (lane == 0) grid_wait(&p.bar[ph - 1], (unsigned)G, ab, p.gabort);
          __syncwarp();
        }
        const int d1 = fine ? dep_index(p, gp, sg.kb0 + sg.nkb - 1) : 0;
        int ready_lo = fine ? dep_index(p, gp, sg.kb0) : 0;  // producers below this one are done
        for (int kk = 0; kk < sg.nkb; ++kk, ++j) {
          if (fine) {
            const int d = dep_index(p, gp, sg.kb0 + kk);
            long long spin = 0;
            while (d >= ready_lo) {
              const bool mine = ready_lo + lane <= d1;
              const unsigned v = mine ? ld_acquire(dep_ptr(p, gp, ph, ready_lo + lane)) : 0u;
              const unsigned mask = __ballot_sync(0xffffffffu, mine && v >= target);
              ready_lo += mask == 0xffffffffu ? 32 : __ffs(~mask) - 1;  // the leading run of done tiles
              if (d < ready_lo) {
                fence_proxy_async_global();
                break;
              }
              int give_up = ++spin > kGridSpin;
              if ((spin & 127) == 0 && lane == 0) give_up |= *ab || *reinterpret_cast<volatile int*>(p.gabort);
              if (__shfl_sync(0xffffffffu, give_up, 0)) {
                if (lane == 0) { *ab = 1; atomicExch(p.gabort, 1); }
                stop = true;
                break;
              }
            }
            if (stop) break;
          }
          if (!waited) {
            if (lane == 0) trace_stamp(p, ph, 1);
            waited = true;
          }
          const int s = j % kS, u = j / kS;
          int ok = 1;
          if (lane == 0) {
            // use u of stage s starts once the MMA released use u - 1; the release of use u
            // needs this copy, so the stage cannot run a phase ahead of it
            if (u > 0 && !wait_ab(&B.empty[s], (u - 1) & 1, ab, p.gabort)) ok = 0;
            else tma_load_2d(stage(s) + kAB, xm, &B.full[s], (sg.kb0 + kk) * 64, 0, pol);
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) {
            stop = true;
            break;
          }
        }
        if (__shfl_sync(0xffffffffu, lane == 0 ? (int)*ab : 0, 0)) stop = true;
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16(128, TN);
      int j = 0, segc = 0;
      for (int ph = 0; ph < P && !*ab; ++ph) {
        if (phase_kind(ph, p.L) != PH_GEMM) continue;
        const GPh gp = gemm_of(ph, p);
        SegIter it((gp.N + 127) / 128, gp.K / 64, G, c);
        Seg sg;
        while (it.next(sg) && !*ab) {
          const int buf = segc & 1;
          if (segc >= 2) wait_ab(&B.acc_empty[buf], ((segc >> 1) - 1) & 1, ab, p.gabort);
          tc_fence_after();
          const uint32_t d = B.tmem + buf * kAccCols;
          for (int kk = 0; kk < sg.nkb; ++kk, ++j) {
            const int s = j % kS, u = j / kS;
            wait_ab(&B.full[s], u & 1, ab, p.gabort);
            tc_fence_after();
            if (!*ab) {
              const uint64_t ad = desc_sw128(stage(s));
              const uint64_t bd = desc_sw128(stage(s) + kAB);
#pragma unroll
              for (int k = 0; k < 4; ++k) mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kk > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(&B.empty[s]);
          }
          mma_commit(&B.acc_full[buf]);
          ++segc;
        }
        trace_stamp(p, ph, 3);
      }
    }
    __syncwarp();
  } else {
    // ---------------- warps 0-3: epilogues and the non-GEMM phases
    AttnUse use = {{0, 0}, 0, 0};
    int segc = 0, red_use = 0;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    for (int ph = 0; ph < P; ++ph) {
      const int kind = phase_kind(ph, p.L);
      if (kind == PH_EMBED) {
        embed_phase(p, c, warp, lane);
      } else if (kind == PH_ATTN || kind == PH_COMB) {
        const int l = (ph - 1) / 6;
        const int units = (p.M / kGamma) * p.nkv;
        const int splits = p.attn_splits[p.layers[l].window > 0];
        const int items = kind == PH_ATTN ? units * splits : units * 32;
        if (c < items) {
          int pre = 0;
          if (kind == PH_ATTN && t == 0) pre = attn_prefetch(p, l, c / splits, c % splits, sA + kAP + kAQ, B);
          if (t == 0) grid_wait(&p.bar[ph - 1], (unsigned)G, ab, p.gabort);
          if (t == 0) trace_stamp(p, ph, 0);
          epi_sync();
          for (int i = c; i < items && !*ab; i += G) {
            if (kind == PH_ATTN) {
              // `pre` is only read by thread 0, which computed it
              attn_item(p, l, i / splits, i % splits, i == c ? pre : 0, sA, B, use, t);
              fence_proxy_async_global();  // o_proj reads the attention output through TMA
              epi_sync();
              // a unit with one split (or none: a bad context) is complete with its item
              if (t == 0 && i % splits == 0 && attn_geom(p, l, i / splits, 0, B.ctx0).nsplit <= 1)
                release_addn(p.head_done + l * 64 + i / splits, 32u);
            } else {
              combine_item(p, l, i / 32, i % 32, t, B.ctx0, sRed, B, red_use);
              fence_proxy_async_global();
              epi_sync();  // the landing buffer is reused by the next item
              if (t == 0 && attn_geom(p, l, i / 32, 0, B.ctx0).nsplit > 1) release_addn(p.head_done + l * 64 + i / 32, 1u);
            }
          }
          if (t == 0) trace_stamp(p, ph, 6);
        }
      } else {
        // GEMM epilogues of this CTA's segments
        const GPh gp = gemm_of(ph, p);
        const int tiles = (gp.N + 127) / 128, nkb = gp.K / 64;
        const int maxc = max_contrib(tiles, nkb, G);
        SegIter it(tiles, nkb, G, c);
        Seg sg;
        bool first = true;
        GemmParams e;
        e.N = gp.N; e.K = gp.K; e.M = p.M; e.Mp = p.M; e.eps = p.eps; e.status = p.status;
        e.ss_n = p.H; e.ss_parts = p.H / 128;
        e.q = p.q; e.inv_pi = p.inv_pi; e.mscale = p.mscale; e.nh = p.nh; e.nkv = p.nkv;
        e.ctx_lens = p.ctx_lens; e.page_tables = p.page_tables; e.mpps = p.mpps; e.g = p.g;
        e.rope_pos0 = p.rope_pos0; e.widths = p.widths;
        e.layer = gp.layer; e.pool = p.pool; e.x = p.x; e.xb = p.xb; e.H = p.H; e.act = p.act; e.F = p.F;
        e.logits = p.logits; e.amax_best = p.amax_best;
        const PersistLayer& Ly = p.layers[gp.layer];
        if (gp.epi == EPI_QKV) {
          e.ss_in = p.ss_b; e.q_norm = Ly.q_norm; e.k_norm = Ly.k_norm;
        } else if (gp.epi == EPI_GATEUP) {
          e.ss_in = p.ss_a;
        } else if (gp.epi == EPI_LMHEAD) {
          e.ss_in = p.ss_b;  // the final RMSNorm's 1/RMS, applied to the logits
        } else {
          const bool is_o = gp.kind == 3;
          e.ss_out = is_o ? p.ss_a : p.ss_b;
          if (is_o) e.xb = p.xb2;
          // the last down projection prepares the lm_head operand bf16(x * norm)
          e.ln_next = is_o ? Ly.ln_post : (gp.layer + 1 < p.L ? p.layers[gp.layer + 1].ln_in : p.norm);
        }
        // the phase the epilogue's inputs come from, and how long to wait for it: the previous
        // projection's every tile where the epilogue needs whole rows (1/RMS of its operand; the
        // residual of down comes from o_proj), every attention unit of the layer for o_proj
        const int nt_h = p.H / 128;
        auto epi_wait = [&]() {  // one thread
          if (!fine_deps(gp)) {
            grid_wait(&p.bar[ph - 1], (unsigned)G, ab, p.gabort);
          } else if (gp.kind == 3) {
            for (int u = 0; u < p.nkv * (p.M / kGamma); ++u)
              count_wait(p.head_done + gp.layer * 64 + u, 32u, ab, p.gabort);
          } else {
            count_wait(p.done + (gp.kind == 5 ? ph - 2 : ph - 1), (unsigned)nt_h, ab, p.gabort);
          }
        };
        if (gp.epi == EPI_LMHEAD && p.final_hidden && c < p.M) {
          // side job (nothing waits for it): the final hidden state of token c
          if (t == 0) epi_wait();
          epi_sync();
          if (t == 0) rsc[0] = row_rscale(p, p.ss_b, c);
          epi_sync();
          final_hidden_row(p, c, rsc[0], t);
          epi_sync();
        }
        while (it.next(sg)) {
          // rank 0 holds the tile's first k-blocks and finishes the tile
          const bool finisher = sg.rank == 0;
          // only a finisher's epilogue reads what the previous phase wrote (whole rows for 1/RMS,
          // the residual): a contributor stores its partial as soon as its MMAs are done
          const bool need_wait = first && finisher;
          const int n = sg.tile * 128 + t;
          EpiPre pre;
          // inputs of the epilogue, fetched while the MMAs run (down's residual is o_proj's
          // output: fetched after the wait for o_proj)
          if (finisher && !(need_wait && gp.kind == 5)) {
            if (gp.epi == EPI_QKV) epilogue_pre<EPI_QKV>(e, pre, t, n, 0, 0, sg.tile, B.ctx0);
            else if (gp.epi == EPI_RESID) epilogue_pre<EPI_RESID>(e, pre, t, n, 0, 0, sg.tile);
          }
          const int buf = segc & 1;
          wait_ab(&B.acc_full[buf], (segc >> 1) & 1, ab, p.gabort);
          if (t == 0) trace_stamp(p, ph, 4);
          tc_fence_after();
          const uint32_t acc = B.tmem + buf * kAccCols + lane_off;
          float v[16];
          tmem_ld16(acc, v);
          tc_fence_before();
          epi_sync();
          if (t == 0) mbar_arrive(&B.acc_empty[buf]);  // accumulator copied: MMA may reuse it
          ++segc;
          // alternate phases use alternate halves of the partials and tile counters: the next
          // phase's contributors may write while this phase's slowest finisher still reads
          float* tile_ws = p.ws + (size_t)(ph & 1) * p.ws_half + (int64_t)sg.tile * maxc * (kEThreads * TN);
          unsigned* cnt = p.counters + (ph & 1) * p.max_tiles;
          if (!finisher) {
            // fp32 partial of this CTA's k-range into slot `rank` (float4 q of thread t at
            // q * 128 + t: the finisher's shared-memory reads are conflict-free), then count it in
            float4* mine = reinterpret_cast<float4*>(tile_ws + (int64_t)sg.rank * kEThreads * TN) + t;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              __stcg(mine + q * kEThreads, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
            epi_sync();
            if (t == 0) release_add(&cnt[sg.tile]);
            if (t == 0) trace_stamp(p, ph, 9);
            continue;
          }
          // finisher: the other ncontrib - 1 partials (warp 0 waits for their count and copies them in
          // with one bulk copy) and the previous phase (warp 1) are waited for at the same time
          const int nother = sg.ncontrib - 1;
          const bool bulk = nother > 0 && nother <= kRedMax;
          if (nother > 0 && warp == 0) {
            // the whole warp polls (one coalesced load)
            for (long long sp = 0; ld_acquire(&cnt[sg.tile]) < (unsigned)nother; ++sp) {
              if (*ab || sp > kGridSpin) {
                if (lane == 0) { *ab = 1; atomicExch(p.gabort, 1); }
                break;
              }
            }
            __syncwarp();
            if (lane == 0) {
              trace_stamp(p, ph, 5);
              cnt[sg.tile] = 0;  // re-armed for the phase after next (it depends on this one)
              if (bulk && !*ab) {
                // the contributors' generic stores, acquired above, then read through the async proxy
                fence_proxy_async_global();
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&B.red_full, nother * kPartBytes);
                bulk_load(sRed, tile_ws + kEThreads * TN, nother * kPartBytes, &B.red_full);
              }
            }
            __syncwarp();
          }
          if (need_wait && t == 32) epi_wait();
          epi_sync();
          if (need_wait) {
            if (t == 0) trace_stamp(p, ph, 0);
            if (e.ss_in && t < TN) rsc[t] = t < p.M ? row_rscale(p, e.ss_in, t) : 1.f;
            if (gp.kind == 5) epilogue_pre<EPI_RESID>(e, pre, t, n, 0, 0, sg.tile);
            epi_sync();
            first = false;
          }
          if (bulk) {
            wait_ab(&B.red_full, red_use & 1, ab, p.gabort);
            if (t == 0) trace_stamp(p, ph, 6);
            ++red_use;
            for (int rk = 0; rk < nother; ++rk) {
              const float4* src = reinterpret_cast<const float4*>(sRed + (size_t)rk * kPartBytes) + t;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float4 f = src[q * kEThreads];
                v[4 * q] += f.x; v[4 * q + 1] += f.y; v[4 * q + 2] += f.z; v[4 * q + 3] += f.w;
              }
            }
          } else if (nother > 0) {
            __threadfence();  // warp 0 saw every partial counted (the barrier above orders the rest)
            for (int rk0 = 1; rk0 < sg.ncontrib; rk0 += 4) {
              float4 q4[4][4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int rk = rk0 + u < sg.ncontrib ? rk0 + u : rk0;
                const float4* src = reinterpret_cast<const float4*>(tile_ws + (int64_t)rk * kEThreads * TN) + t;
#pragma unroll
                for (int q = 0; q < 4; ++q) q4[u][q] = __ldcg(src + q * kEThreads);
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                if (rk0 + u >= sg.ncontrib) break;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  v[4 * q] += q4[u][q].x; v[4 * q + 1] += q4[u][q].y;
                  v[4 * q + 2] += q4[u][q].z; v[4 * q + 3] += q4[u][q].w;
                }
              }
            }
          }
          if (t == 0) trace_stamp(p, ph, 10);
          switch (gp.epi) {
            case EPI_QKV: epilogue_chunk<EPI_QKV>(e, es, rsc, v, t, n, 0, 0, sg.tile, pre); break;
            case EPI_RESID: epilogue_chunk<EPI_RESID>(e, es, rsc, v, t, n, 0, 0, sg.tile, pre); break;
            case EPI_GATEUP: epilogue_chunk<EPI_GATEUP>(e, es, rsc, v, t, n, 0, 0, sg.tile, pre); break;
            default: epilogue_chunk<EPI_LMHEAD>(e, es, rsc, v, t, n, 0, 0, sg.tile, pre); break;
          }
          if (t == 0) trace_stamp(p, ph, 11);
          if (gp.kind >= 3 && gp.kind <= 5) {
            // tile finished: its outputs are the next projection's operand (read through TMA)
            fence_proxy_async_global();
            epi_sync();
            if (t == 0) trace_stamp(p, ph, 12);
            if (t == 0) release_add2(p.ready + (size_t)ph * p.ready_stride + sg.tile, p.done + ph);
          }
          if (gp.epi == EPI_LMHEAD) {
            // the last vocabulary tile to finish turns the running argmaxes into drafts
            __threadfence();
            epi_sync();
            if (t == 0) B.flag = atomicAdd(p.amax_counter, 1u) == (unsigned)(tiles - 1);
            epi_sync();
            if (B.flag) {
              __threadfence();
              if (t < p.M && (t % kGamma) > 0) {
                const unsigned long long k = __ldcg(p.amax_best + t);
                p.drafts[(t / kGamma) * (kGamma - 1) + (t % kGamma) - 1] =
                    (t % kGamma) < block_width(p.widths, t / kGamma) ? argmax_key_index(k) : -1;
              }
            }
          }
        }
      }
      // phase done on this CTA; only the embedding, QKV and attention phases are followed by a
      // grid-wide wait (the others hand over tile by tile)
      if (t == 0) trace_stamp(p, ph, 8);
      epi_sync();
      const bool arrive = kind == PH_EMBED || kind == PH_ATTN || ((ph - 1) % 6 == 0 && ph != 1 + 6 * p.L);
      if (t == 0 && arrive) grid_arrive(&p.bar[ph]);
      if (t == 0) trace_stamp(p, ph, 7);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (t == 0 && *ab) atomicOr(p.status, DFLASH_DEV_TIMEOUT);
  if (*ab) {  // copies issued before a wait gave up: give them time to land
    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
  }
  if (warp == 0) tmem_dealloc(B.tmem, kTmemCols);
}

}  // namespace

int persist_smem_bytes() { return kSmemP; }

int persist_max_hidden() { return kMaxHGroups * 128; }

size_t persist_ws_floats(int H, int F, int nh, int nkv, int V, int num_sms) {
  const int shapes[5][2] = {{(nh + 2 * nkv) * 128, H}, {H, nh * 128}, {2 * F, H}, {H, F}, {V, H}};
  size_t need = 16;
  for (auto& s : shapes) {
    const int tiles = (s[0] + 127) / 128, nkb = s[1] / 64;
    need = std::max(need, (size_t)tiles * max_contrib(tiles, nkb, num_sms) * 128 * TN);
  }
  return need;
}

static int max_tiles_of(int H, int F, int nh, int nkv, int V) {
  return std::max(std::max((nh + 2 * nkv) * 128, H), std::max(2 * F, V)) / 128 + 1;
}

// Tiles of any layer projection (the ones another projection's operand waits on, tile by tile).
static int layer_tiles_of(int H, int F, int nh, int nkv) {
  return std::max(std::max(nh + 2 * nkv, H / 128), (2 * F + 127) / 128);
}

// Control words: the packed argmax of every token (2 words each, first, so 8-byte aligned),
// the phase counters, the abort flag, the lm_head tile counter, two halves of split-K tile
// counters, the per-phase tile-ready flags and counts, the per-layer attention-unit counters.
size_t persist_ctl_words(int L, int H, int F, int nh, int nkv, int V) {
  const size_t P = 2 + 6 * (size_t)L;
  return 2 * (size_t)kPersistMaxM + P + 2 + 2 * (size_t)max_tiles_of(H, F, nh, nkv, V) +
         P * (size_t)layer_tiles_of(H, F, nh, nkv) + P + 64 * (size_t)L;
}

void persist_bind_ctl(PersistParams& p, unsigned* ctl) {
  const int nbar = 2 + 6 * p.L;
  p.amax_best = reinterpret_cast<unsigned long long*>(ctl);
  unsigned* w = ctl + 2 * kPersistMaxM;
  p.bar = w;
  p.gabort = reinterpret_cast<int*>(w + nbar);
  p.amax_counter = w + nbar + 1;
  p.counters = w + nbar + 2;
  p.max_tiles = max_tiles_of(p.H, p.F, p.nh, p.nkv, p.V);
  p.ready = p.counters + 2 * p.max_tiles;
  p.ready_stride = layer_tiles_of(p.H, p.F, p.nh, p.nkv);
  p.done = p.ready + (size_t)nbar * p.ready_stride;
  p.head_done = p.done + nbar;
}

void persist_attn_split(int units, int max_ctx, int window, int G, int* cps, int* splits) {
  int nch = (max_ctx + kGamma + kAKC - 1) / kAKC;
  if (window > 0) nch = std::min(nch, (window + kGamma + kPage + kAKC - 1) / kAKC);
  int c = (units * nch + G - 1) / G;
  if (c < 1) c = 1;
  *cps = c;
  *splits = (nch + c - 1) / c;
}

// The shared-memory limit is a property of the device's context: raise it once per device.
static std::atomic<unsigned long long> g_persist_attr{0};

static cudaError_t persist_attr() { return smem_attr_once(persist_kernel, kSmemP, g_persist_attr); }

cudaError_t persist_occupancy(int* per_sm) {
  cudaError_t e = persist_attr();
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, persist_kernel, kBlockThreads, kSmemP);
}

cudaError_t launch_persist(const PersistParams& p, cudaStream_t st) {
  cudaError_t e0 = persist_attr();
  if (e0 != cudaSuccess) return e0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kBlockThreads);
  cfg.dynamicSmemBytes = kSmemP;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the phase counters need it
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, persist_kernel, p);
}

}  // namespace dflash
