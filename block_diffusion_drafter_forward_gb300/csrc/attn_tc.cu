// Paged GQA block attention on the tensor cores (tcgen05 + TMEM).
//
// What it computes (memra-engine `dflash.rs` forward_round, `sdpa_naive(..., causal =
// false)`; spark_model `from_weights.rs`: paged BF16 prefill kernel with the causal mask
// off): for sequence s, query head h and block row r,
//     o = softmax_j(q . k_j / sqrt(hd) + mask_j) v_j  over keys j = 0 .. ctx_len_s + 15,
// with kv head h / (nh / nkv); on sliding layers key j is masked for the query at position
// p = ctx_len_s + r iff p - j >= window.  Non-causal: every block row sees every block key.
//
// Work unit = (sequence, kv head): its 8 query heads x 16 block rows are the 128 rows of one
// UMMA tile (M = 128), so every K/V byte read from HBM feeds 128 query rows.  Keys go in
// chunks of 64 (4 pages): S = Q K^T is 8 tcgen05.mma (N = 64), O = P V 4 (K = 16 keys each),
// accumulating in TMEM.  Shared memory stays under half an SM so a projection CTA can run
// beside it.  Pages of context rows only are fetched before the wait on the QKV kernel
// (programmatic dependent launch); the page with the block rows after it.  Pages
// are fetched whole (4 KB bulk copies through the page table) into a 2-stage ring; the pool
// stores each page tile in the 8x8-block operand layout, so no reshuffle is needed.
// Softmax runs one query row per thread (no cross-thread reductions), online over chunks.
// Split-KV: a unit's chunks are shared by several CTAs; each writes (O, m, l) partials and
// attn_combine_kernel merges them (all units and rows in parallel, in split order).
#include <float.h>

#include <algorithm>

#include "attn_tc.cuh"
#include "dflash_internal.cuh"
#include "launch_util.cuh"
#include "tc_common.cuh"

namespace dflash {
namespace {

using namespace tc;

constexpr int kKC = 64;               // keys per chunk
constexpr int kPagesPerChunk = kKC / kPage;
constexpr int kTileBytes = kPage * 128 * 2;    // one page of one head: 16 x 128 bf16 = 4 KB
constexpr int kQBytes = 128 * 128 * 2;         // 32 KB
constexpr int kPBytes = 128 * kKC * 2;         // 16 KB
constexpr int kKVStage = 2 * kPagesPerChunk * kTileBytes;  // K + V of one chunk: 32 KB
constexpr int kStages = 2;
constexpr int kSmem = kQBytes + kPBytes + kStages * kKVStage + 256 + 1024;

// Chunks of 128 keys a sequence with `ctx` cached rows visits, starting at *first_key
// (page aligned; on sliding layers the first key any block row can see).
__host__ __device__ inline int chunk_range(int window, int ctx, int* first_key) {
  const int nkeys = ctx + kGamma;
  int k0 = 0;
  if (window > 0) {
    k0 = ctx - window + 1;
    if (k0 < 0) k0 = 0;
    k0 &= ~(kPage - 1);
  }
  *first_key = k0;
  return (nkeys - k0 + kKC - 1) / kKC;
}

__global__ void __launch_bounds__(128, 1) attn_tc_kernel(const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sP = sQ + kQBytes;
  uint8_t* sKV = sP + kPBytes;
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(sKV + kStages * kKVStage);
  uint64_t* s_done = kv_full + kStages;
  uint64_t* o_done = s_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_done + 1);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);

  const int t = threadIdx.x, warp = t >> 5;
  const int unit = blockIdx.x, split = blockIdx.y;
  const int s = unit / p.nkv, g = unit % p.nkv;
  const int group = p.nh / p.nkv;  // 8

  const int ctx = p.ctx_lens[s];  // caller input: not written by the preceding kernel
  if (ctx < 0 || ctx > p.max_ctx || ctx + kGamma > p.mpps * kPage) {
    if (t == 0 && split == 0) atomicOr(p.status, DFLASH_DEV_BAD_CTX);
    return;
  }
  int k0;
  const int nch = chunk_range(p.window, ctx, &k0);
  const int nsplit = (nch + p.chunks_per_split - 1) / p.chunks_per_split;
  if (nsplit > (int)gridDim.y) {  // cannot happen for ctx <= max_ctx; never drop keys silently
    if (t == 0 && split == 0) atomicOr(p.status, DFLASH_DEV_BAD_CTX);
    return;
  }
  if (split >= nsplit) return;
  const int c_begin = split * p.chunks_per_split;
  const int c_end = min(nch, c_begin + p.chunks_per_split);
  const int nkeys = ctx + kGamma;
  const int nvis = ctx + block_width(p.widths, s);  // keys past the active block width are masked
  const int32_t* pt = p.page_tables + (int64_t)s * p.mpps;
  const int npages_seq = (nkeys + kPage - 1) / kPage;

  if (t == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&kv_full[i], 1);
    mbar_init(s_done, 1);
    mbar_init(o_done, 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;

  // issue the page loads of chunk c into stage st (thread 0)
  auto load_chunk = [&](int c, int st) {
    uint8_t* dK = sKV + st * kKVStage;
    uint8_t* dV = dK + kPagesPerChunk * kTileBytes;
    mbar_arrive_expect_tx(&kv_full[st], 2 * kPagesPerChunk * kTileBytes);
    const int pg0 = (k0 + c * kKC) / kPage;
    int pages[kPagesPerChunk];
#pragma unroll
    for (int i = 0; i < kPagesPerChunk; ++i) {  // all page ids in flight together
      const int lp = pg0 + i;
      pages[i] = __ldg(pt + (lp < npages_seq ? lp : 0));
    }
#pragma unroll
    for (int i = 0; i < kPagesPerChunk; ++i) {
      int page = pages[i];
      if (page < 0 || page >= p.g.num_pages) {
        atomicOr(p.status, DFLASH_DEV_BAD_PAGE);
        page = 0;
      }
      const __nv_bfloat16* kt = p.pool + tile_base(p.g, p.layer, page, 0, g);
      const __nv_bfloat16* vt = p.pool + tile_base(p.g, p.layer, page, 1, g);
      bulk_load(dK + i * kTileBytes, kt, kTileBytes, &kv_full[st]);
      bulk_load(dV + i * kTileBytes, vt, kTileBytes, &kv_full[st]);
    }
  };
  // Pages holding only cached context rows are not touched by the preceding QKV kernel (it
  // writes the block rows ctx..ctx+15): fetch those chunks before waiting for it.
  const int safe_keys = ctx & ~(kPage - 1);
  bool early[2] = {false, false};
  if (t == 0) {
    for (int i = 0; i < 2; ++i) {
      const int c = c_begin + i;
      if (c < c_end && k0 + (c + 1) * kKC <= safe_keys) {
        load_chunk(c, i);
        early[i] = true;
      }
    }
  }
  pdl_trigger();
  pdl_wait();
  if (t == 0) {
    for (int i = 0; i < 2; ++i)
      if (c_begin + i < c_end && !early[i]) load_chunk(c_begin + i, i);
  }

  // Q tile: row i = hh * 16 + r  <-  q[s*16 + r, (g*group + hh) * 128 + :], 8x8-block layout
#pragma unroll
  for (int k = 0; k < 16; ++k) stage_q_piece(sQ, p.q, s, g, p.nh, k * 128 + t);
  cp_async_wait_all();
  fence_proxy_async_smem();
  __syncthreads();

  const int r = t & 15;
  const int pos_q = ctx + r;
  const float scale_log2 = 1.4426950408889634f / sqrtf(128.f);
  float m_run = -FLT_MAX, l_run = 0.f;
  float o[128];
#pragma unroll
  for (int i = 0; i < 128; ++i) o[i] = 0.f;
  constexpr uint32_t idesc_s = idesc_bf16(128, kKC);
  constexpr uint32_t idesc = idesc_bf16(128, 128);
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  bool ok = true;

  for (int c = c_begin; c < c_end && ok; ++c) {
    const int it = c - c_begin, st = it & 1;
    uint8_t* sK = sKV + st * kKVStage;
    uint8_t* sV = sK + kPagesPerChunk * kTileBytes;
    if (t == 0) {
      if (!mbar_wait(&kv_full[st], (it >> 1) & 1)) flags[0] = 1;
      tc_fence_after();
      if (!flags[0]) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16(tS, desc_noswz(sQ + k * 256, 128, 2048), desc_noswz(sK + k * 256, 128, 2048), idesc_s,
                   k > 0 ? 1u : 0u);
      }
      mma_commit(s_done);
    }
    if (!mbar_wait(s_done, it & 1)) flags[0] = 1;
    tc_fence_after();
    // ---- softmax of this chunk, one query row per thread (two passes over the S row in
    // TMEM: masked maximum, then probabilities written as the bf16 P operand)
    const int kbase = k0 + c * kKC;
    float mc = -FLT_MAX;
#pragma unroll
    for (int q4 = 0; q4 < kKC / 32; ++q4) {
      float v[32];
      tmem_ld32(tS + lane_off + q4 * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int key = kbase + q4 * 32 + j;
        const bool vis = key < nvis && (p.window <= 0 || pos_q - key < p.window);
        if (vis) mc = fmaxf(mc, v[j] * scale_log2);
      }
    }
    const float m_new = fmaxf(m_run, mc);
    const float alpha = m_new == -FLT_MAX ? 1.f : exp2f(m_run - m_new);
    float lsum = 0.f;
#pragma unroll
    for (int q4 = 0; q4 < kKC / 32; ++q4) {
      float v[32];
      tmem_ld32(tS + lane_off + q4 * 32, v);
#pragma unroll
      for (int j8 = 0; j8 < 4; ++j8) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float pr[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int jj = j8 * 8 + 2 * e + u;
            const int key = kbase + q4 * 32 + jj;
            const bool vis = key < nvis && (p.window <= 0 || pos_q - key < p.window);
            pr[u] = vis ? exp2f(v[jj] * scale_log2 - m_new) : 0.f;
          }
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(pr[0], pr[1]);
          lsum += __low2float(h2) + __high2float(h2);  // the normaliser sums what the MMA uses
          pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(sP + ((t >> 3) * (kKC / 8) + q4 * 4 + j8) * 128 + (t & 7) * 16) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    l_run = l_run * alpha + lsum;
    m_run = m_new;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      if (!flags[0]) {
#pragma unroll
        for (int k = 0; k < kPagesPerChunk; ++k)
          mma_bf16(tO, desc_noswz(sP + k * 256, 128, kKC / 8 * 128), desc_noswz(sV + k * kTileBytes, 128, 256), idesc,
                   k > 0 ? 1u : 0u);
      }
      mma_commit(o_done);
    }
    if (!mbar_wait(o_done, it & 1)) flags[0] = 1;
    tc_fence_after();
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float v[32];
      tmem_ld32(tO + lane_off + q4 * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) o[q4 * 32 + j] = o[q4 * 32 + j] * alpha + v[j];
    }
    tc_fence_before();
    __syncthreads();
    // the stage is free again: prefetch chunk c + 2 into it
    if (t == 0 && c + 2 < c_end && !flags[0]) load_chunk(c + 2, st);
    ok = !flags[0];
  }

  const int hh = t >> 4;
  __nv_bfloat16* dst = p.out + ((int64_t)(s * kGamma + r) * p.nh + g * group + hh) * 128;
  if (!ok) {
    if (t == 0) atomicOr(p.status, DFLASH_DEV_TIMEOUT);
    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
  } else if (nsplit == 1) {
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
    for (int d8 = 0; d8 < 16; ++d8) {
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(o[d8 * 8 + 2 * e] * inv, o[d8 * 8 + 2 * e + 1] * inv);
        pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      reinterpret_cast<uint4*>(dst)[d8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  } else {
    // partial (O unnormalised, m, l) of this split; attn_combine_kernel merges the splits
    const int64_t slot = (int64_t)unit * gridDim.y + split;
#pragma unroll
    for (int i = 0; i < 128; i += 4)
      __stcg(o_part_at(p.o_part, slot, t, i >> 2), make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]));
    __stcg(reinterpret_cast<float2*>(p.ml_part + (slot * 128 + t) * 2), make_float2(m_run, l_run));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------------------
// Kernel for long key ranges: stream-K over the key chunks of the whole batch.  The chunks of
// every (sequence, kv head) unit, in unit order, form one index space of W chunks; CTA b of a
// one-CTA-per-SM grid of G takes chunks [b W / G, (b + 1) W / G) whatever the context lengths,
// so every SM streams the same number of K/V bytes and there is no tail wave.  The range falls
// into segments (unit u, chunks [c_lo, c_hi) of it): a segment that covers its unit whole
// writes the normalised output, the others write fp32 partials (O, m, l) into slot b + u, which
// is unique (along the segments of the batch, b + u grows at every step), merged by
// attn_combine_kernel.  W, the CTA's range and its first unit come from ctx_lens on the device,
// so a captured graph replayed with new context lengths stays balanced.
//
// Inside a CTA the pipeline runs on from one segment into the next.  Keys go in super-chunks of
// two 64-key chunks (128 keys): warp 8 streams their K/V pages into three 64 KB buffers (two
// super-chunks of look-ahead: at full HBM load a page copy takes longer than one softmax pass),
// warp 9 issues the MMAs, warps 0-7 run the softmax: warps w and w + 4 share the TMEM lanes of
// rows 32 (w % 4) .. + 31 and take one 64-key chunk each (their partial row maxima and sums
// meet in shared memory), so two warps per scheduler hide each other's latencies.  While the
// softmax works on super-chunk i, the tensor cores already compute S of super-chunk i + 1 into
// the second TMEM buffer.  Per super-chunk: one max pass and one exp pass (ex2.approx) over the
// scores of a row, P written back as bf16 pairs over its own S columns and read from TMEM by
// the P V MMA, O accumulated in TMEM and rescaled there only when a row's running max grows.
// The next segment's queries are copied in (cp.async) once the last S of the current one is
// done.  Loops stay rolled.  226 KB of shared memory and 512 TMEM columns: one CTA per SM.
constexpr int kScChunks = 2;                                 // chunks per super-chunk
constexpr int kScBuf = kScChunks * kKVStage;                 // 64 KB of K/V per buffer
constexpr int kScBufs = 3;                                   // K/V buffers (super-chunks in flight)
constexpr int kScKV = kScBuf / 2;                            // the K (or V) half of a buffer: 32 KB
constexpr int kChunkKV = kPagesPerChunk * kTileBytes;        // one chunk's K (or V) pages: 16 KB
constexpr int kScCtl = 2560;                                 // barriers, plan, row exchange
constexpr int kScSmem = kQBytes + kScBufs * kScBuf + kScCtl + 128;
constexpr int kScThreads = 352;                              // 8 softmax warps, K producer, MMA, V producer
constexpr int kScSoft = 256;
constexpr int kScWaves = 4;  // partial slots per SM the compact kernel's split size allows

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Chunks unit u visits (0 for a context length out of range), its context and first key.
__device__ __forceinline__ int sk_unit_chunks(const AttnParams& p, int u, int* ctx, int* k0) {
  const int c = __ldg(p.ctx_lens + u / p.nkv);
  *ctx = c;
  *k0 = 0;
  if (c < 0 || c > p.max_ctx || c + kGamma > p.mpps * kPage) return 0;
  return chunk_range(p.window, c, k0);
}

// In the index space a unit with chunks occupies kSkUnitCost slots of no work before them: the
// cost of a segment (its queries, the pipeline restart, its output) in chunks, so a CTA whose
// range opens several segments gets fewer chunks.
constexpr int kSkUnitCost = 8;
__host__ __device__ __forceinline__ long long sk_slots(int nch) { return nch > 0 ? nch + kSkUnitCost : 0; }

// CTA b of G = min(grid, W) owns global chunks [lo, hi) = [floor(b W / G), floor((b + 1) W / G))
// (never empty); global chunk x belongs to CTA ceil((x + 1) G / W) - 1.
__host__ __device__ __forceinline__ int sk_owner(int64_t x, int64_t W, int G) {
  return (int)(((x + 1) * G + W - 1) / W) - 1;
}

struct SkSeg {
  int u, s, g, ctx, k0, nch;  // unit, its sequence, kv head, context, first key, chunks
  int c_lo, c_hi;             // this CTA's chunks of the unit
};

// The segments of index range [lo, hi), walked unit by unit from unit u (first slot pu).
struct SkWalk {
  int64_t lo, hi, pu;
  int u, units;
  __device__ bool next(const AttnParams& p, SkSeg& sg) {
    while (pu < hi && u < units) {
      int ctx, k0;
      const int nch = sk_unit_chunks(p, u, &ctx, &k0);
      const int64_t first = pu + kSkUnitCost;  // the unit's first chunk
      const int uu = u;
      pu += sk_slots(nch);
      ++u;
      if (nch == 0 || hi <= first || lo >= first + nch) continue;  // no chunk of this unit in range
      sg.u = uu;
      sg.s = uu / p.nkv;
      sg.g = uu % p.nkv;
      sg.ctx = ctx;
      sg.k0 = k0;
      sg.nch = nch;
      sg.c_lo = (int)(lo > first ? lo - first : 0);
      sg.c_hi = (int)(hi - first < nch ? hi - first : nch);
      return true;
    }
    return false;
  }
};

// The super-chunks of a walk in order (the MMA issuer looks one ahead).
struct SkIt {
  SkWalk w;
  SkSeg sg;
  int j, nsc, seg;
  bool valid;
  __device__ void start(const AttnParams& p, const SkWalk& w0) {
    w = w0;
    seg = -1;
    j = nsc = 0;
    valid = false;
    step(p);
  }
  __device__ void step(const AttnParams& p) {
    if (valid && j + 1 < nsc) {
      ++j;
      return;
    }
    valid = w.next(p, sg);
    if (valid) {
      ++seg;
      j = 0;
      nsc = (sg.c_hi - sg.c_lo + kScChunks - 1) / kScChunks;
    }
  }
  __device__ int nchk() const { return min(kScChunks, sg.c_hi - sg.c_lo - j * kScChunks); }
};

struct SkShared {
  uint64_t k_full[kScBufs], k_empty[kScBufs], v_full[kScBufs], v_empty[kScBufs];
  uint64_t s_full[2], p_full[2], o_done[2], q_full;
  uint32_t tmem_slot;
  int flags[2];
  long long red[16];
  long long W, pu0;
  int u0, found;
  float xm[2][2][128];  // [super-chunk parity][half][row]: partial row maxima (and sums at a segment's end)
};
static_assert(sizeof(SkShared) <= kScCtl, "stream-K control block overflows its slot");

// This CTA's walk: W by a block reduction over the sequences, then the sequence holding chunk
// lo by a block scan (its first unit starts the walk).  All kScThreads threads.
__device__ SkWalk sk_plan(const AttnParams& p, SkShared& sh, int t) {
  const int warp = t >> 5, lane = t & 31, nwarps = kScThreads / 32;
  long long mine = 0;
  for (int s = t; s < p.nb; s += kScThreads) {
    int ctx, k0;
    mine += sk_slots(sk_unit_chunks(p, s * p.nkv, &ctx, &k0));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) sh.red[warp] = mine;
  if (t == 0) sh.found = 0;
  __syncthreads();
  long long tot = 0;
  for (int w = 0; w < nwarps; ++w) tot += sh.red[w];
  const long long W = tot * p.nkv;
  // fewer chunks than CTAs: the first W CTAs take one each (every range is non-empty)
  const int G = (int)min((long long)gridDim.x, W), b = blockIdx.x;
  SkWalk wk;
  wk.lo = b < G ? (int64_t)b * W / G : 0;
  wk.hi = b < G ? (int64_t)(b + 1) * W / G : 0;
  wk.units = p.nb * p.nkv;
  wk.u = wk.units;
  wk.pu = wk.hi;
  __syncthreads();  // every thread has read red[]
  if (wk.lo >= wk.hi) return wk;
  long long carry = 0;
  for (int s0 = 0; s0 < p.nb; s0 += kScThreads) {
    const int s = s0 + t;
    int ctx, k0;
    const long long n = s < p.nb ? sk_slots(sk_unit_chunks(p, s * p.nkv, &ctx, &k0)) * p.nkv : 0;
    long long inc = n;  // inclusive scan: warp, then across warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) sh.red[warp] = inc;
    __syncthreads();
    long long before = carry;
    for (int w = 0; w < warp; ++w) before += sh.red[w];
    long long tile = 0;
    for (int w = 0; w < nwarps; ++w) tile += sh.red[w];
    const long long excl = before + inc - n;
    if (n > 0 && excl <= wk.lo && wk.lo < excl + n) {
      sh.u0 = s * p.nkv;
      sh.pu0 = excl;
      sh.found = 1;
    }
    carry += tile;
    __syncthreads();
    if (sh.found) break;
  }
  if (sh.found) {
    wk.u = sh.u0;
    wk.pu = sh.pu0;
  }
  return wk;
}

__global__ void __launch_bounds__(kScThreads, 1) attn_sk_kernel(const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  // no-swizzle operand tiles and bulk copies need 16-byte alignment
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* sQ = smem;
  // K slot b at sKV + b * kScKV, V slot b at sKV + (kScBufs + b) * kScKV; in a slot, chunk ci's
  // 4 pages at ci * kChunkKV
  uint8_t* sKV = sQ + kQBytes;
  SkShared& sh = *reinterpret_cast<SkShared*>(sKV + kScBufs * kScBuf);
  volatile int* flags = sh.flags;

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int group = p.nh / p.nkv;
  // a context length out of range contributes no chunks; CTA 0 reports it
  for (int s = t; blockIdx.x == 0 && s < p.nb; s += kScThreads) {
    const int c = __ldg(p.ctx_lens + s);
    if (c < 0 || c > p.max_ctx || c + kGamma > p.mpps * kPage) atomicOr(p.status, DFLASH_DEV_BAD_CTX);
  }
  const SkWalk walk = sk_plan(p, sh, t);
  if (walk.lo >= walk.hi || walk.u >= walk.units) return;  // nothing for this CTA

  if (t == 0) {
    for (int i = 0; i < kScBufs; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.k_empty[i], 1);
      mbar_init(&sh.v_full[i], 1);
      mbar_init(&sh.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_full[i], kScSoft);
    }
    mbar_init(&sh.o_done[0], 1);
    mbar_init(&sh.o_done[1], 1);
    mbar_init(&sh.q_full, kScSoft);
    flags[0] = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&sh.tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;
  const uint32_t tS[2] = {tmem, tmem + 128}, tO = tmem + 256;
  constexpr uint32_t idesc_s = idesc_bf16(128, kKC);
  constexpr uint32_t idesc_o = idesc_bf16(128, 128);
  pdl_trigger();

  if (warp == 8 || warp == 10) {
    // ---------------- page producers: warp 8 the K pages, warp 10 the V pages, each into its own
    // ring of three slots.  A K slot is free once the S MMA that read it is done, a V slot once
    // its P V is done, so the K copies run a softmax pass further ahead than the V copies.  Lane
    // l < 8 copies page l % 4 of chunk l / 4 of a super-chunk; the page ids of the next
    // super-chunk are fetched while the warp waits for a free slot.
    const int kv = warp == 10;
    uint64_t* full = kv ? sh.v_full : sh.k_full;
    uint64_t* empty = kv ? sh.v_empty : sh.k_empty;
    bool waited = false, stop = false;
    SkWalk w = walk;
    SkSeg sg;
    int i = 0;
    while (!stop && w.next(p, sg)) {
      const int32_t* pt = p.page_tables + (int64_t)sg.s * p.mpps;
      const int npages_seq = (sg.ctx + kGamma + kPage - 1) / kPage;
      const int safe_keys = sg.ctx & ~(kPage - 1);
      const int n = sg.c_hi - sg.c_lo, nsc = (n + kScChunks - 1) / kScChunks;
      auto page_of = [&](int jj) {
        const int ci = lane >> 2, q = lane & 3;
        const int c = sg.c_lo + jj * kScChunks + ci;
        if (lane >= kScChunks * kPagesPerChunk || jj >= nsc || c >= sg.c_hi) return 0;
        const int pg = (sg.k0 + c * kKC) / kPage + q;
        return __ldg(pt + (pg < npages_seq ? pg : 0));
      };
      int page = page_of(0);
      for (int jj = 0; jj < nsc; ++jj, ++i) {
        const int b = i % kScBufs;
        if (i >= kScBufs && !mbar_wait_ab(&empty[b], ((i / kScBufs) - 1) & 1, flags)) {
          flags[0] = 1;
          stop = true;
          break;
        }
        const int nchk = min(kScChunks, n - jj * kScChunks);
        if (!waited && sg.k0 + (sg.c_lo + jj * kScChunks + nchk) * kKC > safe_keys) {  // holds block rows
          pdl_wait();
          waited = true;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[b], nchk * kChunkKV);
        __syncwarp();
        if (lane < nchk * kPagesPerChunk) {
          int pg = page;
          if (pg < 0 || pg >= p.g.num_pages) {
            atomicOr(p.status, DFLASH_DEV_BAD_PAGE);
            pg = 0;
          }
          uint8_t* d = sKV + (kv * kScBufs + b) * kScKV + (lane >> 2) * kChunkKV + (lane & 3) * kTileBytes;
          bulk_load(d, p.pool + tile_base(p.g, p.layer, pg, kv, sg.g), kTileBytes, &full[b]);
        }
        page = page_of(jj + 1);
      }
    }
    if (!waited) pdl_wait();
    __syncwarp();
  } else if (warp == 9) {
    // ---------------- MMA issuer (lane 0): S of super-chunk i + 1 and P V of i are independent;
    // each goes out as soon as its inputs are there (S: the K copy, and the segment's queries
    // for a segment's first super-chunk; P V: the softmax's P and the V copy), so a late copy
    // never holds back the MMA that frees a slot
    if (lane == 0) {
      auto issue_s = [&](const SkIt& it, int i) {
        const int b = i & 1, kb = i % kScBufs;
        tc_fence_after();
        if (!flags[0]) {
          for (int ci = 0; ci < it.nchk(); ++ci) {
            const uint8_t* sK = sKV + kb * kScKV + ci * kChunkKV;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_bf16(tS[b] + ci * kKC, desc_noswz(sQ + k * 256, 128, 2048), desc_noswz(sK + k * 256, 128, 2048),
                       idesc_s, k > 0 ? 1u : 0u);
          }
        }
        mma_commit(&sh.s_full[b]);
        mma_commit(&sh.k_empty[kb]);  // the K slot is free once these MMAs are done
      };
      auto s_ready = [&](const SkIt& it, int i) {
        return (it.j != 0 || mbar_test_wait(&sh.q_full, it.seg & 1)) &&
               mbar_test_wait(&sh.k_full[i % kScBufs], (i / kScBufs) & 1);
      };
      SkIt cur, nx;
      cur.start(p, walk);
      nx = cur;
      nx.step(p);
      if (cur.valid) {
        if (!mbar_wait_ab(&sh.q_full, 0, flags)) flags[0] = 1;
        if (!mbar_wait_ab(&sh.k_full[0], 0, flags)) flags[0] = 1;
        issue_s(cur, 0);
      }
      for (int i = 0; cur.valid; ++i) {
        const int b = i & 1, kb = i % kScBufs;
        bool s_out = !nx.valid, pv_out = false;
        for (long long spin = 0; !(s_out && pv_out); ++spin) {
          if (spin > kSpinLimit) flags[0] = 1;
          const bool give_up = flags[0];  // after a timeout: commits only, no MMAs
          if (!s_out && (give_up || s_ready(nx, i + 1))) {
            issue_s(nx, i + 1);
            s_out = true;
          }
          if (!pv_out && (give_up || (mbar_test_wait(&sh.p_full[b], (i >> 1) & 1) &&
                                      mbar_test_wait(&sh.v_full[kb], (i / kScBufs) & 1)))) {
            tc_fence_after();
            if (!give_up) {
              const int nchk = cur.nchk();
              for (int kk = 0; kk < nchk * kPagesPerChunk; ++kk) {  // 16 keys = 8 TMEM columns of P each
                const int ci = kk / kPagesPerChunk, pg = kk % kPagesPerChunk;
                const uint8_t* sV = sKV + (kScBufs + kb) * kScKV + ci * kChunkKV + pg * kTileBytes;
                mma_bf16_tmem_a(tO, tS[b] + ci * kKC + pg * 8, desc_noswz(sV, 128, 256), idesc_o,
                                (cur.j > 0 || kk > 0) ? 1u : 0u);
              }
            }
            mma_commit(&sh.v_empty[kb]);
            mma_commit(&sh.o_done[b]);
            pv_out = true;
          }
        }
        cur = nx;
        if (nx.valid) nx.step(p);
      }
    }
    __syncwarp();
  } else {
    // ---------------- warps 0-7: queries, softmax, output.  Thread t holds row t % 128 (head
    // row / 16, token row % 16); half hf = warp / 4 takes chunk hf of each super-chunk and the
    // O columns 64 hf .. 64 hf + 63.
    pdl_wait();
    const int row = t & 127, hf = warp >> 2, r = row & 15, hh = row >> 4;
    const int pair_bar = 1 + (warp & 3);  // named barrier of warps w % 4 and w % 4 + 4
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float scale_log2 = 1.4426950408889634f / sqrtf(128.f);
    // a unit's queries into sQ: 2048 pieces of 16 bytes over the 256 softmax threads
    auto load_q = [&](const SkSeg& q) {
#pragma unroll
      for (int k = 0; k < 8; ++k) stage_q_piece(sQ, p.q, q.s, q.g, p.nh, k * kScSoft + t);
    };
    auto q_ready = [&]() {
      cp_async_wait_all();
      fence_proxy_async_smem();
      mbar_arrive(&sh.q_full);
    };
    SkWalk w = walk;
    SkSeg sg, nsg;
    bool have = w.next(p, sg);
    if (have) {
      load_q(sg);
      q_ready();
    }
    int i = 0;
    while (have) {
      const bool more = w.next(p, nsg);
      const int n = sg.c_hi - sg.c_lo, nsc = (n + kScChunks - 1) / kScChunks;
      const int nvis = sg.ctx + block_width(p.widths, sg.s);  // keys past the active block width are masked
      const int pos_q = sg.ctx + r;
      float m_run = -FLT_MAX, l_half = 0.f;
#pragma unroll 1
      for (int j = 0; j < nsc; ++j, ++i) {
        const int b = i & 1;
        const int nchk = min(kScChunks, n - j * kScChunks);
        const bool mine = hf < nchk;  // this half's chunk exists
        if (!mbar_wait_ab(&sh.s_full[b], (i >> 1) & 1, flags)) flags[0] = 1;
        tc_fence_after();
        const bool last = j == nsc - 1;
        if (last && more) load_q(nsg);  // every S of this segment is done: sQ is free
        // every key of the super-chunk visible to every row: no masking
        const int kb = sg.k0 + (sg.c_lo + j * kScChunks) * kKC;
        const bool full = kb + nchk * kKC <= nvis && (p.window <= 0 || sg.ctx + kGamma - 1 - kb < p.window);
        const int kh = kb + hf * kKC;  // first key of this half's chunk
        // this half's 64 scores, read from TMEM once (the max and the exp pass both use them)
        float sv[64];
        float mc = -FLT_MAX;
        if (mine) {
          tmem_ld64(tS[b] + lane_off + hf * kKC, sv);
          if (!full) {
#pragma unroll
            for (int e = 0; e < 64; ++e) {
              const int key = kh + e;
              if (!(key < nvis && (p.window <= 0 || pos_q - key < p.window))) sv[e] = -FLT_MAX;
            }
          }
#pragma unroll
          for (int e = 0; e < 64; ++e) mc = fmaxf(mc, sv[e]);
        }
        // the row's maximum over both chunks (buffer by super-chunk parity: the next write to
        // this one comes after the next exchange, which the partner reaches after its read)
        sh.xm[b][hf][row] = mc;
        named_barrier(pair_bar, 64);
        mc = fmaxf(mc, sh.xm[b][hf ^ 1][row]);
        // The reference maximum m_run moves only when the chunk's maximum exceeds it by more than
        // 8 (log2 units): otherwise P = 2^(s c - m_run) <= 2^8 stays exact in fp32 and bf16, and O
        // and l need no rescale (the final O / l is the same).  max(s) * c == max(s * c) for c > 0.
        const float mcs = mc == -FLT_MAX ? -FLT_MAX : mc * scale_log2;
        const bool grow = mcs > m_run + 8.f;
        const float m_new = grow ? mcs : m_run;
        const float alpha = (grow && m_run != -FLT_MAX) ? ex2_approx(m_run - m_new) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // this half's O columns hold the segment's super-chunks before this one once P V of
          // i - 1 is done.  P V of i alternate between two barriers: S(i) went out after P V of
          // i - 2, so the barrier of i - 1 is at most one phase behind and the parity wait exact
          if (!mbar_wait_ab(&sh.o_done[(i - 1) & 1], ((i - 1) >> 1) & 1, flags)) flags[0] = 1;
          tc_fence_after();
#pragma unroll 1
          for (int q4 = 0; q4 < 2; ++q4) {
            float v[32];
            tmem_ld32(tO + lane_off + (2 * hf + q4) * 32, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] *= alpha;
            tmem_st32(tO + lane_off + (2 * hf + q4) * 32, v);
          }
        }
        // P = 2^(s c - m) as bf16 pairs: the 64 keys of chunk hf into the first 32 of its own 64
        // S columns (scores already in registers; the other half's columns stay untouched);
        // masked keys hold -FLT_MAX, whose exp2 is 0 (also while a row has seen no visible key:
        // m_new is -FLT_MAX then and the offset is taken as 0)
        float lsum = 0.f;
        if (mine) {
          const float mneg = m_new == -FLT_MAX ? 0.f : -m_new;
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(ex2_approx(fmaf(sv[2 * e], scale_log2, mneg)),
                                                            ex2_approx(fmaf(sv[2 * e + 1], scale_log2, mneg)));
            lsum += __low2float(h2) + __high2float(h2);
            pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          tmem_st32u(tS[b] + lane_off + hf * kKC, pk);
        }
        l_half = l_half * alpha + lsum;
        m_run = m_new;
        tc_fence_before();
        mbar_arrive(&sh.p_full[b]);
        if (last && more) q_ready();
      }
      // the row's sum over both halves (slot parity of super-chunk i + 1, written after the next
      // exchange; the barrier first keeps the partner's last maximum read ahead of this write)
      named_barrier(pair_bar, 64);
      sh.xm[(i + 1) & 1][hf][row] = l_half;
      named_barrier(pair_bar, 64);
      const float l_run = l_half + sh.xm[(i + 1) & 1][hf ^ 1][row];
      // the segment's O (its last P V done, hence every earlier one): normalised bf16 rows when
      // it covers the unit, else an fp32 partial
      if (!mbar_wait_ab(&sh.o_done[(i - 1) & 1], ((i - 1) >> 1) & 1, flags)) flags[0] = 1;
      tc_fence_after();
      const bool whole = sg.c_lo == 0 && sg.c_hi == sg.nch;
      if (!flags[0]) {
        __nv_bfloat16* dst = p.out + ((int64_t)(sg.s * kGamma + r) * p.nh + sg.g * group + hh) * 128 + hf * 64;
        const int64_t slot = (int64_t)blockIdx.x + sg.u;
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
        for (int q4 = 0; q4 < 2; ++q4) {
          float v[32];
          tmem_ld32(tO + lane_off + (2 * hf + q4) * 32, v);
          if (whole) {
#pragma unroll
            for (int d8 = 0; d8 < 4; ++d8) {
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[d8 * 8 + 2 * e] * inv, v[d8 * 8 + 2 * e + 1] * inv);
                pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
              }
              reinterpret_cast<uint4*>(dst)[q4 * 4 + d8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              __stcg(o_part_at(p.o_part, slot, row, hf * 16 + q4 * 8 + (e >> 2)),
                     make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]));
          }
        }
        if (!whole && hf == 0)
          __stcg(reinterpret_cast<float2*>(p.ml_part + (slot * 128 + row) * 2), make_float2(m_run, l_run));
      }
      tc_fence_before();  // O read out before the next segment's first P V overwrites it
      sg = nsg;
      have = more;
    }
    if (flags[0]) {
      if (t == 0) atomicOr(p.status, DFLASH_DEV_TIMEOUT);
      for (int k = 0; k < 2000; ++k) __nanosleep(1000);  // copies still in flight land first
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Merge the split partials of every (sequence, kv head) unit with more than one split, in
// split order with a running maximum: o = sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q.
// Block (unit, rb) owns rows 4 rb .. 4 rb + 3, 4 dims per thread.
// sk_grid > 0: the partials of the stream-K kernel over sk_grid CTAs (the unit's splits are
// the CTAs whose chunk ranges overlap it, slots b + unit); else those of the compact kernel
// (splits_launched slots per unit).
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnParams p, int splits_launched, int sk_grid) {
  pdl_trigger();  // the next projection may start streaming its weights
  pdl_wait();
  const int unit = blockIdx.x, t = threadIdx.x;
  const int s = unit / p.nkv, g = unit % p.nkv;
  const int ctx = p.ctx_lens[s];
  if (ctx < 0 || ctx > p.max_ctx || ctx + kGamma > p.mpps * kPage) return;
  int k0;
  const int nch = chunk_range(p.window, ctx, &k0);
  int nsplit;
  int64_t base;
  if (sk_grid > 0) {
    // the unit's first chunk in the batch's chunk space, and the space's size
    __shared__ long long red[2][4];
    long long before = 0, all = 0;
    for (int s2 = t; s2 < p.nb; s2 += 128) {
      const int c2 = __ldg(p.ctx_lens + s2);
      int f2;
      const long long n2 =
          (c2 < 0 || c2 > p.max_ctx || c2 + kGamma > p.mpps * kPage) ? 0 : sk_slots(chunk_range(p.window, c2, &f2));
      all += n2;
      if (s2 < s) before += n2;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    if ((t & 31) == 0) {
      red[0][t >> 5] = before;
      red[1][t >> 5] = all;
    }
    __syncthreads();
    const long long first =
        (red[0][0] + red[0][1] + red[0][2] + red[0][3]) * p.nkv + (long long)g * sk_slots(nch) + kSkUnitCost;
    const long long W = (red[1][0] + red[1][1] + red[1][2] + red[1][3]) * p.nkv;
    const int G = (int)min((long long)sk_grid, W);  // CTAs with a non-empty range
    const int b0 = sk_owner(first, W, G), b1 = sk_owner(first + nch - 1, W, G);
    if (b0 == b1) return;  // one CTA covered the unit and wrote the output
    nsplit = b1 - b0 + 1;
    base = (int64_t)b0 + unit;
  } else {
    nsplit = (nch + p.chunks_per_split - 1) / p.chunks_per_split;
    if (nsplit <= 1 || nsplit > splits_launched) return;
    base = (int64_t)unit * splits_launched;
  }
  // thread t: row 4 rb + t % 4, dims 4 (t / 4) ..: the block reads 2 KB contiguous per split
  const int row = blockIdx.y * 4 + (t & 3), db = t >> 2, d0 = db * 4;
  float M = -FLT_MAX, L = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  for (int q0 = 0; q0 < nsplit; q0 += 4) {
    float2 ml[4];
    float4 ov[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t sl = base + q0 + u;
      const bool v = q0 + u < nsplit;
      ml[u] = v ? __ldcg(reinterpret_cast<const float2*>(p.ml_part + (sl * 128 + row) * 2)) : make_float2(-FLT_MAX, 0.f);
      ov[u] = v ? __ldcg(o_part_at(p.o_part, sl, row, db)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
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
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(a0 * inv, a1 * inv);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(a2 * inv, a3 * inv);
  const int hh = row >> 4, r = row & 15;
  __nv_bfloat16* dst = p.out + ((int64_t)(s * kGamma + r) * p.nh + g * (p.nh / p.nkv) + hh) * 128 + d0;
  *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<const uint32_t*>(&h0),
                                              *reinterpret_cast<const uint32_t*>(&h1));
}

}  // namespace

// Partial slots any launch needs: the compact kernel's units * splits <= kScWaves * num_sms +
// units (splits = ceil(nch / cps) with cps >= units * nch / (kScWaves * num_sms)); the stream-K
// kernel's slots b + unit < num_sms + units.
int64_t attn_tc_partial_slots(int num_sms, int max_units) { return kScWaves * (int64_t)num_sms + max_units; }

cudaError_t launch_attn_tc(AttnParams p, int nb, int max_ctx_len, int num_sms, cudaStream_t st) {
  static std::atomic<unsigned long long> attr{0}, attr2{0};
  if (cudaError_t e = smem_attr_once(attn_tc_kernel, kSmem, attr); e != cudaSuccess) return e;
  if (cudaError_t e = smem_attr_once(attn_sk_kernel, kScSmem, attr2); e != cudaSuccess) return e;
  const int units = nb * p.nkv;
  p.nb = nb;
  p.max_ctx = max_ctx_len;
  // the most chunks any sequence with ctx <= max_ctx_len visits
  int k0;
  int nch = chunk_range(0, max_ctx_len, &k0);
  if (p.window > 0) nch = std::min(nch, (p.window + kGamma + kPage + kKC - 1) / kKC);
  int cps = (units * nch + num_sms - 1) / num_sms;
  if (cps < 1) cps = 1;
  cudaLaunchAttribute aa[1];
  aa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  aa[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t ac = {};
  ac.stream = st;
  ac.attrs = aa;
  ac.numAttrs = 1;
  // many chunks per SM: the stream-K kernel (one CTA per SM, an equal share of the batch's
  // chunks each); a few: the compact kernel, split on the host from max_ctx_len (it fits beside
  // a projection CTA on one SM, so it overlaps the QKV kernel under programmatic launch)
  const bool sk = cps >= 4;
  int splits_l = 1;
  cudaError_t e;
  if (sk) {
    ac.gridDim = dim3(num_sms);
    ac.blockDim = dim3(kScThreads);
    ac.dynamicSmemBytes = kScSmem;
    e = cudaLaunchKernelEx(&ac, attn_sk_kernel, p);
  } else {
    splits_l = (nch + cps - 1) / cps;
    p.chunks_per_split = cps;
    ac.gridDim = dim3(units, splits_l);
    ac.blockDim = dim3(128);
    ac.dynamicSmemBytes = kSmem;
    e = cudaLaunchKernelEx(&ac, attn_tc_kernel, p);
  }
  if (e != cudaSuccess || (!sk && splits_l == 1)) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units, 32);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cfg.attrs = aa;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel, p, splits_l, sk ? num_sms : 0);
}

}  // namespace dflash
