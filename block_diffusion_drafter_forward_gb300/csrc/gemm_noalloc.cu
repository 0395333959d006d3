// Split-K tensor-core projection GEMM that allocates no memory.
//
// Who needs it: callers that are not allowed to call cudaMalloc once they are running --
// an allocator-free serving loop that reserved all device memory up front, code running
// under a memory pool that owns the whole device, or an embedding runtime that forbids
// driver allocations after start-up.  The regular entry points take their scratch from
// buffers allocated by dflash_create; this one takes it from a fixed array that lives in
// the library's own device image instead.
//
// The scratch (split-K fp32 partials and per-tile arrival counters) is a file-scope
// __device__ array of fixed size.  Every GPU that loads the library holds it until the
// process exits.  All calls share it, so two calls that overlap on the GPU (different
// streams, or different host threads) race on it and produce garbage: serialise them.
// A bounded wait inside the kernel that gives up (only on a GPU starved for many seconds)
// leaves its tile unwritten; this entry point has no status word to report that.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "dflash_internal.cuh"
#include "gemm_tc.cuh"

namespace dflash {
namespace {

// 8 MiB of fp32 split-K partials and 4096 tile counters.
constexpr size_t kNoAllocPartials = 2u << 20;   // floats
constexpr int kNoAllocCounters = 4096;

static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];
static __device__ __align__(256) unsigned g_noalloc_counters[kNoAllocCounters];

struct NoAllocScratch {
  float* partials = nullptr;
  unsigned* counters = nullptr;
};

// Device addresses of the arrays, looked up with the device current.  (In host code the array
// names are host-side stand-ins, not device addresses.)  An address belongs to the context the
// library's module was loaded into: after cudaDeviceReset, or after the primary context was
// released and created again, the module is loaded anew and the arrays may move.  So the cache
// is keyed on the current context's unique id, and a new context means a new lookup.
std::mutex g_mu;
NoAllocScratch g_scratch[64];
unsigned long long g_ctx_id[64] = {};  // 0: not looked up yet

// Driver entry points through the runtime (the library does not link libcuda itself).
typedef CUresult (*PFN_ctx_get_current)(CUcontext*);
typedef CUresult (*PFN_ctx_get_id)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name, int version) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(ptr);
}

// Unique id of the calling thread's current context (0 if none or not available).
unsigned long long current_ctx_id() {
  static PFN_ctx_get_current get_current = nullptr;
  static PFN_ctx_get_id get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<PFN_ctx_get_current>("cuCtxGetCurrent", 4000);
    get_id = driver_fn<PFN_ctx_get_id>("cuCtxGetId", 12000);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

cudaError_t scratch_for_current_device(NoAllocScratch* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long id = current_ctx_id();
  if (id == 0 || id != g_ctx_id[dev]) {
    NoAllocScratch s;
    // the first lookup also makes the device's primary context current
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.partials), g_noalloc_partials);
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.counters), g_noalloc_counters);
    if (e != cudaSuccess) return e;
    g_scratch[dev] = s;
    g_ctx_id[dev] = current_ctx_id();
  }
  *out = g_scratch[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace dflash

extern "C" int dflash_gemm_bf16_noalloc(const void* W, int32_t N, int32_t K, const void* X, int32_t M, float* out,
                                        int32_t nsplit, dflash_stream stream) {
  using namespace dflash;
  if (!W || !X || !out) return DFLASH_EINVAL;
  if (N < 1 || M < 1 || K < 64 || K % 64 || nsplit < 1 || nsplit > kMaxSplits || nsplit > K / 64)
    return DFLASH_EINVAL;
  const int tn = pick_tn(M);
  const int64_t tiles = (int64_t)((N + 127) / 128) * ((M + tn - 1) / tn);
  if (tiles > kNoAllocCounters || (size_t)(tiles * nsplit * 128 * tn) > kNoAllocPartials)
    return DFLASH_ECAPACITY;  // beyond the fixed scratch: use dflash_gemm_bf16 / dflash_propose
  NoAllocScratch s;
  if (scratch_for_current_device(&s) != cudaSuccess) return DFLASH_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the counters must start at zero; a previous call that gave up may have left them set
  if (cudaMemsetAsync(s.counters, 0, sizeof(unsigned) * (size_t)tiles, st) != cudaSuccess) return DFLASH_ECUDA;
  GemmParams p;
  p.out = out;
  p.ldo = N;
  p.ws = s.partials;
  p.counters = s.counters;
  if (launch_gemm_tc(EPI_STORE, W, N, K, X, K, M, p, nsplit, st, false) != cudaSuccess) return DFLASH_ECUDA;
  return DFLASH_OK;
}
