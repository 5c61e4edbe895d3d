// check_noalloc.cu -- mask validation that never allocates device memory.
//
// nm_check_masks needs an 8-byte device counter and gets it with
// cudaMallocAsync on every call.  Some callers cannot allow that: a serving
// process that has handed all device memory to its own caching allocator or a
// fixed arena at start-up (an allocation behind the allocator's back can fail
// or fragment that budget), or a latency-critical loop where a stream-ordered
// allocation may stall on the memory pool.  nm_check_masks_noalloc gives them
// the same count with its scratch in a fixed array that lives in this
// library's own device image: every GPU that loads the library holds it until
// the process exits, and no call allocates anything.
//
// The kernel is a deterministic two-pass variant of check_masks_kernel: pass 1
// writes one partial count per block (no atomics), pass 2 adds the partials in
// block order into one total.  Every slot a call reads is written earlier in
// the same call, so nothing needs clearing between calls; but all calls share
// the array, so calls that overlap on the GPU (two streams, two host threads)
// race and must be serialised by the caller.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/nm_spmv.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWordsPerThread = 64;
constexpr int64_t kWordsPerBlock = (int64_t)kThreads * kWordsPerThread;  // 16384
constexpr int kMaxBlocks = 4096;

static_assert(NM_CHECK_NOALLOC_MAX_WORDS == kWordsPerBlock * kMaxBlocks,
              "header limit must match the scratch array");

// [0, kMaxBlocks): per-block partial counts; [kMaxBlocks]: the total.
static __device__ __align__(256) unsigned long long g_check_scratch[kMaxBlocks + 1];

__global__ void __launch_bounds__(kThreads) count_partial_kernel(const uint32_t* __restrict__ masks,
                                                                 int64_t n,
                                                                 unsigned long long* partial) {
  __shared__ unsigned warp_bad[kThreads / 32];
  const int64_t base = (int64_t)blockIdx.x * kWordsPerBlock;
  unsigned bad = 0;
#pragma unroll 4
  for (int j = 0; j < kWordsPerThread; ++j) {
    const int64_t i = base + (int64_t)j * kThreads + threadIdx.x;  // coalesced
    if (i < n) bad += (__popc(masks[i]) != 16) ? 1u : 0u;
  }
  bad = __reduce_add_sync(0xFFFFFFFFu, bad);
  if ((threadIdx.x & 31) == 0) warp_bad[threadIdx.x >> 5] = bad;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long s = 0;
    for (int w = 0; w < kThreads / 32; ++w) s += warp_bad[w];
    partial[blockIdx.x] = s;
  }
}

__global__ void sum_partials_kernel(unsigned long long* scratch, int blocks) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    unsigned long long s = 0;
    for (int b = 0; b < blocks; ++b) s += scratch[b];  // fixed order
    scratch[kMaxBlocks] = s;
  }
}

// The device address of g_check_scratch.  In host code the symbol's name is
// only a host-side stand-in; the address belongs to the module loaded into a
// CUDA context, so it is looked up (cudaGetSymbolAddress) once per context,
// with that context current, and cached under the context's unique id.  A
// context made after cudaDeviceReset, or a second driver-API context on the
// same device, has a new id and gets its own lookup.  The lookup also loads
// the module, which is why the first call in a context should come before any
// stream capture.  If the driver entry points for the context id cannot be
// had, the address is looked up on every call instead (a host-only query).
using CtxGetCurrentFn = int (*)(void** ctx);
using CtxGetIdFn = int (*)(void* ctx, unsigned long long* id);

struct CtxEntry {
  unsigned long long id;
  unsigned long long* ptr;
};

constexpr int kCachedContexts = 64;
std::mutex g_scratch_mutex;
CtxEntry g_scratch_cache[kCachedContexts];
int g_scratch_cached = 0;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
bool g_driver_looked_up = false;

// Unique id of the current context; false if there is none or it is unknown.
bool current_context_id(unsigned long long* id) {
  if (!g_driver_looked_up) {
    g_driver_looked_up = true;
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f1);
      g_ctx_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
  }
  if (!g_ctx_current || !g_ctx_id) return false;
  void* ctx = nullptr;
  if (g_ctx_current(&ctx) != 0 || ctx == nullptr) return false;
  return g_ctx_id(ctx, id) == 0;
}

cudaError_t scratch_in_current_context(unsigned long long** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long id = 0;
  if (current_context_id(&id)) {
    for (int i = 0; i < g_scratch_cached; ++i)
      if (g_scratch_cache[i].id == id) {
        *out = g_scratch_cache[i].ptr;
        return cudaSuccess;
      }
  }
  unsigned long long* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_check_scratch);
  if (e != cudaSuccess) return e;
  // the lookup made the device's context current if none was; cache under it
  if (current_context_id(&id)) {
    const int slot = g_scratch_cached < kCachedContexts ? g_scratch_cached++
                                                        : (int)(id % kCachedContexts);
    g_scratch_cache[slot] = {id, p};
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" int64_t nm_check_masks_noalloc(const uint32_t* masks, int64_t rows, int64_t cols,
                                          void* stream) {
  if (!masks) return -NM_ERR_NULL;
  if (rows < 0 || cols <= 0 || cols % 32 != 0) return -NM_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(masks) & 3u) != 0) return -NM_ERR_ALIGN;
  // bound before multiplying, so that no product can wrap past the limit
  const int64_t words = cols / 32;
  if (words > NM_CHECK_NOALLOC_MAX_WORDS || rows > NM_CHECK_NOALLOC_MAX_WORDS / words)
    return -NM_ERR_WORKSPACE;
  const int64_t n = rows * words;
  if (n == 0) return 0;
  unsigned long long* scratch = nullptr;
  if (scratch_in_current_context(&scratch) != cudaSuccess) return -NM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int blocks = (int)((n + kWordsPerBlock - 1) / kWordsPerBlock);
  count_partial_kernel<<<blocks, kThreads, 0, s>>>(masks, n, scratch);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    sum_partials_kernel<<<1, 32, 0, s>>>(scratch, blocks);
    e = cudaGetLastError();
  }
  unsigned long long total = 0;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&total, scratch + kMaxBlocks, sizeof(total), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? (int64_t)total : -NM_ERR_CUDA;
}
