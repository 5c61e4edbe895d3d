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

#include <atomic>

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

constexpr int kMaxDevices = 64;
std::atomic<unsigned long long*> g_scratch_ptr[kMaxDevices];

// The device address of g_check_scratch on the current device, looked up once
// per device (in host code the symbol's name is only a host-side stand-in).
cudaError_t scratch_on_current_device(unsigned long long** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_check_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev].store(p, std::memory_order_release);
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
  const int64_t n = rows * (cols / 32);
  if (n > NM_CHECK_NOALLOC_MAX_WORDS) return -NM_ERR_WORKSPACE;
  if (n == 0) return 0;
  unsigned long long* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return -NM_ERR_CUDA;
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
