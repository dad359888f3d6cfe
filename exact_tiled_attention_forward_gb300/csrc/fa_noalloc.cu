// fa_forward_noalloc: the fused forward for callers that cannot allocate device
// memory. Same kernels and same work split as fa_forward; the only difference
// is where the split-key and decode partials live. fa_forward takes them from a
// stream-ordered pool; this entry point uses a fixed array that is part of the
// library's own device image, so no call ever allocates.
//
// Who needs this: code that runs where a device allocation is not allowed or
// not safe — a serving loop that must never block on cudaMalloc/cudaFree (both
// can synchronise the device and take unbounded time), a process whose device
// memory is entirely pre-reserved by another allocator so any new request
// fails, or a deployment that must size all of its memory before it starts.
#include "fa_internal.h"
#include "fa.h"

#include <mutex>

namespace fa {
namespace {

// Scratch for the partials: per split prefill CTA, kBlockRows rows of FP32
// O (d values) plus (m, l); per decode chunk, R rows of the same. 32 MiB holds
// up to 252 split CTAs at d = 128 (the 1-head N = 8192 workload uses 128 of
// them, 17 MiB; batch-16 decode over 8192 keys uses 17 MiB). Every GPU that
// loads libfa holds this array until the process exits. Nothing in it needs
// to start at zero: every partial row a merge reads is written first by the
// same call.
constexpr size_t kScratchBytes = 32u << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the array, looked up once per device with that device current.
void* scratch_address(int* err) {
  static void* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *err = (int)(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *err = (int)e;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace fa

using namespace fa;

namespace fa {
namespace {

int scratch_acquire(size_t bytes, cudaStream_t, void** ptr) {
  if (bytes > kScratchBytes) return FA_ERR_TOO_LARGE;
  int err = 0;
  void* base = scratch_address(&err);
  if (!base) return cuda_fail((cudaError_t)err);
  *ptr = base;
  return FA_OK;
}

const WorkspaceSource kScratchSource{scratch_acquire, nullptr};

}  // namespace
}  // namespace fa

extern "C" int fa_forward_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal,
                                  float scale, void* stream) {
  return forward_impl(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, causal, scale,
                      static_cast<cudaStream_t>(stream), kScratchSource);
}
