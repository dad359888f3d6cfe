// fa_forward_noalloc: the fused forward for callers that cannot allocate device
// memory. Same kernel and same work split as fa_forward; the only difference is
// where the split-key partials live. fa_forward takes them from a
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

// Scratch for the split-key partials: per split CTA, kBlockRows rows of FP32
// O (d values) plus (m, l). 32 MiB holds up to 252 split CTAs at d = 128
// (the 1-head N = 8192 workload uses 128 of them, 17 MiB). Every GPU that
// loads libfa holds this array until the process exits. Nothing in it needs
// to start at zero: every partial row the merge reads is written first by
// the same call.
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

extern "C" int fa_forward_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal,
                                  float scale, void* stream) {
  const Shape s{B, H_q, H_kv, N_q, N_k, d};
  int st = validate(q, k, v, o, lse, s, scale);
  if (st != FA_OK) return st;
  if ((long long)B * H_q * N_q == 0) return FA_OK;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  if (N_k == 0 || B * H_kv == 0) return fill_empty(o, lse, (long long)B * H_q * N_q, d, strm);

  int* status = device_status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());

  FwdParams p{};
  p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q; p.N_k = N_k;
  p.causal = causal ? 1 : 0;
  p.kv_off = N_k - N_q;
  p.n_qb = (N_q + kBlockRows - 1) / kBlockRows;
  p.n_kv_tiles = (N_k + kTileN - 1) / kTileN;
  p.c = scale * 1.4426950408889634f;
  p.o = o;
  p.lse = lse;
  p.status = status;
  const long long blocks = (long long)B * H_q * p.n_qb;
  const int kv_eff = causal ? (p.n_kv_tiles + 1) / 2 : p.n_kv_tiles;
  const FwdPlan pl = plan_forward(blocks, kv_eff, causal != 0, d, num_sms());
  if (pl.units >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  p.u_full = pl.u_full;
  p.n_tail = pl.n_tail;
  p.s_tail = pl.s_tail;
  const long long units = pl.units;

  if (pl.n_tail > 0) {
    if (pl.part_bytes > kScratchBytes) return FA_ERR_TOO_LARGE;
    int err = 0;
    char* base = static_cast<char*>(scratch_address(&err));
    if (!base) return cuda_fail((cudaError_t)err);
    p.part_o = reinterpret_cast<float*>(base);
    p.part_ml = reinterpret_cast<float*>(base + (size_t)pl.n_tail * pl.s_tail * kBlockRows * d * 4);
  }

  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16_3d(&tq, q, d, N_q, (uint64_t)B * H_q, d, 128) ||
      !make_tmap_bf16_3d(&tk, k, d, N_k, (uint64_t)B * H_kv, d, 128) ||
      !make_tmap_bf16_3d(&tv, v, d, N_k, (uint64_t)B * H_kv, d, 128))
    return cuda_fail(cudaErrorInvalidValue);
  cudaError_t e = launch_fwd(d, tq, tk, tv, p, (int)units, strm);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}
