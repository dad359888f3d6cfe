// fa_forward_host: forward requests whose tensors live in host memory. The
// pages compute on tensors already in device memory; this is the serving-side
// runtime around that path (declared in include/fa.h).
//
// Each request's Q, K, V are copied into one of three device slots (taken
// from libfa's stream-ordered pool), the fused forward runs on the caller's
// stream, and O and LSE are copied back. Copies in and out run on two
// library-owned streams, so later requests' copies in and earlier requests'
// copies out overlap request i's kernels; events keep each slot from being
// refilled before its last reader is done. In the packed form a request's Q|K|V and O|LSE are one host
// buffer each and move with one copy per direction (fewer, larger copies run
// closer to the host link's rate). Separate tensors are always copied one by
// one: two host buffers that merely sit next to each other may belong to
// different allocations, which one copy may not span.
#include "fa_internal.h"
#include "fa.h"

#include <cmath>
#include <mutex>

namespace fa {
namespace {

// Per-device copy streams, created on first use and kept for the process.
struct CopyStreams {
  std::mutex mu;   // one enqueue at a time per device: the streams are shared
  cudaStream_t in = nullptr, out = nullptr;
};

CopyStreams* copy_streams(int dev) {
  static CopyStreams s[64];
  return (dev >= 0 && dev < 64) ? &s[dev] : nullptr;
}

// Device slots a call cycles through. Measured on GB300 (one head, N = 8192: 6.3
// MB in and 2.1 MB out per request against a 32 us kernel): 42.9 us per request
// with two slots, 39.8 with three, 39.7 with four; with three the host link
// (~210 GB/s for both directions at once at these sizes) is the limit.
constexpr int kSlots = 3;

struct Events {
  cudaEvent_t start = nullptr, in[kSlots] = {}, k[kSlots] = {}, out[kSlots] = {};
  cudaError_t create() {
    cudaError_t e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming);
    for (int b = 0; b < kSlots && e == cudaSuccess; ++b) {
      e = cudaEventCreateWithFlags(&in[b], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&k[b], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&out[b], cudaEventDisableTiming);
    }
    return e;
  }
  // events still pending in a stream are released once they complete
  ~Events() {
    if (start) cudaEventDestroy(start);
    for (int b = 0; b < kSlots; ++b) {
      if (in[b]) cudaEventDestroy(in[b]);
      if (k[b]) cudaEventDestroy(k[b]);
      if (out[b]) cudaEventDestroy(out[b]);
    }
  }
};

// packed: q[i] holds Q|K|V back to back and o[i] holds O|LSE (k, v, lse unused)
int host_requests(int n, const void* const* q, const void* const* k, const void* const* v,
                  void* const* o, float* const* lse, bool packed, int B, int H_q, int H_kv, int N_q,
                  int N_k, int d, int causal, float scale, int dtype, void* stream) {
  if (n < 0 || (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16)) return FA_ERR_INVALID_ARG;
  const Shape s{B, H_q, H_kv, N_q, N_k, d};
  int st = validate_shape(s);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  if (!q || !o || (!packed && (!k || !v))) return FA_ERR_INVALID_ARG;
  const long long rows_q = (long long)B * H_q * N_q;
  const long long rows_k = (long long)B * H_kv * N_k;
  if (rows_q == 0) return FA_OK;   // nothing to compute, nothing to copy
  for (int i = 0; i < n; ++i)
    if (!q[i] || !o[i] || (!packed && rows_k > 0 && (!k[i] || !v[i]))) return FA_ERR_INVALID_ARG;

  const size_t qb = (size_t)rows_q * d * 2, kb = (size_t)rows_k * d * 2;
  const size_t ob = qb, lb = (size_t)rows_q * 4;
  // slot layout Q | K | V | O | LSE: every part starts 16-byte aligned (qb, kb are
  // multiples of 128 bytes for d = 64, 128); a packed request's Q|K|V and O|LSE
  // buffers map onto the slot as one block each
  const size_t slot_bytes = (qb + 2 * kb + ob + lb + 255) / 256 * 256;
  const int n_slots = n < kSlots ? n : kSlots;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaGetLastError());
  CopyStreams* cs = copy_streams(dev);
  if (!cs) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(cs->mu);
  if (!cs->in) {
    cudaError_t e = cudaStreamCreateWithFlags(&cs->in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs->out, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  Events ev;
  cudaError_t e = ev.create();
  if (e != cudaSuccess) return cuda_fail(e);

  const WorkspaceSource& pool = pool_workspace();
  void* ws = nullptr;
  st = pool.acquire(slot_bytes * n_slots, strm, &ws);
  if (st != FA_OK) return st;
  char* base = static_cast<char*>(ws);

  // the copy streams start after everything already on the caller's stream
  // (including the slots' allocation)
  e = cudaEventRecord(ev.start, strm);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->in, ev.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->out, ev.start, 0);
  for (int i = 0; i < n && e == cudaSuccess && st == FA_OK; ++i) {
    const int b = i % n_slots;
    char* dq = base + (size_t)b * slot_bytes;
    char* dk = dq + qb;
    char* dv = dk + kb;
    char* d_o = dv + kb;
    float* dl = reinterpret_cast<float*>(d_o + ob);
    // copy in, once request i - kSlots' kernels have read this slot
    if (i >= n_slots) e = cudaStreamWaitEvent(cs->in, ev.k[b], 0);
    if (e != cudaSuccess) break;
    if (rows_k == 0) {
      e = cudaMemcpyAsync(dq, q[i], qb, cudaMemcpyHostToDevice, cs->in);
    } else if (packed) {
      e = cudaMemcpyAsync(dq, q[i], qb + 2 * kb, cudaMemcpyHostToDevice, cs->in);
    } else {
      e = cudaMemcpyAsync(dq, q[i], qb, cudaMemcpyHostToDevice, cs->in);
      if (e == cudaSuccess) e = cudaMemcpyAsync(dk, k[i], kb, cudaMemcpyHostToDevice, cs->in);
      if (e == cudaSuccess) e = cudaMemcpyAsync(dv, v[i], kb, cudaMemcpyHostToDevice, cs->in);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev.in[b], cs->in);
    // the forward on the caller's stream, once the inputs are in and request
    // i - kSlots' outputs have left the slot
    if (e == cudaSuccess) e = cudaStreamWaitEvent(strm, ev.in[b], 0);
    if (e == cudaSuccess && i >= n_slots) e = cudaStreamWaitEvent(strm, ev.out[b], 0);
    if (e != cudaSuccess) break;
    st = forward_impl(dq, dk, dv, d_o, dl, B, H_q, H_kv, N_q, N_k, d, causal, scale, strm, pool, dtype);
    if (st != FA_OK) break;
    e = cudaEventRecord(ev.k[b], strm);
    // copy out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->out, ev.k[b], 0);
    if (e != cudaSuccess) break;
    float* hl = (!packed && lse) ? lse[i] : nullptr;
    if (packed) {
      e = cudaMemcpyAsync(o[i], d_o, ob + lb, cudaMemcpyDeviceToHost, cs->out);
    } else {
      e = cudaMemcpyAsync(o[i], d_o, ob, cudaMemcpyDeviceToHost, cs->out);
      if (e == cudaSuccess && hl) e = cudaMemcpyAsync(hl, dl, lb, cudaMemcpyDeviceToHost, cs->out);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev.out[b], cs->out);
  }
  // whatever was enqueued, the caller's stream waits for all of it before the
  // slots go back to the pool (a failed record leaves an event that completes at once)
  cudaStreamWaitEvent(strm, ev.start, 0);
  for (int b = 0; b < n_slots; ++b) {
    cudaEventRecord(ev.in[b], cs->in);
    cudaEventRecord(ev.out[b], cs->out);
    cudaStreamWaitEvent(strm, ev.in[b], 0);
    cudaStreamWaitEvent(strm, ev.out[b], 0);
  }
  if (pool.release) pool.release(ws, strm);
  if (st != FA_OK) return st;
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" int fa_forward_host(int n, const void* const* q, const void* const* k, const void* const* v,
                               void* const* o, float* const* lse, int B, int H_q, int H_kv, int N_q,
                               int N_k, int d, int causal, float scale, int dtype, void* stream) {
  return host_requests(n, q, k, v, o, lse, false, B, H_q, H_kv, N_q, N_k, d, causal, scale, dtype,
                       stream);
}

extern "C" int fa_forward_host_packed(int n, const void* const* qkv, void* const* out, int B, int H_q,
                                      int H_kv, int N_q, int N_k, int d, int causal, float scale,
                                      int dtype, void* stream) {
  return host_requests(n, qkv, nullptr, nullptr, out, nullptr, true, B, H_q, H_kv, N_q, N_k, d, causal,
                       scale, dtype, stream);
}
