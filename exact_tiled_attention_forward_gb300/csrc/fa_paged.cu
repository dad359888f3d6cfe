// fa_decode_paged: decode attention (a few query rows per KV head) over a K/V
// cache kept in fixed pages of 128 keys, each sequence with its own length and
// its own list of pages.
//
// The pages describe decode as one query against many cached keys, bound by
// reading K and V once per KV head ("FlashAttention HBM bytes, one head, 8K",
// "What interviewers probe next"); they say nothing about how a cache is laid
// out. This entry point serves callers whose caches grow page by page: the
// attention computed is exactly fa_forward's over each sequence's keys in
// order, with the same kernel (fa_decode_kernel) — only the address of each
// 128-key chunk comes from the block table, and the key count from seqlens.
#include "fa_internal.h"
#include "fa.h"

#include <cmath>
#include <cstdint>

namespace fa {
namespace {

constexpr int kPageKeys = 128;   // keys per page = the decode kernel's chunk

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

int paged_impl(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
               const int* seqlens, void* o, float* lse, int B, int H_q, int H_kv, int N_q, int num_pages,
               int max_pages, int d, int causal, float scale, int elem, cudaStream_t strm) {
  if (elem != FA_DTYPE_BF16 && elem != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  if (B < 0 || N_q < 0 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || num_pages < 1 || max_pages < 1)
    return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const int G = H_q / H_kv;
  if ((long long)G * N_q > kDecodeMaxRows) return FA_ERR_UNSUPPORTED;   // the decode kernel's rows
  const long long rows_q = (long long)B * H_q * N_q;
  if (rows_q >= (1ll << 31) || (long long)num_pages * H_kv >= (1ll << 31) ||
      (long long)max_pages * kPageKeys >= (1ll << 31) || (long long)B * max_pages >= (1ll << 31))
    return FA_ERR_INVALID_ARG;
  if (rows_q == 0) return FA_OK;   // nothing to write
  if (!q || !o || !k_cache || !v_cache || !block_table || !seqlens) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      (lse && !aligned(lse, 16)) || !aligned(block_table, 4) || !aligned(seqlens, 4))
    return FA_ERR_INVALID_ARG;
  const size_t qb = (size_t)rows_q * d * 2;
  const size_t cb = (size_t)num_pages * H_kv * kPageKeys * d * 2;
  const size_t tb = (size_t)B * max_pages * 4, sl = (size_t)B * 4, lb = lse ? (size_t)rows_q * 4 : 0;
  const void* ins[5] = {q, k_cache, v_cache, block_table, seqlens};
  const size_t in_bytes[5] = {qb, cb, cb, tb, sl};
  for (int i = 0; i < 5; ++i)
    if (overlap(o, qb, ins[i], in_bytes[i]) || (lse && overlap(lse, lb, ins[i], in_bytes[i])))
      return FA_ERR_INVALID_ARG;
  if (lse && overlap(lse, lb, o, qb)) return FA_ERR_INVALID_ARG;
  {
    const void* all[7] = {q, k_cache, v_cache, block_table, seqlens, o, lse};
    const int dst = check_current_device(all, 7);
    if (dst != FA_OK) return dst;
  }

  int* status = device_status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());
  // K and V as 3-D tensors (d, 128 keys, num_pages * H_kv): one slab per
  // (page, KV head), one TMA box row per key
  CUtensorMap tk, tv;
  if (!make_tmap_bf16_3d(&tk, k_cache, d, kPageKeys, (uint64_t)num_pages * H_kv, d, kPageKeys) ||
      !make_tmap_bf16_3d(&tv, v_cache, d, kPageKeys, (uint64_t)num_pages * H_kv, d, kPageKeys))
    return cuda_fail(cudaErrorInvalidValue);

  DecParams p{};
  p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q;
  p.N_k = max_pages * kPageKeys;   // the longest a sequence can be; each has its own length
  p.G = G; p.R = G * N_q;
  p.causal = causal ? 1 : 0;
  p.kv_off = p.N_k - N_q;
  p.n_chunks = max_pages;
  const DecPlan dp = decode_plan((long long)B * H_kv, max_pages, d, num_sms(), cluster_merge_enabled());
  p.cpc = dp.cpc;
  p.n_parts = dp.n_parts;
  p.cm = dp.cm;
  p.c = scale * 1.4426950408889634f;
  p.q = static_cast<const uint16_t*>(q);
  p.elem = elem;
  p.o = o;
  p.lse = lse;
  p.status = status;
  p.paged = 1;
  p.max_pages = max_pages;
  p.block_table = block_table;
  p.seqlens = seqlens;
  if ((long long)B * H_kv * p.n_parts >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  const size_t bytes = p.cm ? 0 : decode_part_bytes(B, H_kv, p.R, p.n_parts, d);
  const WorkspaceSource& pool = pool_workspace();
  void* ws = nullptr;
  if (bytes > 0) {
    const int st = pool.acquire(bytes, strm, &ws);
    if (st != FA_OK) return st;
  }
  p.part_o = static_cast<float*>(ws);
  p.part_ml = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + (size_t)B * H_kv * p.n_parts * p.R * d * 4)
                 : nullptr;
  cudaError_t e = launch_decode(d, tk, tv, p, strm);
  if (ws && pool.release) pool.release(ws, strm);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // namespace
}  // namespace fa

extern "C" int fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                               const int* seqlens_k, void* o, float* lse, int B, int H_q, int H_kv, int N_q,
                               int num_pages, int max_pages, int d, int causal, float scale, int dtype,
                               void* stream) {
  return fa::paged_impl(q, k_cache, v_cache, block_table, seqlens_k, o, lse, B, H_q, H_kv, N_q, num_pages,
                        max_pages, d, causal, scale, dtype, static_cast<cudaStream_t>(stream));
}
