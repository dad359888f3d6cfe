// C ABI of libfa: argument validation, tensor-map construction, work split
// and launches. Declared in include/fa.h.
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa.h"

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace fa {

thread_local int g_last_cuda_error = 0;

namespace {
__device__ int g_device_status;  // one per device (module-scope device variable)
}  // namespace

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  cudaGetLastError();
  return FA_ERR_CUDA;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

// Shared validation of the fa_forward / fa_naive_forward arguments.
int validate_shape(const Shape& s) {
  if (s.B < 0 || s.N_q < 0 || s.N_k < 0 || s.H_q < 1 || s.H_kv < 1 || s.d < 1)
    return FA_ERR_INVALID_ARG;
  if (s.H_q % s.H_kv != 0) return FA_ERR_INVALID_ARG;
  // indices inside the kernels are 32-bit per (batch*head) row
  const long long rows_q = (long long)s.B * s.H_q * s.N_q;
  const long long rows_k = (long long)s.B * s.H_kv * s.N_k;
  if (rows_q >= (1ll << 31) || rows_k >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (s.d != 64 && s.d != 128 && s.d != 256) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int validate(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const Shape& s, float scale, bool check_device, int in_esz) {
  int st = validate_shape(s);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long rows_q = (long long)s.B * s.H_q * s.N_q;
  const long long rows_k = (long long)s.B * s.H_kv * s.N_k;
  if (rows_q == 0) return FA_OK;  // nothing to write
  if (!q || !o || !aligned16(q) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (lse && !aligned16(lse)) return FA_ERR_INVALID_ARG;
  if (rows_k > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return FA_ERR_INVALID_ARG;
  const size_t qb = (size_t)rows_q * s.d * in_esz, kb = (size_t)rows_k * s.d * in_esz;
  const size_t ob = (size_t)rows_q * s.d * 2;
  const size_t lb = lse ? (size_t)rows_q * 4 : 0;
  // outputs may not overlap any input or each other
  if (overlaps(o, ob, q, qb) || overlaps(o, ob, k, kb) || overlaps(o, ob, v, kb))
    return FA_ERR_INVALID_ARG;
  if (lse && (overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, kb) ||
              overlaps(lse, lb, o, ob)))
    return FA_ERR_INVALID_ARG;
  if (!check_device) return FA_OK;
  const void* ptrs[5] = {q, rows_k > 0 ? k : nullptr, rows_k > 0 ? v : nullptr, o, lse};
  return check_current_device(ptrs, 5);
}

// The kernels and their tensor maps address only the current device's own
// memory: a host pointer, or memory of another GPU reached through unified
// addressing, is rejected before anything is enqueued.
int check_current_device(const void* const* ptrs, int n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  for (int i = 0; i < n; ++i) {
    if (!ptrs[i]) continue;
    cudaPointerAttributes a{};
    e = cudaPointerGetAttributes(&a, ptrs[i]);
    if (e == cudaErrorInvalidValue) {   // not a pointer the runtime knows
      cudaGetLastError();
      return FA_ERR_INVALID_ARG;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    if ((a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) || a.device != dev)
      return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

namespace {
// O = 0, LSE = -inf for every row (no key at all: N_k == 0)
__global__ void fill_empty_kernel(__nv_bfloat16* o, float* lse, long long rows, int d) {
  const long long n = rows * d;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    o[i] = __float2bfloat16_rn(0.f);
    if (lse && i < rows) lse[i] = -INFINITY;
  }
}

}  // namespace

int fill_empty(void* o, float* lse, long long rows, int d, cudaStream_t st) {
  cudaError_t e = launch_kernel(fill_empty_kernel, dim3(256), dim3(256), 0, st,
                                reinterpret_cast<__nv_bfloat16*>(o), lse, rows, d);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

namespace {
// Library-owned stream-ordered pool for split/decode partials, one per device.
// Its release threshold is the maximum, so memory freed at the end of one call
// stays reserved for the next instead of going back to the driver at every
// synchronisation (which would make each call pay a fresh physical allocation).
cudaMemPool_t workspace_pool() {
  static cudaMemPool_t pools[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!pools[dev]) {
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t thr = ~0ull;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    pools[dev] = pool;
  }
  return pools[dev];
}

}  // namespace

// In-cluster merge of split partials: on unless FA_CLUSTER_MERGE=0 (read at every call).
bool cluster_merge_enabled() {
  const char* e = getenv("FA_CLUSTER_MERGE");
  return !(e && e[0] == '0');
}

// Causal block order (block_of in fa_fwd.cu): how many query heads run
// interleaved, longest blocks first. As many KV heads as keep their K and V
// within half of the L2 cache (64 MiB), at most 8, with the query heads that
// share them (measured on 32 heads: 8 beats 16 and 32 at N = 4096 by 2 %, where
// all 32 fit; 8 is also the best at N = 16384). FA_CAUSAL_HEAD_GROUP=n (n >= 1)
// sets it instead: a hook for tests of groups that do not divide the head count.
int causal_head_group(int H_q, int H_kv, int N_k, int d, int n_bh) {
  long long g = 0;
  const char* e = getenv("FA_CAUSAL_HEAD_GROUP");
  if (e && atoi(e) >= 1) {
    g = atoi(e);
  } else {
    const long long kv_bytes = 4ll * N_k * d;   // K and V of one KV head, BF16
    const long long kv_heads = std::min(8ll, std::max(1ll, (64ll << 20) / std::max(1ll, kv_bytes)));
    g = kv_heads * (H_q / H_kv);
  }
  return (int)std::min<long long>(std::max(1ll, g), (long long)n_bh);
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

// Cut the query blocks into CTAs. Whole blocks fill complete waves of the
// GPU; the blocks of an incomplete last wave (all blocks, when there are fewer
// than one wave) have their key range split into s parts when that shortens
// the tail. The parts are combined either by a merge kernel (partials through
// the workspace) or, when every block is split, inside a cluster of the s CTAs
// of each block (distributed shared memory, no workspace). Cost model, in
// key-tile steps of one CTA: a wave costs 2 (set-up and epilogue) + its key
// tiles; the merge kernel costs 3 more (its launch and the partials' round trip
// through L2), the in-cluster merge 0.5. Causal problems with at least a wave
// of blocks are not split: their blocks differ in length and the in-order
// dispatch of longest-first blocks balances them.
FwdPlan plan_forward(long long blocks, int kv_tiles, bool causal, int d, int sms, const int* cluster_cap) {
  FwdPlan pl{};
  pl.u_full = (int)blocks;
  pl.n_tail = 0;
  pl.s_tail = 1;
  pl.units = blocks;
  pl.part_bytes = 0;
  pl.cluster_merge = 0;
  if (blocks <= 0 || kv_tiles <= 1 || sms <= 0) return pl;
  // fewer blocks than SMs: split every block, merging inside clusters of s CTAs
  int cm_s = 1;
  double cm_cost = 2.0 + (double)kv_tiles;   // unsplit: one wave
  if (blocks < sms && cluster_cap) {
    for (int s = 2; s <= 8 && s <= kv_tiles; s *= 2) {   // s divides the block's 256 rows
      if (cluster_cap[s] <= 0) continue;
      const long long waves = (blocks + cluster_cap[s] - 1) / cluster_cap[s];
      const double cost = (double)waves * (2.0 + (double)kv_tiles / s) + 0.5;
      if (cost < cm_cost - 1e-9) {
        cm_cost = cost;
        cm_s = s;
      }
    }
  }
  long long tail = 0;
  if (blocks < sms) {
    tail = blocks;
  } else if (!causal) {
    tail = blocks % sms;
  }
  if (tail == 0) return pl;
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= 16 && s <= kv_tiles; ++s) {
    const long long waves = (tail * s + sms - 1) / sms;
    const double cost = (double)waves * (2.0 + (double)kv_tiles / s) + (s > 1 ? 3.0 : 0.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  if (cm_s > 1 && cm_cost <= best_cost + 1e-9) {
    pl.u_full = 0;
    pl.n_tail = (int)blocks;
    pl.s_tail = cm_s;
    pl.units = blocks * cm_s;
    pl.cluster_merge = 1;
    return pl;
  }
  if (best == 1) return pl;
  pl.u_full = (int)(blocks - tail);
  pl.n_tail = (int)tail;
  pl.s_tail = best;
  pl.units = (blocks - tail) + tail * best;
  pl.part_bytes = (size_t)tail * best * kBlockRows * ((size_t)d * 4 + 8);
  return pl;
}

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t outer, uint64_t row_stride_elems, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {row_stride_elems * 2, row_stride_elems * 2 * rows};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_u8_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                     uint64_t outer, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  // rows of 64 bytes (d = 64) take 64-byte boxes with the 64-byte swizzle
  const bool narrow = inner < 128;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {inner, inner * rows};
  cuuint32_t box[3] = {narrow ? 64u : 128u, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int* device_status_ptr() {
  static int* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

namespace {

int pool_acquire(size_t bytes, cudaStream_t stream, void** ptr) {
  // test hook: FA_TEST_WORKSPACE_FAIL=1 makes every workspace allocation fail
  const char* fail = getenv("FA_TEST_WORKSPACE_FAIL");
  if (fail && fail[0] == '1') return FA_ERR_NO_MEMORY;
  cudaMemPool_t pool = workspace_pool();
  if (!pool) return cuda_fail(cudaGetLastError());
  cudaError_t e = cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
  if (e != cudaSuccess) {
    g_last_cuda_error = (int)e;
    return FA_ERR_NO_MEMORY;
  }
  return FA_OK;
}

void pool_release(void* ptr, cudaStream_t stream) { cudaFreeAsync(ptr, stream); }

}  // namespace

const WorkspaceSource& pool_workspace() {
  static const WorkspaceSource src{pool_acquire, pool_release};
  return src;
}

// The plan fa_forward uses for a prefill request on the current device.
FwdPlan prefill_plan(int B, int H_q, int N_q, int N_k, int d, int causal) {
  const int n_qb = (N_q + kBlockRows - 1) / kBlockRows;
  const int n_kv = (N_k + kTileN - 1) / kTileN;
  const long long blocks = (long long)B * H_q * n_qb;
  // causal blocks see on average about half the key tiles
  const int kv_eff = causal ? (n_kv + 1) / 2 : n_kv;
  const int sms = num_sms();
  int cap[9] = {0};
  const bool cm_ok = cluster_merge_enabled() && blocks < sms;
  if (cm_ok)
    for (int s2 = 2; s2 <= 8; s2 *= 2) cap[s2] = fwd_cluster_capacity(d, s2);
  return plan_forward(blocks, kv_eff, causal != 0, d, sms, cm_ok ? cap : nullptr);
}

int forward_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
                 int H_kv, int N_q, int N_k, int d, int causal, float scale, cudaStream_t strm,
                 const WorkspaceSource& wsrc, int elem, PairedLaunch paired, const float* descale) {
  if (elem != 0 && elem != 1 && elem != 2) return FA_ERR_INVALID_ARG;
  const bool fp8 = elem == 2;
  float qk_factor = 1.f, o_scale = 1.f;
  if (fp8) {
    if (!descale) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
      if (!std::isfinite(descale[i]) || !(descale[i] > 0.f)) return FA_ERR_INVALID_ARG;
    qk_factor = descale[0] * descale[1];
    o_scale = descale[2];
    if (!std::isfinite(scale * qk_factor)) return FA_ERR_INVALID_ARG;
  }
  const Shape s{B, H_q, H_kv, N_q, N_k, d};
  int st = validate_shape(s);
  if (st != FA_OK) return st;
  if (fp8 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  st = validate(q, k, v, o, lse, s, scale, true, fp8 ? 1 : 2);
  if (st != FA_OK) return st;
  if ((long long)B * H_q * N_q == 0) return FA_OK;
  if (N_k == 0 || B * H_kv == 0) return fill_empty(o, lse, (long long)B * H_q * N_q, d, strm);

  int* status = device_status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());
  const int G = H_q / H_kv;
  CUtensorMap tk, tv;
  if (fp8 ? (!make_tmap_u8_3d(&tk, k, d, N_k, (uint64_t)B * H_kv, 128) ||
             !make_tmap_u8_3d(&tv, v, d, N_k, (uint64_t)B * H_kv, 128))
          : (!make_tmap_bf16_3d(&tk, k, d, N_k, (uint64_t)B * H_kv, d, 128) ||
             !make_tmap_bf16_3d(&tv, v, d, N_k, (uint64_t)B * H_kv, d, 128)))
    return cuda_fail(cudaErrorInvalidValue);

  if (d == 256) {
    // one 128-row query tile per CTA; every query row takes this kernel
    D256Params p{};
    p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q; p.N_k = N_k;
    p.causal = causal ? 1 : 0;
    p.kv_off = N_k - N_q;
    p.n_qt = (N_q + 127) / 128;
    p.n_kv_tiles = (N_k + 127) / 128;
    p.elem = elem;
    p.hgroup = causal ? causal_head_group(H_q, H_kv, N_k, d, B * H_q) : 1;
    p.c = scale * 1.4426950408889634f;
    p.lse = lse;
    p.status = status;
    const long long units = (long long)B * H_q * p.n_qt;
    if (units >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    CUtensorMap tq, to;
    if (!make_tmap_bf16_3d(&tq, q, d, N_q, (uint64_t)B * H_q, d, 128) ||
        !make_tmap_bf16_3d(&to, o, d, N_q, (uint64_t)B * H_q, d, 128))
      return cuda_fail(cudaErrorInvalidValue);
    cudaError_t e = launch_fwd_tile(d, tq, tk, tv, to, p, (int)units, strm);
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
  }

  // (FP8 inputs always take the prefill kernel, which handles any number of rows)
  if (!fp8 && (long long)G * N_q <= kDecodeMaxRows) {
    // decode / few queries: every query row of a KV head fits one m16 MMA
    DecParams p{};
    p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q; p.N_k = N_k;
    p.G = G; p.R = G * N_q;
    p.causal = causal ? 1 : 0;
    p.kv_off = N_k - N_q;
    p.n_chunks = (N_k + 127) / 128;
    const DecPlan dp = decode_plan((long long)B * H_kv, p.n_chunks, d, num_sms(), cluster_merge_enabled());
    p.cpc = dp.cpc;
    p.n_parts = dp.n_parts;
    p.cm = dp.cm;
    p.c = scale * 1.4426950408889634f;
    p.q = static_cast<const uint16_t*>(q);
    p.elem = elem;
    p.o = o;
    p.lse = lse;
    p.status = status;
    if ((long long)B * H_kv * p.n_parts >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    const size_t bytes = p.cm ? 0 : decode_part_bytes(B, H_kv, p.R, p.n_parts, d);
    void* ws = nullptr;
    if (bytes > 0) {
      st = wsrc.acquire(bytes, strm, &ws);
      if (st != FA_OK) return st;
    }
    p.part_o = static_cast<float*>(ws);
    p.part_ml = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) +
                                              (size_t)B * H_kv * p.n_parts * p.R * d * 4)
                   : nullptr;
    cudaError_t e = launch_decode(d, tk, tv, p, strm);
    if (ws && wsrc.release) wsrc.release(ws, strm);
    return e == cudaSuccess ? FA_OK : cuda_fail(e);
  }

  FwdParams p{};
  p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q; p.N_k = N_k;
  p.causal = causal ? 1 : 0;
  p.kv_off = N_k - N_q;
  p.n_qb = (N_q + kBlockRows - 1) / kBlockRows;
  p.n_kv_tiles = (N_k + kTileN - 1) / kTileN;
  p.c = scale * qk_factor * 1.4426950408889634f;
  p.o_scale = o_scale;
  p.o = o;
  p.lse = lse;
  p.status = status;
  const FwdPlan pl = prefill_plan(B, H_q, N_q, N_k, d, causal);
  if (pl.units >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  p.u_full = pl.u_full;
  p.n_tail = pl.n_tail;
  p.s_tail = pl.s_tail;
  p.n_units = (int)pl.units;
  p.cm = pl.cluster_merge;
  // (the paired-load variant is built for BF16 only)
  const bool multicast = paired && pl.n_tail == 0 && pl.units >= 2 && elem == 0;
  p.elem = elem;
  p.n_bh = B * H_q;
  // the multicast variant pairs adjacent blocks of one head: head-major there
  p.hgroup = (causal && !multicast) ? causal_head_group(H_q, H_kv, N_k, d, B * H_q) : 1;

  FwdMaps maps{};
  maps.k = tk;
  maps.v = tv;
  // O boxes: a 128-row query tile, or the 256 / s rows one CTA of a cluster finishes
  const uint32_t o_box_rows = pl.cluster_merge ? (uint32_t)(kBlockRows / pl.s_tail) : 128u;
  if (!(fp8 ? make_tmap_u8_3d(&maps.q, q, d, N_q, (uint64_t)B * H_q, 128)
            : make_tmap_bf16_3d(&maps.q, q, d, N_q, (uint64_t)B * H_q, d, 128)) ||
      !make_tmap_bf16_3d(&maps.o, o, d, N_q, (uint64_t)B * H_q, d, o_box_rows))
    return cuda_fail(cudaErrorInvalidValue);
  if (multicast) {
    // each CTA of a pair fetches half the rows of every K/V tile
    if (!make_tmap_bf16_3d(&maps.k, k, d, N_k, (uint64_t)B * H_kv, d, 64) ||
        !make_tmap_bf16_3d(&maps.v, v, d, N_k, (uint64_t)B * H_kv, d, 64))
      return cuda_fail(cudaErrorInvalidValue);
  }
  void* ws = nullptr;
  if (pl.part_bytes > 0) {
    st = wsrc.acquire(pl.part_bytes, strm, &ws);
    if (st != FA_OK) return st;
    const uint64_t part_rows = (uint64_t)pl.n_tail * pl.s_tail * kBlockRows;
    p.part_o = static_cast<float*>(ws);
    p.part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + part_rows * d * 4);
    if (!make_tmap_f32_2d(&maps.part, p.part_o, d, part_rows)) {
      if (wsrc.release) wsrc.release(ws, strm);
      return cuda_fail(cudaErrorInvalidValue);
    }
  }
  cudaError_t e = multicast ? paired(d, maps, p, (int)pl.units, strm)
                            : launch_fwd(d, maps, p, (int)pl.units, strm);
  if (ws && wsrc.release) wsrc.release(ws, strm);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return (0 << 16) | 1; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_NO_MEMORY: return "out of memory / workspace too small";
    case FA_ERR_TIMEOUT: return "kernel wait timed out";
    case FA_ERR_TOO_LARGE: return "request needs more scratch than the static scratch array holds";
    case FA_ERR_BOUNDS: return "a bounds check of the FA_DEBUG build failed";
    default: return "unknown status";
  }
}

int fa_get_last_cuda_error(void) { return g_last_cuda_error; }

int fa_device_status(int reset) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  int* p = device_status_ptr();
  if (!p) return cuda_fail(cudaGetLastError());
  int h = 0;
  e = cudaMemcpy(&h, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (reset && h != 0) {
    int zero = 0;
    e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return h == 0 ? FA_OK : (h == FA_DEV_BOUNDS ? FA_ERR_BOUNDS : FA_ERR_TIMEOUT);
}

int fa_forward_plan(int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal, long long* ctas,
                    int* launches, size_t* workspace_bytes) {
  const fa::Shape s{B, H_q, H_kv, N_q, N_k, d};
  int st = fa::validate_shape(s);
  if (st != FA_OK) return st;
  long long c = 0;
  int n = 0;
  size_t ws = 0;
  if ((long long)B * H_q * N_q == 0) {
    // nothing to compute
  } else if (N_k == 0) {
    c = 256;   // O = 0, LSE = -inf fill
    n = 1;
  } else if (d == 256) {
    c = (long long)B * H_q * ((N_q + 127) / 128);   // one CTA per 128-row query tile
    n = 1;
  } else if ((long long)(H_q / H_kv) * N_q <= fa::kDecodeMaxRows) {
    const int chunks = (N_k + 127) / 128;
    const fa::DecPlan dp = fa::decode_plan((long long)B * H_kv, chunks, d, fa::num_sms(),
                                           fa::cluster_merge_enabled());
    c = (long long)B * H_kv * dp.n_parts;
    n = dp.cm ? 1 : 2;
    ws = dp.cm ? 0 : fa::decode_part_bytes(B, H_kv, (H_q / H_kv) * N_q, dp.n_parts, d);
  } else {
    const fa::FwdPlan pl = fa::prefill_plan(B, H_q, N_q, N_k, d, causal);
    c = pl.units;
    n = pl.part_bytes > 0 ? 2 : 1;
    ws = pl.part_bytes;
  }
  if (ctas) *ctas = c;
  if (launches) *launches = n;
  if (workspace_bytes) *workspace_bytes = ws;
  return FA_OK;
}

size_t fa_naive_workspace_bytes(int B, int H_q, int N_q, int N_k) {
  if (B < 0 || H_q < 1 || N_q < 0 || N_k < 0) return 0;
  const size_t ld = ((size_t)N_k + 7) / 8 * 8;
  return (size_t)B * H_q * N_q * ld * 2;
}

int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
               int H_kv, int N_q, int N_k, int d, int causal, float scale, void* stream) {
  return forward_impl(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, causal, scale,
                      static_cast<cudaStream_t>(stream), pool_workspace());
}

int fa_forward_fp16(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H_q, int H_kv, int N_q, int N_k, int d, int causal, float scale, void* stream) {
  return forward_impl(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, causal, scale,
                      static_cast<cudaStream_t>(stream), pool_workspace(), 1);
}

int fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
                   int H_kv, int N_q, int N_k, int d, int causal, float scale, float descale_q,
                   float descale_k, float descale_v, void* stream) {
  const float descale[3] = {descale_q, descale_k, descale_v};
  return forward_impl(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, causal, scale,
                      static_cast<cudaStream_t>(stream), pool_workspace(), 2, nullptr, descale);
}

int fa_naive_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H_q, int H_kv, int N_q, int N_k, int d, int causal, float scale,
                     void* workspace, size_t workspace_bytes, void* stream) {
  const Shape s{B, H_q, H_kv, N_q, N_k, d};
  int st = validate(q, k, v, o, lse, s, scale, false);
  if (st != FA_OK) return st;
  if (d == 256) return FA_ERR_UNSUPPORTED;   // the unfused baseline covers d = 64 and 128
  if ((long long)B * H_q * N_q == 0) return FA_OK;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  if (N_k == 0) {
    const void* outs[2] = {o, lse};
    st = check_current_device(outs, 2);
    return st != FA_OK ? st : fill_empty(o, lse, (long long)B * H_q * N_q, d, strm);
  }
  const size_t need = fa_naive_workspace_bytes(B, H_q, N_q, N_k);
  if (!workspace || workspace_bytes < need) return FA_ERR_NO_MEMORY;
  if (!aligned16(workspace)) return FA_ERR_INVALID_ARG;
  const size_t qb = (size_t)B * H_q * N_q * d * 2, kb = (size_t)B * H_kv * N_k * d * 2;
  if (overlaps(workspace, need, q, qb) || overlaps(workspace, need, k, kb) ||
      overlaps(workspace, need, v, kb) || overlaps(workspace, need, o, qb) ||
      overlaps(workspace, need, lse, lse ? (size_t)B * H_q * N_q * 4 : 0))
    return FA_ERR_INVALID_ARG;
  const void* ptrs[6] = {q, k, v, o, lse, workspace};
  st = check_current_device(ptrs, 6);
  if (st != FA_OK) return st;
  int* status = device_status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());

  const int ld = (N_k + 7) / 8 * 8;
  const int G = H_q / H_kv;
  CUtensorMap tq, tk, ts, tv;
  if (!make_tmap_bf16_3d(&tq, q, d, N_q, (uint64_t)B * H_q, d, 128) ||
      !make_tmap_bf16_3d(&tk, k, d, N_k, (uint64_t)B * H_kv, d, 128) ||
      !make_tmap_bf16_3d(&ts, workspace, ld, N_q, (uint64_t)B * H_q, ld, 128) ||
      !make_tmap_bf16_3d(&tv, v, d, N_k, (uint64_t)B * H_kv, d, 64))
    return cuda_fail(cudaErrorInvalidValue);

  // kernel 1: S = scale * Q K^T  ->  workspace (BF16, rows padded to ld)
  GemmParams g1{};
  g1.M = N_q; g1.N = N_k; g1.K = d; g1.batches = B * H_q;
  g1.heads = H_q; g1.heads_kv = H_kv; g1.group = G;
  g1.alpha = scale; g1.c = workspace; g1.ldc = ld;
  cudaError_t e = launch_gemm(false, 128, tq, tk, g1, status, strm);
  if (e != cudaSuccess) return cuda_fail(e);
  // kernel 2: P = softmax(S) in place, LSE
  SoftmaxParams sp{};
  sp.s = workspace; sp.lse = lse; sp.rows = B * H_q * N_q; sp.n_q = N_q; sp.n_k = N_k; sp.ld = ld;
  sp.causal = causal ? 1 : 0; sp.kv_off = N_k - N_q;
  e = launch_row_softmax(sp, strm);
  if (e != cudaSuccess) return cuda_fail(e);
  // kernel 3: O = P V
  GemmParams g3{};
  g3.M = N_q; g3.N = d; g3.K = ld; g3.batches = B * H_q;
  g3.heads = H_q; g3.heads_kv = H_kv; g3.group = G;
  g3.alpha = 1.f; g3.c = o; g3.ldc = d;
  e = launch_gemm(true, d, ts, tv, g3, status, strm);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // extern "C"
