// Internal launch interface between the C ABI (fa_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <utility>

namespace fa {

// ---- fused prefill forward ------------------------------------------------------
constexpr int kTileM = 128;          // query rows per tile (one tcgen05 M=128 MMA)
constexpr int kTileN = 128;          // keys per K/V tile
constexpr int kBlockRows = 2 * kTileM;  // query rows per CTA work unit (two ping-pong tiles)

struct FwdParams {
  int B, H_q, H_kv, N_q, N_k;
  int causal;
  int kv_off;       // N_k - N_q: query i sees key j iff j <= i + kv_off (causal)
  int n_qb;         // query blocks of kBlockRows rows per (b, h)
  int n_bh;         // B * H_q
  int hgroup;       // causal block order: heads per group (>= 1; 1 = head-major)
  int n_kv_tiles;   // ceil(N_k / kTileN)
  int u_full;       // units [0, u_full) are whole query blocks (query blocks 0 .. u_full-1)
  int n_tail;       // query blocks u_full .. u_full+n_tail-1 are split ...
  int s_tail;       // ... into s_tail key ranges each (units u_full + t*s_tail + s)
  int n_units;      // work units (the grid may hold one more, idle, CTA to complete a cluster)
  int cm;           // 1: every block is split and its s_tail CTAs (one cluster) merge in-kernel
  int elem;         // element type of Q, K, V: 0 = BF16, 1 = FP16 (O the same), 2 = FP8 E4M3 (O BF16)
  float c;          // scale * log2(e) (FP8: times the Q and K factors)
  float o_scale;    // factor on the normalised output: 1, or the V factor of FP8 inputs
  void* o;          // 16-bit [B][H_q][N_q][d]
  float* lse;       // fp32 [B][H_q][N_q] or nullptr
  float* part_o;    // fp32 [n_tail*s_tail][kBlockRows][d]        (n_tail > 0)
  float* part_ml;   // fp32 [n_tail*s_tail][kBlockRows][2] (m, l)  (n_tail > 0)
  int* status;      // device status word
};

// How the query blocks of one call are cut into CTAs (see FwdParams).
struct FwdPlan {
  int u_full, n_tail, s_tail;
  long long units;      // CTAs of the fused kernel
  size_t part_bytes;    // workspace for the split partials (0 without a merge kernel)
  int cluster_merge;    // 1: all blocks split, partials merged inside each cluster of s_tail CTAs
};
// cluster_cap[s] (s = 2..8): clusters of s CTAs the device holds at once, 0 if
// unusable; nullptr disables the in-cluster merge.
FwdPlan plan_forward(long long blocks, int kv_tiles, bool causal, int d, int sms, const int* cluster_cap);
// Clusters of s fused-kernel CTAs (head dim d) resident at once on the current device.
int fwd_cluster_capacity(int d, int s);

// Shared-memory bytes the fused kernel needs for head dim d (64 or 128).
size_t fwd_smem_bytes(int d);

// Tensor maps of one forward call: Q, K, V, O (BF16, [B*H][N][d], 64-column
// boxes, 128-byte swizzle) and the FP32 split partials ([rows][d], 32-column boxes).
struct FwdMaps {
  CUtensorMap q, k, v, o, part;
};
// Launch the fused kernel over `units` CTAs, then (if p.n_tail > 0) the merge
// kernel as its programmatic dependent on the same stream.
cudaError_t launch_fwd(int d, const FwdMaps& m, const FwdParams& p, int units, cudaStream_t stream);
// A launcher of the paired-load variant (CTAs in clusters of two sharing K/V
// tile loads by cluster multicast; plans without split tails; tk / tv built
// with 64-row boxes). Only the single-GPU library has one; libfa passes none.
typedef cudaError_t (*PairedLaunch)(int d, const FwdMaps& m, const FwdParams& p, int units,
                                    cudaStream_t stream);

// ---- fused forward for head dimension 256 (one 128-row query tile per CTA) -----------
struct D256Params {
  int B, H_q, H_kv, N_q, N_k;
  int causal;
  int kv_off;       // N_k - N_q
  int n_qt;         // ceil(N_q / 128) query tiles per (b, h)
  int n_kv_tiles;   // ceil(N_k / 128)
  int elem;         // 0 = BF16, 1 = FP16
  int hgroup;       // causal tile order: heads per group (>= 1)
  float c;          // scale * log2(e)
  float* lse;       // fp32 [B][H_q][N_q] or nullptr
  int* status;
};
// One CTA per query tile (B * H_q * n_qt CTAs), as a programmatic dependent
// launch; head dimension d = 128 or 256.
cudaError_t launch_fwd_tile(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const D256Params& p, int units, cudaStream_t stream);

// ---- decode / few queries per KV head -------------------------------------------------
constexpr int kDecodeMaxRows = 16;   // R = G * N_q rows per KV head must fit one m16 MMA

struct DecParams {
  int B, H_q, H_kv, N_q, N_k;
  int G, R;          // G = H_q / H_kv; R = G * N_q query rows per (batch, KV head)
  int causal, kv_off;
  int n_chunks;      // ceil(N_k / 128)
  int cpc;           // chunks per CTA (a run of consecutive chunks)
  int n_parts;       // ceil(n_chunks / cpc): CTAs, and partials, per (batch, KV head)
  int cm;            // 1: the n_parts CTAs of a KV head form a cluster and merge in-kernel
  int elem;          // element type of Q, K, V, O: 0 = BF16, 1 = FP16 (host-side dispatch)
  float c;           // scale * log2(e)
  const uint16_t* q;  // [B][H_q][N_q][d], 16-bit elements (BF16 or FP16)
  void* o;
  float* lse;
  float* part_o;     // fp32 [B*H_kv][n_parts][R][d]
  float* part_ml;    // fp32 [B*H_kv][n_parts][R][2]
  int* status;
  // paged K/V (paged = 1): K and V are [num_pages][H_kv][128][d]; sequence b's
  // chunk c is page block_table[b * max_pages + c]; its key count is
  // seqlens[b] (clamped to [0, max_pages * 128]); N_k and n_chunks are then
  // the maxima (max_pages * 128, max_pages)
  int paged;
  int max_pages;
  const int* block_table;
  const int* seqlens;
};
size_t decode_part_bytes(int B, int H_kv, int R, int n_parts, int d);
// How the decode kernel cuts `heads` = B * H_kv KV heads of n_chunks chunks each.
struct DecPlan {
  int cpc, n_parts, cm;   // chunks per CTA, CTAs per KV head, in-cluster merge
};
DecPlan decode_plan(long long heads, int n_chunks, int d, int sms, bool cluster_merge);
// Launch the decode kernel, then the chunk merge as its programmatic dependent.
cudaError_t launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p,
                          cudaStream_t stream);

// ---- unfused baseline -------------------------------------------------------------
struct GemmParams {
  int M, N, K;          // per batch: C[M][N] = alpha * A[M][K] * B
  int batches;          // grid z
  int a_heads_per_b;    // A batch index = z
  int group;            // B batch index = (z / heads) * heads_kv + (z % heads) / group
  int heads, heads_kv;
  float alpha;
  void* c;              // bf16 output, row stride ldc elements, batch stride M*ldc
  int ldc;
};
cudaError_t launch_gemm(bool b_mn_major, int bn, const CUtensorMap& ta, const CUtensorMap& tb,
                        const GemmParams& p, int* status, cudaStream_t stream);
size_t gemm_smem_bytes(int bn);

struct SoftmaxParams {
  void* s;          // bf16 [rows][ld]: scores in, probabilities out (in place)
  float* lse;       // fp32 [rows] or nullptr
  int rows, n_q, n_k, ld;
  int causal, kv_off;
};
cudaError_t launch_row_softmax(const SoftmaxParams& p, cudaStream_t stream);

// ---- host helpers -------------------------------------------------------------------
struct Shape {
  int B, H_q, H_kv, N_q, N_k, d;
};
// Shape checks alone (sizes, H_q % H_kv, 32-bit row counts, d): fa_status code.
int validate_shape(const Shape& s);
// Argument checks shared by the forward entry points (fa_status code; FA_OK when valid);
// check_device: also require every pointer to be memory of the current device.
// in_esz: bytes per element of q, k, v (2, or 1 for FP8; o is always 16-bit).
int validate(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const Shape& s, float scale, bool check_device = true, int in_esz = 2);
// O = 0 and LSE = -inf for `rows` rows (every row sees no key).
int fill_empty(void* o, float* lse, long long rows, int d, cudaStream_t st);
// Record a CUDA error for fa_get_last_cuda_error and return FA_ERR_CUDA; the
// runtime's per-thread last error is cleared (the code now carries it).
int cuda_fail(cudaError_t e);

// Launch whose return value is that launch's own status (cudaLaunchKernelEx),
// not the thread's last error, which an earlier unrelated call may have left set.
template <typename... K, typename... A>
inline cudaError_t launch_kernel(void (*kernel)(K...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, A&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}
int num_sms();
bool cluster_merge_enabled();   // in-cluster merge of partials unless FA_CLUSTER_MERGE=0
extern thread_local int g_last_cuda_error;

// 3-D BF16 tensor map over [outer][rows][inner] with a {64, 128, 1} box, 128-byte swizzle.
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t outer, uint64_t row_stride_elems, uint32_t box_rows);
// 3-D 8-bit tensor map over [outer][rows][inner] with a {128, box_rows, 1} box and
// 128-byte swizzle ({64, box_rows, 1} and 64-byte swizzle when inner < 128).
bool make_tmap_u8_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                     uint64_t outer, uint32_t box_rows);

// 2-D FP32 tensor map over [rows][inner] with a {32, 128} box, 128-byte swizzle.
bool make_tmap_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows);

int* device_status_ptr();   // address of the current device's status word (nullptr on error)

// Where a forward call gets its split / decode partials from. acquire returns
// FA_OK with *ptr set, or an fa_status code (nothing enqueued); release is
// called (stream-ordered) after the kernels that use the memory.
struct WorkspaceSource {
  int (*acquire)(size_t bytes, cudaStream_t stream, void** ptr);
  void (*release)(void* ptr, cudaStream_t stream);
};
const WorkspaceSource& pool_workspace();   // library-owned stream-ordered pool
// The whole fused forward (validation, decode or prefill plan, launches);
// elem: 0 = BF16, 1 = FP16 tensors.
// paired: the paired-load launcher, used for BF16 plans without split tails
// (nullptr: the plain kernel always).
// elem 2 (FP8 E4M3): descale = the Q, K, V factors (else ignored).
int forward_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
                 int H_kv, int N_q, int N_k, int d, int causal, float scale, cudaStream_t stream,
                 const WorkspaceSource& ws, int elem = 0, PairedLaunch paired = nullptr,
                 const float* descale = nullptr);
// Every non-null pointer is device memory of the current device (FA_OK),
// else FA_ERR_INVALID_ARG; FA_ERR_CUDA when the device cannot be queried.
int check_current_device(const void* const* ptrs, int n);

}  // namespace fa
