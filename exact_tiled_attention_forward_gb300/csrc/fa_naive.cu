// Unfused attention, kept as the measured traffic baseline
// ("FlashAttention HBM bytes, one head, 8K", "A strong answer": the unfused
// kernel writes S = QK^T, reads it for the softmax, writes P and reads P for
// PV; "Why is standard attention memory-bound...", Step 1: three kernels).
//
//   kernel 1  S = scale * Q K^T           tcgen05 GEMM, BF16 S to device memory
//   kernel 2  P = softmax_row(S), LSE     in place, BF16, one CTA per row
//   kernel 3  O = P V                     tcgen05 GEMM (V is the MN-major operand)
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {

namespace {

constexpr int kGemmThreads = 128;
constexpr int kGemmStages = 4;

template <int BN, bool B_MN>
struct GemmCfg {
  static constexpr int kABytes = 128 * 64 * 2;               // A box: 128 rows x 64 K
  static constexpr int kBBytes = BN * 64 * 2;                // B: BN x 64 K (either major)
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kOffBar = kGemmStages * kStageBytes;
  static constexpr int kSmemBytes = kOffBar + (2 * kGemmStages + 2) * 8 + 16 + 1024;
  static constexpr uint32_t kTmemCols = BN < 32 ? 32 : BN;
};

// One 128 x BN output tile per CTA. Warp 0 lane 0 loads, warp 1 lane 0 issues
// the MMAs, all four warps run the epilogue (warp w owns TMEM lanes 32w..).
template <int BN, bool B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmParams p, int* status) {
  using C = GemmCfg<BN, B_MN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8 * i; };
  const int kFull = 0, kEmpty = kGemmStages, kDone = 2 * kGemmStages, kDrain = 2 * kGemmStages + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + (2 * kGemmStages + 2) * 8);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * 128;
  const int z = blockIdx.z;
  const int zb = (z / p.heads) * p.heads_kv + (z % p.heads) / p.group;
  const int nk = (p.K + 63) / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(bar(kFull + s), 1);
      mbar_init(bar(kEmpty + s), 1);
    }
    mbar_init(bar(kDone), 1);
    mbar_init(bar(kDrain), 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    int issued = 0;
    for (int kt = 0; kt < nk; ++kt) {
      const int st = kt % kGemmStages;
      const uint32_t ph = (uint32_t)(kt / kGemmStages) & 1u;
      if (!mbar_wait(bar(kEmpty + st), ph ^ 1u, s_abort, status)) break;
      mbar_arrive_expect_tx(bar(kFull + st), C::kStageBytes);
      const uint32_t a_dst = sb + st * C::kStageBytes;
      const uint32_t b_dst = a_dst + C::kABytes;
      tma_load_3d(a_dst, &tmA, bar(kFull + st), kt * 64, m0, z);
      if (B_MN) {
        // B stored [K][N] (N contiguous): boxes of 64 N-columns x 64 K-rows
#pragma unroll
        for (int bx = 0; bx < BN / 64; ++bx)
          tma_load_3d(b_dst + bx * 64 * 128, &tmB, bar(kFull + st), n0 + bx * 64, kt * 64, zb);
      } else {
        tma_load_3d(b_dst, &tmB, bar(kFull + st), kt * 64, n0, zb);
      }
      ++issued;
    }
    volatile int never = 0;
    for (int st = 0; st < kGemmStages; ++st) {
      const int n_st = issued > st ? (issued - st + kGemmStages - 1) / kGemmStages : 0;
      if (n_st > 0) mbar_wait(bar(kFull + st), (uint32_t)(n_st - 1) & 1u, &never, status);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, BN, B_MN);
    bool ok = true;
    for (int kt = 0; kt < nk && ok; ++kt) {
      const int st = kt % kGemmStages;
      const uint32_t ph = (uint32_t)(kt / kGemmStages) & 1u;
      if (!(ok = mbar_wait(bar(kFull + st), ph, s_abort, status))) break;
      tc_fence_after();
      const uint32_t a_s = sb + st * C::kStageBytes;
      const uint32_t b_s = a_s + C::kABytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = smem_desc_sw128(a_s + kk * 32, 16, 1024);
        const uint64_t bd = B_MN ? smem_desc_sw128(b_s + kk * 16 * 128, 64 * 128, 1024)
                                 : smem_desc_sw128(b_s + kk * 32, 16, 1024);
        mma_ss(tmem, ad, bd, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(bar(kEmpty + st));
    }
    mma_commit(bar(kDone));
    mma_commit(bar(kDrain));
    volatile int never = 0;
    mbar_wait(bar(kDrain), 0, &never, status);
  }
  __syncwarp();

  // epilogue: every warp
  const bool ok = mbar_wait(bar(kDone), 0, s_abort, status);
  tc_fence_after();
  if (ok) {
    const int row = m0 + warp * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    __nv_bfloat16* crow = reinterpret_cast<__nv_bfloat16*>(p.c) +
                          ((size_t)z * p.M + row) * (size_t)p.ldc;
#pragma unroll 1
    for (int cc = 0; cc < BN; cc += 32) {
      float v[32];
      tmem_ld32(taddr + cc, v);
      tmem_wait_ld();
      if (row < p.M) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int col = n0 + cc + 8 * g;
          if (col + 8 <= p.N) {
            st_global_v4(crow + col, pack_bf16x2(v[8 * g] * p.alpha, v[8 * g + 1] * p.alpha),
                         pack_bf16x2(v[8 * g + 2] * p.alpha, v[8 * g + 3] * p.alpha),
                         pack_bf16x2(v[8 * g + 4] * p.alpha, v[8 * g + 5] * p.alpha),
                         pack_bf16x2(v[8 * g + 6] * p.alpha, v[8 * g + 7] * p.alpha));
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (col + i < p.N) crow[col + i] = __float2bfloat16_rn(v[8 * g + i] * p.alpha);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Row softmax over BF16 scores, in place. One CTA (256 threads) per row.
// Pass 1: masked row max and sum of exp(s - max) (per-thread online, then a
// block reduction); pass 2: write P = exp(s - max) / sum, and 0 in the padding
// columns [n_k, ld). LSE = max + ln(sum). A row with no visible key gets
// P = 0 and LSE = -inf.
constexpr int kSmThreads = 256;

__device__ __forceinline__ void online_merge(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  l = l * __expf(m - mn) + l2 * __expf(m2 - mn);
  m = mn;
}

__global__ void __launch_bounds__(kSmThreads)
    row_softmax_kernel(const SoftmaxParams p) {
  const int rowg = blockIdx.x;  // flattened (b, h, i)
  const int i = rowg % p.n_q;
  __nv_bfloat16* srow = reinterpret_cast<__nv_bfloat16*>(p.s) + (size_t)rowg * p.ld;
  const int lim = p.causal ? min(p.n_k, max(0, i + p.kv_off + 1)) : p.n_k;  // visible keys

  float m = -INFINITY, l = 0.f;
  for (int j0 = threadIdx.x * 8; j0 < lim; j0 += kSmThreads * 8) {
    const uint4 raw = *reinterpret_cast<const uint4*>(srow + j0);
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw);
    float vals[8];
    float mloc = -INFINITY;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      vals[t] = (j0 + t < lim) ? __bfloat162float(e[t]) : -INFINITY;
      mloc = fmaxf(mloc, vals[t]);
    }
    if (mloc == -INFINITY) continue;
    float lloc = 0.f;
#pragma unroll
    for (int t = 0; t < 8; ++t) lloc += __expf(vals[t] - mloc);
    online_merge(m, l, mloc, lloc);
  }
  // block reduction of (m, l)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    online_merge(m, l, m2, l2);
  }
  __shared__ float sm[kSmThreads / 32], sl[kSmThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm[warp] = m;
    sl[warp] = l;
  }
  __syncthreads();
  m = sm[0];
  l = sl[0];
  for (int w = 1; w < kSmThreads / 32; ++w) online_merge(m, l, sm[w], sl[w]);
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float mb = (m == -INFINITY) ? 0.f : m;
  for (int j0 = threadIdx.x * 8; j0 < p.ld; j0 += kSmThreads * 8) {
    const uint4 raw = *reinterpret_cast<const uint4*>(srow + j0);
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw);
    float pr[8];
#pragma unroll
    for (int t = 0; t < 8; ++t)
      pr[t] = (j0 + t < lim) ? __expf(__bfloat162float(e[t]) - mb) * inv : 0.f;
    st_global_v4(srow + j0, pack_bf16x2(pr[0], pr[1]), pack_bf16x2(pr[2], pr[3]),
                 pack_bf16x2(pr[4], pr[5]), pack_bf16x2(pr[6], pr[7]));
  }
  if (threadIdx.x == 0 && p.lse) p.lse[rowg] = l > 0.f ? m + logf(l) : -INFINITY;
}

template <int BN, bool B_MN>
cudaError_t launch_gemm_t(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                          int* status, cudaStream_t stream) {
  using C = GemmCfg<BN, B_MN>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<BN, B_MN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((p.N + BN - 1) / BN, (p.M + 127) / 128, p.batches);
  return launch_kernel(gemm_bf16_kernel<BN, B_MN>, grid, dim3(kGemmThreads), C::kSmemBytes, stream, ta, tb,
                       p, status);
}

}  // namespace

size_t gemm_smem_bytes(int bn) {
  return bn == 128 ? (size_t)GemmCfg<128, false>::kSmemBytes : (size_t)GemmCfg<64, false>::kSmemBytes;
}

cudaError_t launch_gemm(bool b_mn_major, int bn, const CUtensorMap& ta, const CUtensorMap& tb,
                        const GemmParams& p, int* status, cudaStream_t stream) {
  if (p.M <= 0 || p.N <= 0 || p.batches <= 0) return cudaSuccess;
  if (bn == 128) {
    return b_mn_major ? launch_gemm_t<128, true>(ta, tb, p, status, stream)
                      : launch_gemm_t<128, false>(ta, tb, p, status, stream);
  }
  return b_mn_major ? launch_gemm_t<64, true>(ta, tb, p, status, stream)
                    : launch_gemm_t<64, false>(ta, tb, p, status, stream);
}

cudaError_t launch_row_softmax(const SoftmaxParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  return launch_kernel(row_softmax_kernel, dim3((unsigned)p.rows), dim3(kSmThreads), 0, stream, p);
}

}  // namespace fa
