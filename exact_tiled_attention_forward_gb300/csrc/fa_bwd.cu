// Exact attention backward for sm_103a: dQ, dK, dV of O = softmax(scale Q K^T) V.
//
// The backward recomputes the scores tile by tile from Q, K and the per-row
// log-sum-exp the forward saved, instead of storing the N x N matrices ("Why
// is standard attention memory-bound...", Step 4; "Why does the backward pass
// recompute the scores?"). With P = exp(S - LSE) rebuilt exactly:
//   dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Two launches on the caller's stream:
//  * fa_bwd_prep_kernel: per query row, lse2 = LSE log2(e) (+inf where the row
//    sees no key, and on the padding rows of the last tile) and D, into arrays
//    padded to whole 128-row tiles.
//  * fa_bwd_kernel, whose CTAs take one of two roles (they share no data, so
//    both run side by side in one grid, the dK/dV CTAs of a KV head followed by
//    the dQ CTAs of its query heads, so its tiles are read from L2 the second time):
//    - dK/dV: one CTA per (batch, KV head, block of 128 keys). K and V of the
//      block stay in shared memory; the CTA walks the query tiles of every
//      query head that reads the KV head (GQA sums them in place, no atomics).
//      Keys are the TMEM lanes: S^T = K Q^T and dP^T = V dO^T (SS MMAs), then
//      each thread (one key) turns its row into P^T and dS^T (BF16 or FP16,
//      written back over its S^T / dP^T columns) and the MMA warp accumulates
//      dV += P^T dO and dK += dS^T Q with A read from tensor memory.
//    - dQ: one CTA per (batch, query head, 128-row tile); query rows are the
//      TMEM lanes: S = Q K^T, dP = dO V^T, then dS, then dQ += dS K.
//    Each step's score-shaped products run as two halves of 64 columns, and
//    half h of the next step is issued right behind this half's accumulating
//    products, so the element-wise pass over one half overlaps the tensor
//    core's work on the other.
// Every operand form is one the forward kernel uses: K-major SW128 tiles for
// the score-shaped products, A from tensor memory with an MN-major B for the
// accumulating ones. S and dP are computed twice (once per role): 14 N^2 d
// FLOPs of work for the 10 N^2 d of the usual count, in exchange for no
// atomic accumulation and deterministic results.
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa.h"

#include <cmath>

namespace fa {
namespace {

// warps 0-7 element-wise: two warpgroups on the same 128 TMEM lanes, warpgroup g
// taking columns [32g, 32g+32) of every 64-column half; warp 8 TMA, warp 9 MMA
constexpr int kBwdThreads = 320;
constexpr int kBwdEwThreads = 256;
constexpr int kBwdWarpProducer = 8;
constexpr int kBwdWarpMma = 9;
constexpr int kT = 128;            // query rows per tile = keys per block
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int B, H_q, H_kv, N_q, N_k, G;
  int causal, kv_off;      // kv_off = N_k - N_q: row i sees key j iff j <= i + kv_off
  int n_qt, n_kb, nq_pad;  // query tiles, key blocks, n_qt * 128
  float c;                 // scale * log2(e)
  float scale;
  const float* lse2;       // [B*H_q][nq_pad]
  const float* dsum;       // [B*H_q][nq_pad]
  void* dq;                // [B][H_q][N_q][d]
  void* dk;                // [B][H_kv][N_k][d]
  void* dv;
  int* status;
};

template <int D>
struct BwdCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = 128 * 128;        // 128 rows x 128 bytes
  static constexpr int kTileBytes = kT * D * 2;
  static constexpr int kVecBytes = kT * 4;
  static constexpr int kStages = 2;
  // resident tiles (two) and their two 128-float vectors, then the stages (two
  // tiles each, plus two vectors for the dK/dV kernel); 1024-byte aligned parts
  static constexpr int kOffRes = 0;
  static constexpr int kOffResVec = 2 * kTileBytes;
  static constexpr int kOffStages = kOffResVec + 1024;
  static constexpr int kStageBytes = 2 * kTileBytes + 1024;
  static constexpr int kOffBar = kOffStages + kStages * kStageBytes;
  // kBarS + h / kBarP + h: half h of the score-shaped products done / its
  // element-wise results stored (h = 0, 1)
  static constexpr int kBarRes = 0, kBarFull = 1, kBarEmpty = 1 + kStages, kBarS = 1 + 2 * kStages,
                       kBarP = 3 + 2 * kStages, kBarDone = 5 + 2 * kStages, kBarDrain = 6 + 2 * kStages,
                       kNumBars = 7 + 2 * kStages;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
  // launched with at least 116 KiB so that one CTA holds an SM: each CTA takes all
  // 512 tensor-memory columns, and a second one would only wait in its allocation
  static constexpr int kLaunchSmem = kSmemBytes < 116 * 1024 ? 116 * 1024 : kSmemBytes;
  static_assert(kLaunchSmem <= 227 * 1024, "shared memory");
  static constexpr uint32_t kTmemCols = 512;
  // tensor memory: [0,128) S or S^T, [128,256) dP or dP^T, each as four
  // chunks of 32 columns (two per 64-column half); the 16-bit P / P^T or dS /
  // dS^T of a chunk's 32 rows or keys is packed over the chunk's own first 16
  // columns (so neither warpgroup writes a column the other still reads);
  // [256,256+D) dV or dQ, [384,384+D) dK
  static constexpr uint32_t kTmS = 0, kTmP = 128, kTmA = 256, kTmB = 384;
};

// 1-D bulk copy global -> shared, completion counted on an mbarrier (both
// addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Tensor-memory column of the packed 16-bit operand for K-step kk (16 rows or
// keys) of half h: chunk kk / 2 of the half, its first 16 columns.
__device__ __forceinline__ uint32_t packed_col(int h, int kk) {
  return 64u * (uint32_t)h + (uint32_t)(kk >> 1) * 32u + (uint32_t)(kk & 1) * 8u;
}

__device__ __forceinline__ void bwd_publish(uint32_t bar) {
  tmem_wait_st();
  tc_fence_before();
  mbar_arrive(bar);
}

__device__ __forceinline__ void bwd_drain_wait(uint32_t bar, uint32_t parity, int* status) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, status);
}

// A 16-bit element of either type widened to FP32.
template <Elem E>
__device__ __forceinline__ float widen16(uint16_t bits) {
  if constexpr (E == Elem::F16) return __half2float(__ushort_as_half(bits));
  else return __uint_as_float((uint32_t)bits << 16);
}

// One row of 128 x D FP32 tensor-memory columns (this thread's lane) to global
// memory as 16-bit values times `mul`; `zero` writes zeros instead (no MMA ran).
// Called by every lane of the warp with warp-uniform `zero` (the tensor-memory
// load is a warp-collective instruction); only lanes with `valid` store.
// Columns [c0, c1), multiples of 32.
template <int D, Elem E>
__device__ __forceinline__ void store_row(uint32_t t_row, uint16_t* dst, float mul, bool zero, bool valid,
                                          int c0 = 0, int c1 = D) {
#pragma unroll 1
  for (int cc = c0; cc < c1; cc += 32) {
    float v[32];
    if (zero) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.f;
    } else {
      tmem_ld32(t_row + (uint32_t)cc, v);
      tmem_wait_ld();
    }
    if (!valid) continue;
#pragma unroll
    for (int g = 0; g < 4; ++g)
      st_global_v4(dst + cc + 8 * g, pack2<E>(v[8 * g] * mul, v[8 * g + 1] * mul),
                   pack2<E>(v[8 * g + 2] * mul, v[8 * g + 3] * mul), pack2<E>(v[8 * g + 4] * mul, v[8 * g + 5] * mul),
                   pack2<E>(v[8 * g + 6] * mul, v[8 * g + 7] * mul));
  }
}

// lse2 and D per query row, padded to whole tiles. One warp per padded row.
template <int D, Elem E>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const uint16_t* o, const uint16_t* dout,
                                                          const float* lse, float* lse2, float* dsum,
                                                          int N_q, int nq_pad, long long n_rows) {
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= n_rows) return;
  const long long bh = w / nq_pad;
  const int r = (int)(w - bh * nq_pad);
  if (r >= N_q) {
    if (lane == 0) {
      lse2[w] = INFINITY;
      dsum[w] = 0.f;
    }
    return;
  }
  const size_t row = ((size_t)bh * N_q + r) * D;
  constexpr int kPer = D / 32;   // elements per lane (2 or 4)
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int col = lane * kPer + i;
    acc += widen16<E>(o[row + col]) * widen16<E>(dout[row + col]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    const float l = lse[(size_t)bh * N_q + r];
    lse2[w] = (l == -INFINITY) ? INFINITY : l * kLog2e;
    dsum[w] = acc;
  }
}

// ---------------------------------------------------------------- dK, dV
template <int D, Elem E>
__device__ __forceinline__ void bwd_dkdv_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                             const CUtensorMap& tmdO, const BwdParams& p, int blk) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int bhk = blk / p.n_kb;
  const int kb = blk - bhk * p.n_kb;   // ascending: under a causal mask the first blocks are the longest
  const int b = bhk / p.H_kv, hk = bhk - b * p.H_kv;
  const int j0 = kb * kT;
  // query tiles that see at least one key of the block
  int t_lo = 0;
  if (p.causal) {
    const int first = j0 - p.kv_off;                // the first row that sees key j0
    t_lo = first <= 0 ? 0 : first / kT;
  }
  const int n_t = t_lo < p.n_qt ? p.n_qt - t_lo : 0;
  const int n_steps = p.G * n_t;

  if (warp == kBwdWarpProducer && lane == 0) {
    mbar_init(bar(C::kBarRes), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(C::kBarS + h), 1);
      mbar_init(bar(C::kBarP + h), kBwdEwThreads);
    }
    mbar_init(bar(C::kBarDone), 1);
    mbar_init(bar(C::kBarDrain), 1);
    *s_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kBwdWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kBwdWarpProducer) {
    if (lane == 0 && n_steps > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(bar(C::kBarRes), 2 * C::kTileBytes);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_3d(sb + C::kOffRes + bx * C::kBoxBytes, &tmK, bar(C::kBarRes), bx * 64, j0, bhk);
        tma_load_3d(sb + C::kOffRes + C::kTileBytes + bx * C::kBoxBytes, &tmV, bar(C::kBarRes), bx * 64, j0, bhk);
      }
      int issued = 0;
      for (int i = 0; i < n_steps; ++i, ++issued) {
        const int st = i % C::kStages;
        const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
        if (!mbar_wait(bar(C::kBarEmpty + st), ph ^ 1u, s_abort, p.status)) break;
        const int hl = i / n_t, t = t_lo + (i - hl * n_t);
        const int bhq = b * p.H_q + hk * p.G + hl;
        const int q0 = t * kT;
        const uint32_t sq = sb + C::kOffStages + st * C::kStageBytes;
        mbar_arrive_expect_tx(bar(C::kBarFull + st), 2 * C::kTileBytes + 2 * C::kVecBytes);
        const size_t vo = (size_t)bhq * p.nq_pad + q0;
        // FA_DEBUG: the stage lies in shared memory, the tile and its two vectors in their tensors
        if (!FA_DBG_OK(p.status, st < C::kStages && q0 + kT <= p.nq_pad && bhq < p.B * p.H_q))
          continue;   // reported, not loaded (the consumer's bounded wait then gives up)
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_load_3d(sq + bx * C::kBoxBytes, &tmQ, bar(C::kBarFull + st), bx * 64, q0, bhq);
          tma_load_3d(sq + C::kTileBytes + bx * C::kBoxBytes, &tmdO, bar(C::kBarFull + st), bx * 64, q0, bhq);
        }
        bulk_load_1d(sq + 2 * C::kTileBytes, p.lse2 + vo, C::kVecBytes, bar(C::kBarFull + st));
        bulk_load_1d(sq + 2 * C::kTileBytes + C::kVecBytes, p.dsum + vo, C::kVecBytes, bar(C::kBarFull + st));
      }
      // every load issued has landed before the CTA may exit
      bwd_drain_wait(bar(C::kBarRes), 0, p.status);
      for (int st = 0; st < C::kStages; ++st) {   // loads issued into stage st: its phases to wait for
        const int n_st = issued > st ? (issued - st + C::kStages - 1) / C::kStages : 0;
        if (n_st > 0) bwd_drain_wait(bar(C::kBarFull + st), (uint32_t)(n_st - 1) & 1u, p.status);
      }
    }
    __syncwarp();
  } else if (warp == kBwdWarpMma) {
    if (n_steps > 0) {
      constexpr uint32_t idS = idesc_f32(128, kT / 2, false, E);   // one half: 64 query rows
      constexpr uint32_t idO = idesc_f32(128, D, true, E);
      constexpr uint32_t kHi = desc_sw128_hi(1024);
      constexpr uint32_t kBox16 = C::kBoxBytes >> 4;
      constexpr uint32_t kHalfRows16 = (kT / 2) * 128 / 16;     // 64 rows of a 128-byte box, 16-byte units
      const uint32_t lk = desc_sw128_lo(sb + C::kOffRes, 16);
      const uint32_t lv = desc_sw128_lo(sb + C::kOffRes + C::kTileBytes, 16);
      // S^T = K Q^T and dP^T = V dO^T for the query rows of half h of step i
      // (keys on the lanes, 64 columns each), K-steps of 16 over d
      auto scores = [&](int i, int h) {
        const uint32_t sq = sb + C::kOffStages + (i % C::kStages) * C::kStageBytes;
        const uint32_t lq = desc_sw128_lo(sq, 16) + (uint32_t)h * kHalfRows16;
        const uint32_t ldo = desc_sw128_lo(sq + C::kTileBytes, 16) + (uint32_t)h * kHalfRows16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kBox16 + (uint32_t)(kk & 3) * 2u;
          mma_ss_lh_w(tmem + C::kTmS + 64u * h, lk + off, kHi, lq + off, kHi, idS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kBox16 + (uint32_t)(kk & 3) * 2u;
          mma_ss_lh_w(tmem + C::kTmP + 64u * h, lv + off, kHi, ldo + off, kHi, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(bar(C::kBarS + h));
      };
      bool ok = mbar_wait_w(bar(C::kBarRes), 0, s_abort, p.status) &&
                mbar_wait_w(bar(C::kBarFull + 0), 0, s_abort, p.status);
      if (ok) {
        tc_fence_after();
        scores(0, 0);
        scores(0, 1);
      }
      for (int i = 0; i < n_steps && ok; ++i) {
        const int st = i % C::kStages;
        const uint32_t sq = sb + C::kOffStages + st * C::kStageBytes;
        const uint32_t bdo = desc_sw128_lo(sq + C::kTileBytes, C::kBoxBytes);
        const uint32_t bq = desc_sw128_lo(sq, C::kBoxBytes);
        for (int h = 0; h < 2 && ok; ++h) {
          if (!(ok = mbar_wait_w(bar(C::kBarP + h), (uint32_t)i & 1u, s_abort, p.status))) break;
          tc_fence_after();
          // dV += P^T dO and dK += dS^T Q over the 64 rows of half h: A (keys x
          // rows) from tensor memory, B the row-major tile as an MN-major
          // operand; K-steps of 16 rows
#pragma unroll
          for (int kk = 0; kk < kT / 32; ++kk)
            mma_ts_lh_w(tmem + C::kTmA, tmem + C::kTmS + packed_col(h, kk),
                        bdo + (uint32_t)h * kHalfRows16 + (uint32_t)kk * (16u * 128u >> 4), kHi, idO,
                        (i > 0 || h > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kT / 32; ++kk)
            mma_ts_lh_w(tmem + C::kTmB, tmem + C::kTmP + packed_col(h, kk),
                        bq + (uint32_t)h * kHalfRows16 + (uint32_t)kk * (16u * 128u >> 4), kHi, idO,
                        (i > 0 || h > 0 || kk > 0) ? 1u : 0u);
          if (h == 1) mma_commit_w(bar(C::kBarEmpty + st));   // the stage's last reader
          if (i + 1 < n_steps) {
            // half h of the next step's scores, behind this half's products in
            // the pipe (they read the columns the new scores overwrite)
            if (h == 0) {
              const int i1 = i + 1;
              if (!(ok = mbar_wait_w(bar(C::kBarFull + i1 % C::kStages), (uint32_t)(i1 / C::kStages) & 1u,
                                     s_abort, p.status)))
                break;
              tc_fence_after();
            }
            scores(i + 1, h);
          }
        }
      }
      mma_commit_w(bar(C::kBarDone));
      mma_commit_w(bar(C::kBarDrain));
      bwd_drain_wait(bar(C::kBarDrain), 0, p.status);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ---- element-wise: this thread is key k of the block (TMEM lane k), in
    // warpgroup grp, which takes the 32-row chunk grp of every half
    const int grp = warp >> 2;
    const int k = (warp & 3) * 32 + lane;
    const int key = j0 + k;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::kTmS, tP = tmem + lane_base + C::kTmP;
    const float c = p.c;
    bool ok = true;
    for (int i = 0; i < n_steps && ok; ++i) {
      const int st = i % C::kStages;
      const int hl = i / n_t, t = t_lo + (i - hl * n_t);
      const int q0 = t * kT;
      const float* vl = reinterpret_cast<const float*>(smem + C::kOffStages + st * C::kStageBytes + 2 * C::kTileBytes);
      const float* vd = vl + kT;
      // rows r with key > row + kv_off are masked (causal)
      const int r_min = p.causal ? key - p.kv_off - q0 : -1;   // rows below r_min see no key k
      for (int h = 0; h < 2; ++h) {
        if (!(ok = mbar_wait_w(bar(C::kBarS + h), (uint32_t)i & 1u, s_abort, p.status))) break;
        tc_fence_after();
        // the stage's lse2 / D vectors came by TMA: observe their barrier directly
        // (it cannot move on before this thread publishes this step's second half)
        if (h == 0 &&
            !(ok = mbar_wait_w(bar(C::kBarFull + st), (uint32_t)(i / C::kStages) & 1u, s_abort, p.status)))
          break;
        const uint32_t cc = 64u * h + 32u * grp;   // this warpgroup's 32 columns = rows
        float s[32], dp[32];
        if (!FA_DBG_OK(p.status, tmem_in(lane_base + C::kTmS + cc, 32) && tmem_in(lane_base + C::kTmP + cc, 32))) {
          ok = false;   // FA_DEBUG: reported; this step is not processed
          break;
        }
        tmem_ld32(tS + cc, s);
        tmem_ld32(tP + cc, dp);
        tmem_wait_ld();
        uint32_t pk[16], dk2[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int r = (int)cc + e;
          float p0 = ex2_approx(s[e] * c - vl[r]);
          float p1 = ex2_approx(s[e + 1] * c - vl[r + 1]);
          if (r < r_min) p0 = 0.f;
          if (r + 1 < r_min) p1 = 0.f;
          pk[e >> 1] = pack2<E>(p0, p1);
          dk2[e >> 1] = pack2<E>(p0 * (dp[e] - vd[r]), p1 * (dp[e + 1] - vd[r + 1]));
        }
        // P^T / dS^T of the chunk's 32 rows over its own first 16 columns (read above)
        tmem_st16(tS + cc, pk);
        tmem_st16(tP + cc, dk2);
        bwd_publish(bar(C::kBarP + h));
      }
    }
    if (ok && n_steps > 0) {
      ok = mbar_wait_w(bar(C::kBarDone), 0, s_abort, p.status);
      tc_fence_after();
    }
    if (ok && !FA_DBG_OK(p.status, bhk < p.B * p.H_kv && tmem_in(lane_base + C::kTmA, D) &&
                                      tmem_in(lane_base + C::kTmB, D)))
      ok = false;   // FA_DEBUG: reported; nothing stored
    if (ok) {   // warp-uniform; keys past N_k (a ragged last block) load but do not store
      const bool valid = key < p.N_k;
      const size_t row = ((size_t)bhk * p.N_k + (valid ? key : 0)) * D;
      if (grp == 0)   // warpgroup 0 writes dV, warpgroup 1 dK
        store_row<D, E>(tmem + lane_base + C::kTmA, static_cast<uint16_t*>(p.dv) + row, 1.f, n_steps == 0, valid);
      else
        store_row<D, E>(tmem + lane_base + C::kTmB, static_cast<uint16_t*>(p.dk) + row, p.scale, n_steps == 0,
                        valid);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- dQ
template <int D, Elem E>
__device__ __forceinline__ void bwd_dq_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                           const CUtensorMap& tmdO, const BwdParams& p, int blk) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int bhq = blk / p.n_qt;
  const int t = p.n_qt - 1 - (blk - bhq * p.n_qt);   // descending: under a causal mask the last tiles are the longest
  const int b = bhq / p.H_q, h = bhq - b * p.H_q;
  const int bhk = b * p.H_kv + h / p.G;
  const int q0 = t * kT;
  // key blocks seen by some row of the tile
  int n_steps = p.n_kb;
  if (p.causal) {
    const int last = min(q0 + kT - 1, p.N_q - 1) + p.kv_off;   // the last key the tile sees
    n_steps = last < 0 ? 0 : min(p.n_kb, last / kT + 1);
  }

  if (warp == kBwdWarpProducer && lane == 0) {
    mbar_init(bar(C::kBarRes), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(C::kBarS + h), 1);
      mbar_init(bar(C::kBarP + h), kBwdEwThreads);
    }
    mbar_init(bar(C::kBarDone), 1);
    mbar_init(bar(C::kBarDrain), 1);
    *s_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kBwdWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kBwdWarpProducer) {
    if (lane == 0 && n_steps > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(bar(C::kBarRes), 2 * C::kTileBytes + 2 * C::kVecBytes);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_3d(sb + C::kOffRes + bx * C::kBoxBytes, &tmQ, bar(C::kBarRes), bx * 64, q0, bhq);
        tma_load_3d(sb + C::kOffRes + C::kTileBytes + bx * C::kBoxBytes, &tmdO, bar(C::kBarRes), bx * 64, q0, bhq);
      }
      const size_t vo = (size_t)bhq * p.nq_pad + q0;
      bulk_load_1d(sb + C::kOffResVec, p.lse2 + vo, C::kVecBytes, bar(C::kBarRes));
      bulk_load_1d(sb + C::kOffResVec + C::kVecBytes, p.dsum + vo, C::kVecBytes, bar(C::kBarRes));
      int issued = 0;
      for (int j = 0; j < n_steps; ++j, ++issued) {
        const int st = j % C::kStages;
        const uint32_t ph = (uint32_t)(j / C::kStages) & 1u;
        if (!mbar_wait(bar(C::kBarEmpty + st), ph ^ 1u, s_abort, p.status)) break;
        const uint32_t sk = sb + C::kOffStages + st * C::kStageBytes;
        mbar_arrive_expect_tx(bar(C::kBarFull + st), 2 * C::kTileBytes);
        if (!FA_DBG_OK(p.status, st < C::kStages && j < p.n_kb && bhk < p.B * p.H_kv))
          continue;   // FA_DEBUG: reported, not loaded
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_load_3d(sk + bx * C::kBoxBytes, &tmK, bar(C::kBarFull + st), bx * 64, j * kT, bhk);
          tma_load_3d(sk + C::kTileBytes + bx * C::kBoxBytes, &tmV, bar(C::kBarFull + st), bx * 64, j * kT, bhk);
        }
      }
      bwd_drain_wait(bar(C::kBarRes), 0, p.status);
      for (int st = 0; st < C::kStages; ++st) {   // loads issued into stage st: its phases to wait for
        const int n_st = issued > st ? (issued - st + C::kStages - 1) / C::kStages : 0;
        if (n_st > 0) bwd_drain_wait(bar(C::kBarFull + st), (uint32_t)(n_st - 1) & 1u, p.status);
      }
    }
    __syncwarp();
  } else if (warp == kBwdWarpMma) {
    if (n_steps > 0) {
      constexpr uint32_t idS = idesc_f32(128, kT / 2, false, E);   // one half: 64 keys
      constexpr uint32_t idO = idesc_f32(128, D, true, E);
      constexpr uint32_t kHi = desc_sw128_hi(1024);
      constexpr uint32_t kBox16 = C::kBoxBytes >> 4;
      constexpr uint32_t kHalfRows16 = (kT / 2) * 128 / 16;     // 64 rows of a 128-byte box, 16-byte units
      const uint32_t lq = desc_sw128_lo(sb + C::kOffRes, 16);
      const uint32_t ldo = desc_sw128_lo(sb + C::kOffRes + C::kTileBytes, 16);
      // S = Q K^T and dP = dO V^T for the keys of half h of step j (rows on the
      // lanes, 64 columns each)
      auto scores = [&](int j, int h) {
        const uint32_t sk = sb + C::kOffStages + (j % C::kStages) * C::kStageBytes;
        const uint32_t lk = desc_sw128_lo(sk, 16) + (uint32_t)h * kHalfRows16;
        const uint32_t lv = desc_sw128_lo(sk + C::kTileBytes, 16) + (uint32_t)h * kHalfRows16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kBox16 + (uint32_t)(kk & 3) * 2u;
          mma_ss_lh_w(tmem + C::kTmS + 64u * h, lq + off, kHi, lk + off, kHi, idS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kBox16 + (uint32_t)(kk & 3) * 2u;
          mma_ss_lh_w(tmem + C::kTmP + 64u * h, ldo + off, kHi, lv + off, kHi, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(bar(C::kBarS + h));
      };
      bool ok = mbar_wait_w(bar(C::kBarRes), 0, s_abort, p.status) &&
                mbar_wait_w(bar(C::kBarFull + 0), 0, s_abort, p.status);
      if (ok) {
        tc_fence_after();
        scores(0, 0);
        scores(0, 1);
      }
      for (int j = 0; j < n_steps && ok; ++j) {
        const int st = j % C::kStages;
        const uint32_t bk = desc_sw128_lo(sb + C::kOffStages + st * C::kStageBytes, C::kBoxBytes);
        for (int h = 0; h < 2 && ok; ++h) {
          if (!(ok = mbar_wait_w(bar(C::kBarP + h), (uint32_t)j & 1u, s_abort, p.status))) break;
          tc_fence_after();
          // dQ += dS K over the 64 keys of half h: dS from tensor memory, K's
          // tile as an MN-major operand
#pragma unroll
          for (int kk = 0; kk < kT / 32; ++kk)
            mma_ts_lh_w(tmem + C::kTmA, tmem + C::kTmS + packed_col(h, kk),
                        bk + (uint32_t)h * kHalfRows16 + (uint32_t)kk * (16u * 128u >> 4), kHi, idO,
                        (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
          if (h == 1) mma_commit_w(bar(C::kBarEmpty + st));   // the stage's last reader
          if (j + 1 < n_steps) {
            if (h == 0) {
              const int j1 = j + 1;
              if (!(ok = mbar_wait_w(bar(C::kBarFull + j1 % C::kStages), (uint32_t)(j1 / C::kStages) & 1u,
                                     s_abort, p.status)))
                break;
              tc_fence_after();
            }
            scores(j + 1, h);
          }
        }
      }
      mma_commit_w(bar(C::kBarDone));
      mma_commit_w(bar(C::kBarDrain));
      bwd_drain_wait(bar(C::kBarDrain), 0, p.status);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ---- element-wise: this thread is query row r of the tile (TMEM lane r),
    // in warpgroup grp, which takes the 32-key chunk grp of every half
    const int grp = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int row = q0 + r;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::kTmS, tP = tmem + lane_base + C::kTmP;
    const float c = p.c;
    bool ok = true;
    float l2 = INFINITY, dd = 0.f;
    if (n_steps > 0) {
      ok = mbar_wait_w(bar(C::kBarRes), 0, s_abort, p.status);
      const float* vl = reinterpret_cast<const float*>(smem + C::kOffResVec);
      l2 = vl[r];
      dd = vl[kT + r];
    }
    // keys at or past `lim` are masked (ragged key range, causal diagonal)
    const int lim = p.causal ? min(p.N_k, row + p.kv_off + 1) : p.N_k;
    for (int j = 0; j < n_steps && ok; ++j) {
      for (int h = 0; h < 2; ++h) {
        if (!(ok = mbar_wait_w(bar(C::kBarS + h), (uint32_t)j & 1u, s_abort, p.status))) break;
        tc_fence_after();
        const uint32_t cc = 64u * h + 32u * grp;   // this warpgroup's 32 columns = keys
        const int key0 = j * kT + (int)cc;
        float s[32], dp[32];
        if (!FA_DBG_OK(p.status, tmem_in(lane_base + C::kTmS + cc, 32) && tmem_in(lane_base + C::kTmP + cc, 32))) {
          ok = false;   // FA_DEBUG: reported; this step is not processed
          break;
        }
        tmem_ld32(tS + cc, s);
        tmem_ld32(tP + cc, dp);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int kx = key0 + e;
          float p0 = ex2_approx(s[e] * c - l2);
          float p1 = ex2_approx(s[e + 1] * c - l2);
          if (kx >= lim) p0 = 0.f;
          if (kx + 1 >= lim) p1 = 0.f;
          pk[e >> 1] = pack2<E>(p0 * (dp[e] - dd), p1 * (dp[e + 1] - dd));
        }
        // dS of the chunk's 32 keys over its own first 16 columns (read above)
        tmem_st16(tS + cc, pk);
        bwd_publish(bar(C::kBarP + h));
      }
    }
    if (ok && n_steps > 0) {
      ok = mbar_wait_w(bar(C::kBarDone), 0, s_abort, p.status);
      tc_fence_after();
    }
    if (ok && !FA_DBG_OK(p.status, bhq < p.B * p.H_q && tmem_in(lane_base + C::kTmA, D)))
      ok = false;   // FA_DEBUG: reported; nothing stored
    if (ok) {   // warp-uniform; rows past N_q (a ragged last tile) load but do not store
      const bool valid = row < p.N_q;   // warpgroup g writes columns [g D/2, (g+1) D/2)
      store_row<D, E>(tmem + lane_base + C::kTmA,
                      static_cast<uint16_t*>(p.dq) + ((size_t)bhq * p.N_q + (valid ? row : 0)) * D, p.scale,
                      n_steps == 0, valid, grp * (D / 2), (grp + 1) * (D / 2));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// One launch for both halves of the work. CTAs come in groups, one per KV
// head: its n_kb dK/dV CTAs, then the G * n_qt dQ CTAs of its query heads, so
// the second role reads the head's Q, K, V and dO tiles while they are still in
// L2 (the whole first role before the whole second left them to be read from
// DRAM twice when many heads run). Within each role of a group the longest work
// goes first (key blocks ascending, query tiles descending: under a causal mask
// those are the long ones), the group's query heads interleaved. A finer
// alternation (dK/dV block i, dQ rank i, ...) measured slower.
template <int D, Elem E>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const BwdParams p) {
  const int per = p.n_kb + p.G * p.n_qt;        // CTAs of one KV head's group
  const int grp = (int)blockIdx.x / per;        // = b * H_kv + KV head
  const int w = (int)blockIdx.x - grp * per;
  if (w < p.n_kb) {
    bwd_dkdv_cta<D, E>(tmQ, tmK, tmV, tmdO, p, grp * p.n_kb + w);
  } else {
    const int idx = w - p.n_kb;
    // rank idx / G of query head G * (KV head) + idx % G
    const int gi = idx % p.G, rank = idx / p.G;
    bwd_dq_cta<D, E>(tmQ, tmK, tmV, tmdO, p, (grp * p.G + gi) * p.n_qt + rank);
  }
}

template <int D, Elem E>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdParams& p, const void* o, const void* dout,
                         const float* lse, float* lse2, float* dsum, cudaStream_t stream) {
  using C = BwdCfg<D>;
  static bool attr[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_kernel<D, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kLaunchSmem);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  const long long rows = (long long)p.B * p.H_q * p.nq_pad;
  cudaError_t e = launch_kernel(fa_bwd_prep_kernel<D, E>, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, stream,
                                static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse, lse2,
                                dsum, p.N_q, p.nq_pad, rows);
  if (e != cudaSuccess) return e;
  const unsigned ctas = (unsigned)(p.B * p.H_kv * p.n_kb + p.B * p.H_q * p.n_qt);
  return launch_kernel(fa_bwd_kernel<D, E>, dim3(ctas), dim3(kBwdThreads), C::kLaunchSmem, stream, tq, tk, tv,
                       tdo, p);
}

bool aligned16p(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

int backward_impl(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal,
                  float scale, int elem, cudaStream_t strm) {
  const Shape s{B, H_q, H_kv, N_q, N_k, d};
  int st = validate_shape(s);
  if (st != FA_OK) return st;
  if (d == 256) return FA_ERR_UNSUPPORTED;   // the backward kernels cover d = 64 and 128
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long rows_q = (long long)B * H_q * N_q, rows_k = (long long)B * H_kv * N_k;
  const size_t qb = (size_t)rows_q * d * 2, kb = (size_t)rows_k * d * 2;
  const void* ins[6] = {q, k, v, o, lse, dout};
  const size_t in_bytes[6] = {qb, kb, kb, qb, (size_t)rows_q * 4, qb};
  void* outs[3] = {dq, dk, dv};
  const size_t out_bytes[3] = {qb, kb, kb};
  for (int i = 0; i < 6; ++i)
    if (in_bytes[i] && (!ins[i] || !aligned16p(ins[i]))) return FA_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i) {
    if (out_bytes[i] && (!outs[i] || !aligned16p(outs[i]))) return FA_ERR_INVALID_ARG;
    for (int j = 0; j < 6; ++j)
      if (overlap(outs[i], out_bytes[i], ins[j], in_bytes[j])) return FA_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)
      if (overlap(outs[i], out_bytes[i], outs[j], out_bytes[j])) return FA_ERR_INVALID_ARG;
  }
  {
    const void* all[9];
    for (int i = 0; i < 6; ++i) all[i] = in_bytes[i] ? ins[i] : nullptr;
    for (int i = 0; i < 3; ++i) all[6 + i] = out_bytes[i] ? outs[i] : nullptr;
    st = check_current_device(all, 9);
    if (st != FA_OK) return st;
  }
  // nothing to differentiate through: every gradient that exists is zero
  if (rows_q == 0 || rows_k == 0) {
    for (int i = 0; i < 3; ++i) {
      if (!out_bytes[i]) continue;
      cudaError_t e = cudaMemsetAsync(outs[i], 0, out_bytes[i], strm);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return FA_OK;
  }
  int* status = device_status_ptr();
  if (!status) return cuda_fail(cudaGetLastError());
  BwdParams p{};
  p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q; p.N_k = N_k; p.G = H_q / H_kv;
  p.causal = causal ? 1 : 0;
  p.kv_off = N_k - N_q;
  p.n_qt = (N_q + kT - 1) / kT;
  p.n_kb = (N_k + kT - 1) / kT;
  p.nq_pad = p.n_qt * kT;
  p.c = scale * kLog2e;
  p.scale = scale;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.status = status;
  if ((long long)B * H_q * p.n_qt + (long long)B * H_kv * p.n_kb >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_bf16_3d(&tq, q, d, N_q, (uint64_t)B * H_q, d, kT) ||
      !make_tmap_bf16_3d(&tdo, dout, d, N_q, (uint64_t)B * H_q, d, kT) ||
      !make_tmap_bf16_3d(&tk, k, d, N_k, (uint64_t)B * H_kv, d, kT) ||
      !make_tmap_bf16_3d(&tv, v, d, N_k, (uint64_t)B * H_kv, d, kT))
    return cuda_fail(cudaErrorInvalidValue);
  const WorkspaceSource& pool = pool_workspace();
  const size_t vec = (size_t)B * H_q * p.nq_pad * 4;
  void* ws = nullptr;
  st = pool.acquire(2 * vec, strm, &ws);
  if (st != FA_OK) return st;
  float* lse2 = static_cast<float*>(ws);
  float* dsum = reinterpret_cast<float*>(static_cast<char*>(ws) + vec);
  p.lse2 = lse2;
  p.dsum = dsum;
  cudaError_t e;
  if (elem == (int)Elem::F16)
    e = d == 128 ? launch_bwd_t<128, Elem::F16>(tq, tk, tv, tdo, p, o, dout, lse, lse2, dsum, strm)
                 : launch_bwd_t<64, Elem::F16>(tq, tk, tv, tdo, p, o, dout, lse, lse2, dsum, strm);
  else
    e = d == 128 ? launch_bwd_t<128, Elem::BF16>(tq, tk, tv, tdo, p, o, dout, lse, lse2, dsum, strm)
                 : launch_bwd_t<64, Elem::BF16>(tq, tk, tv, tdo, p, o, dout, lse, lse2, dsum, strm);
  if (pool.release) pool.release(ws, strm);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // namespace
}  // namespace fa

extern "C" int fa_backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                           const void* dout, void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int N_q,
                           int N_k, int d, int causal, float scale, int dtype, void* stream) {
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  return fa::backward_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d, causal, scale, dtype,
                           static_cast<cudaStream_t>(stream));
}
