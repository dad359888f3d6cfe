// Fused exact attention forward for sm_103a: TMA-staged Q/K/V tiles, tcgen05
// MMAs with TMEM accumulators, FP32 online softmax in registers.
//
// Method ("Flash Attention Mechanics", "The Tiling Algorithm"; "Why is standard
// attention memory-bound...", Step 3): each CTA owns a block of query rows,
// sweeps its K/V tiles, keeps a running row max m and sum l, rescales the
// partial output by exp(m_old - m_new) when the max rises, and divides by l at
// the end; the score tile lives only in tensor memory. Query-block-outer order
// with a head-major grid ("FlashAttention HBM bytes, one head, 8K", "A strong
// answer"): the CTAs of one head run together, so its K/V tiles are served
// from L2 after the first touch. Causal tiles that are fully masked are never
// loaded ("What interviewers probe next").
//
// CTA layout (320 threads, one CTA per SM):
//   warps 0-3  softmax + epilogue for query tile A (rows q0 .. q0+127)
//   warps 4-7  softmax + epilogue for query tile B (rows q0+128 .. q0+255)
//   warp  8    TMA producer (Q once, then K_j, V_j into a ring of stages)
//   warp  9    TMEM allocator and tcgen05 MMA issuer
// Tensor memory (512 columns x 128 lanes, FP32):
//   [0,128) S_A / P_A   [128,256) S_B / P_B   [256,256+d) O_A   [384,384+d) O_B
// P (BF16, two per column) overwrites the first 64 columns of its S tile and
// is the A operand of the PV MMA straight from tensor memory.
// MMA issue order per key tile j (ping-pong between the two query tiles):
//   PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
// so the tensor core works on one tile while the other tile's softmax runs.
// The commit that signals S_X(j+1) also covers PV_X(j): when a softmax warp
// sees S_X(j+1) the accumulator O_X is stable and may be rescaled in place.
//
// Lazy rescale: a row keeps its reference max until a tile's max exceeds it by
// more than 2^8 (log2 units); until then P <= 2^8, exact in the final O / l
// because O and l share the same stale reference.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {

namespace {

constexpr int kThreads = 320;
constexpr float kTau = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Cfg {
  static constexpr int kBoxes = D / 64;               // 64-column (128-byte) boxes per tile row
  static constexpr int kBoxBytes = 128 * 128;         // 128 rows x 128 bytes
  static constexpr int kTileBytes = 128 * D * 2;      // one Q, K or V tile (BF16)
  static constexpr int kStages = (D == 128) ? 4 : 8;  // K/V ring depth
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  // barriers
  static constexpr int kBarQ = 0;
  static constexpr int kBarFull = 1;
  static constexpr int kBarEmpty = 1 + kStages;
  static constexpr int kBarS = 1 + 2 * kStages;      // 2
  static constexpr int kBarP = 3 + 2 * kStages;      // 2
  static constexpr int kBarO = 5 + 2 * kStages;
  static constexpr int kBarDrain = 6 + 2 * kStages;
  static constexpr int kNumBars = 7 + 2 * kStages;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  // tensor-memory column of S_X / P_X and of O_X
  __device__ static constexpr uint32_t tm_s(int X) { return X ? 128u : 0u; }
  __device__ static constexpr uint32_t tm_o(int X) { return X ? 384u : 256u; }
};

__device__ __forceinline__ int min_i(int a, int b) { return a < b ? a : b; }
__device__ __forceinline__ int max_i(int a, int b) { return a > b ? a : b; }

// Bounded wait used on drain paths: ignores the abort flag, still gives up after the timeout.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, status);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  volatile int* s_last = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: (b, h, query block, key-range split), head-major, longest first
  const int S = p.splits;
  const int u = blockIdx.x;
  const int split = u % S;
  const int t_ = u / S;
  const int qr = t_ % p.n_qb;
  const int bh = t_ / p.n_qb;
  const int qb = p.causal ? (p.n_qb - 1 - qr) : qr;
  const int b = bh / p.H_q;
  const int h = bh - b * p.H_q;
  const int bhk = b * p.H_kv + h / (p.H_q / p.H_kv);
  const int q0 = qb * kBlockRows;

  // key tiles each query tile needs: [0, kv_hi[X]); fully masked tiles are never visited
  int kv_hi[2];
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    const int first = q0 + X * kTileM;
    if (first >= p.N_q) {
      kv_hi[X] = 0;
    } else if (!p.causal) {
      kv_hi[X] = p.n_kv_tiles;
    } else {
      const int last_key = min_i(first + kTileM - 1, p.N_q - 1) + p.kv_off;
      kv_hi[X] = last_key < 0 ? 0 : min_i(p.n_kv_tiles, last_key / kTileN + 1);
    }
  }
  const int n_all = max_i(kv_hi[0], kv_hi[1]);
  const int lo = (int)(((long long)split * n_all) / S);
  const int hi = (int)(((long long)(split + 1) * n_all) / S);
  int nX[2];
  nX[0] = max_i(0, min_i(hi, kv_hi[0]) - lo);
  nX[1] = max_i(0, min_i(hi, kv_hi[1]) - lo);
  const int nmax = max_i(nX[0], nX[1]);

  // ---- set-up
  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarQ), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    mbar_init(bar(C::kBarS + 0), 1);
    mbar_init(bar(C::kBarS + 1), 1);
    mbar_init(bar(C::kBarP + 0), 128);
    mbar_init(bar(C::kBarP + 1), 128);
    mbar_init(bar(C::kBarO), 1);
    mbar_init(bar(C::kBarDrain), 1);
    *s_abort = 0;
    *s_last = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ======================= TMA producer =======================
    if (lane == 0 && nmax > 0) {
      int issued = 0;  // K/V tile loads issued
      mbar_arrive_expect_tx(bar(C::kBarQ), 2 * C::kTileBytes);
#pragma unroll
      for (int X = 0; X < 2; ++X)
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_3d(sb + C::kOffQ + X * C::kTileBytes + bx * C::kBoxBytes, &tmQ, bar(C::kBarQ),
                      bx * 64, q0 + X * kTileM, bh);
      const uint64_t pol = policy_evict_last();
      bool ok = true;
      for (int j = 0; j < nmax && ok; ++j) {
        const int tile = lo + j;
#pragma unroll
        for (int sel = 0; sel < 2; ++sel) {  // 0: K tile, 1: V tile
          const int it = 2 * j + sel;
          const int st = it % C::kStages;
          const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
          if (!mbar_wait(bar(C::kBarEmpty + st), ph ^ 1u, s_abort, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::kBarFull + st), C::kTileBytes);
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_3d_hint(sb + C::kOffKV + st * C::kTileBytes + bx * C::kBoxBytes,
                             sel ? (const void*)&tmV : (const void*)&tmK, bar(C::kBarFull + st),
                             bx * 64, tile * kTileN, bhk, pol);
          ++issued;
        }
      }
      // drain: every load issued has landed before the CTA may exit
      drain_wait(bar(C::kBarQ), 0, p.status);
      for (int st = 0; st < C::kStages; ++st) {
        const int n_st = issued > st ? (issued - st + C::kStages - 1) / C::kStages : 0;
        if (n_st > 0) drain_wait(bar(C::kBarFull + st), (uint32_t)(n_st - 1) & 1u, p.status);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ======================= tcgen05 MMA issuer =======================
    if (lane == 0 && nmax > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, kTileN, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, true);
      auto issue_S = [&](int X, int st) {
        const uint32_t qa = sb + C::kOffQ + X * C::kTileBytes;
        const uint32_t kb = sb + C::kOffKV + st * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
          mma_ss(tmem + C::tm_s(X), smem_desc_sw128(qa + off, 16, 1024),
                 smem_desc_sw128(kb + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_PV = [&](int X, int st, bool acc) {
        const uint32_t vb = sb + C::kOffKV + st * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          mma_ts(tmem + C::tm_o(X), tmem + C::tm_s(X) + kk * 8,
                 smem_desc_sw128(vb + kk * 16 * 128, C::kBoxBytes, 1024), idO,
                 (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(bar(C::kBarQ), 0, s_abort, p.status);
      if (ok) ok = mbar_wait(bar(C::kBarFull + 0), 0, s_abort, p.status);
      if (ok) {
        tc_fence_after();
        if (nX[0] > 0) { issue_S(0, 0); mma_commit(bar(C::kBarS + 0)); }
        if (nX[1] > 0) { issue_S(1, 0); mma_commit(bar(C::kBarS + 1)); }
        mma_commit(bar(C::kBarEmpty + 0));
      }
      for (int j = 0; j < nmax && ok; ++j) {
        const int itV = 2 * j + 1, itK = 2 * j + 2;
        const int stV = itV % C::kStages, stK = itK % C::kStages;
        const uint32_t phV = (uint32_t)(itV / C::kStages) & 1u;
        const uint32_t phK = (uint32_t)(itK / C::kStages) & 1u;
        const bool next = (j + 1) < nmax;
        if (!(ok = mbar_wait(bar(C::kBarFull + stV), phV, s_abort, p.status))) break;
        tc_fence_after();
        if (j < nX[0]) {
          if (!(ok = mbar_wait(bar(C::kBarP + 0), (uint32_t)j & 1u, s_abort, p.status))) break;
          tc_fence_after();
          issue_PV(0, stV, j > 0);
        }
        if (next) {
          if (!(ok = mbar_wait(bar(C::kBarFull + stK), phK, s_abort, p.status))) break;
          tc_fence_after();
          if (j + 1 < nX[0]) { issue_S(0, stK); mma_commit(bar(C::kBarS + 0)); }
        }
        if (j < nX[1]) {
          if (!(ok = mbar_wait(bar(C::kBarP + 1), (uint32_t)j & 1u, s_abort, p.status))) break;
          tc_fence_after();
          issue_PV(1, stV, j > 0);
        }
        mma_commit(bar(C::kBarEmpty + stV));
        if (next) {
          if (j + 1 < nX[1]) { issue_S(1, stK); mma_commit(bar(C::kBarS + 1)); }
          mma_commit(bar(C::kBarEmpty + stK));
        }
      }
      mma_commit(bar(C::kBarO));
      // drain: all MMAs done before tensor memory is released
      mma_commit(bar(C::kBarDrain));
      drain_wait(bar(C::kBarDrain), 0, p.status);
    }
    __syncwarp();
  } else {
    // ======================= softmax warpgroups =======================
    const int X = warp >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;           // row within the query tile = TMEM lane
    const int row = q0 + X * kTileM + r;      // query row within the head
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::tm_s(X);
    const uint32_t tO = tmem + lane_base + C::tm_o(X);
    const int n = nX[X];
    const float c = p.c;
    const int tile_first_row = q0 + X * kTileM;
    float m_ref = -INFINITY;  // reference max, scaled log2 units
    float l = 0.f;
    bool ok = true;

    for (int j = 0; j < n; ++j) {
      if (!(ok = mbar_wait(bar(C::kBarS + X), (uint32_t)j & 1u, s_abort, p.status))) break;
      tc_fence_after();
      float s[kTileN];
      tmem_ld32(tS + 0, s);
      tmem_ld32(tS + 32, s + 32);
      tmem_ld32(tS + 64, s + 64);
      tmem_ld32(tS + 96, s + 96);
      tmem_wait_ld();
      const int key0 = (lo + j) * kTileN;
      // mask: ragged key tail, and keys after the causal diagonal
      if (key0 + kTileN > p.N_k || (p.causal && key0 + kTileN - 1 > tile_first_row + p.kv_off)) {
        int lim = p.N_k - key0;
        if (p.causal) lim = min_i(lim, row + p.kv_off + 1 - key0);
#pragma unroll
        for (int i = 0; i < kTileN; ++i)
          if (i >= lim) s[i] = -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int i = 4; i < kTileN; i += 4) {
        mx0 = fmaxf(mx0, s[i]);
        mx1 = fmaxf(mx1, s[i + 1]);
        mx2 = fmaxf(mx2, s[i + 2]);
        mx3 = fmaxf(mx3, s[i + 3]);
      }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
      const bool need = m_tile > m_ref + kTau;
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m_ref - m_tile);  // 0 on the first live tile
        m_ref = m_tile;
        l *= alpha;
      }
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O_X holds PV_X(0..j-1) and is stable (covered by the S_X(j) commit)
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float ov[32];
          tmem_ld32(tO + cc, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] *= alpha;
          tmem_st32(tO + cc, ov);
        }
      }
      const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2_approx(fmaf(s[cc * 32 + 2 * i], c, -mb));
          const float p1 = ex2_approx(fmaf(s[cc * 32 + 2 * i + 1], c, -mb));
          rs0 += p0;
          rs1 += p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + cc * 16, pk);
      }
      l += rs0 + rs1;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBarP + X));
    }
    if (ok && n > 0) {
      ok = mbar_wait(bar(C::kBarO), 0, s_abort, p.status);
      tc_fence_after();
    }
    const bool valid_row = row < p.N_q;
    if (S == 1) {
      // ---- final epilogue: O / l -> BF16, LSE
      if (ok) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow =
            reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)bh * p.N_q + row) * D;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float ov[32];
          if (n > 0) {
            tmem_ld32(tO + cc, ov);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = 0.f;
          }
          if (valid_row) {
#pragma unroll
            for (int g = 0; g < 4; ++g)
              st_global_v4(orow + cc + 8 * g, pack_bf16x2(ov[8 * g + 0] * inv, ov[8 * g + 1] * inv),
                           pack_bf16x2(ov[8 * g + 2] * inv, ov[8 * g + 3] * inv),
                           pack_bf16x2(ov[8 * g + 4] * inv, ov[8 * g + 5] * inv),
                           pack_bf16x2(ov[8 * g + 6] * inv, ov[8 * g + 7] * inv));
          }
        }
        if (valid_row && p.lse)
          p.lse[(size_t)bh * p.N_q + row] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      }
    } else {
      // ---- partial: unnormalised O, (m, l) to the workspace; last CTA of the block merges
      const size_t blk = (size_t)bh * p.n_qb + qb;
      const size_t prow = (blk * S + split) * kBlockRows + X * kTileM + r;
      if (ok) {
        float* po = p.part_o + prow * D;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float ov[32];
          if (n > 0) {
            tmem_ld32(tO + cc, ov);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = 0.f;
          }
#pragma unroll
          for (int g = 0; g < 8; ++g)
            __stcg(reinterpret_cast<float4*>(po + cc) + g,
                   make_float4(ov[4 * g], ov[4 * g + 1], ov[4 * g + 2], ov[4 * g + 3]));
        }
        __stcg(reinterpret_cast<float2*>(p.part_ml) + prow, make_float2(l > 0.f ? m_ref : -INFINITY, l));
        __threadfence();
      }
      named_bar_sync(1, 256);
      if (threadIdx.x == 0) {
        int last = 0;
        if (!*s_abort) last = (atomicAdd(p.counters + blk, 1) == S - 1);
        *s_last = last;
      }
      named_bar_sync(1, 256);
      if (*s_last && ok) {
        __threadfence();
        const size_t rbase = blk * S * kBlockRows + X * kTileM + r;
        float M = -INFINITY;
        for (int s2 = 0; s2 < S; ++s2) {
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + rbase + (size_t)s2 * kBlockRows);
          if (ml.y > 0.f) M = fmaxf(M, ml.x);
        }
        float L = 0.f;
        for (int s2 = 0; s2 < S; ++s2) {
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + rbase + (size_t)s2 * kBlockRows);
          if (ml.y > 0.f) L += ex2_approx(ml.x - M) * ml.y;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        if (valid_row) {
          __nv_bfloat16* orow =
              reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)bh * p.N_q + row) * D;
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 8) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
            for (int s2 = 0; s2 < S; ++s2) {
              const size_t pr = rbase + (size_t)s2 * kBlockRows;
              const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + pr);
              if (!(ml.y > 0.f)) continue;
              const float w = ex2_approx(ml.x - M) * inv;
              const float4 a = __ldcg(reinterpret_cast<const float4*>(p.part_o + pr * D + cc));
              const float4 b2 = __ldcg(reinterpret_cast<const float4*>(p.part_o + pr * D + cc) + 1);
              acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
              acc[4] += w * b2.x; acc[5] += w * b2.y; acc[6] += w * b2.z; acc[7] += w * b2.w;
            }
            st_global_v4(orow + cc, pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                         pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
          }
          if (p.lse)
            p.lse[(size_t)bh * p.N_q + row] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
        }
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace

size_t fwd_smem_bytes(int d) {
  return d == 128 ? (size_t)Cfg<128>::kSmemBytes : (size_t)Cfg<64>::kSmemBytes;
}

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int units, cudaStream_t stream) {
  if (units <= 0) return cudaSuccess;
  if (d == 128) {
    static bool attr = false;  // benign race: setting the attribute twice is harmless
    if (!attr) {
      cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Cfg<128>::kSmemBytes);
      if (e != cudaSuccess) return e;
      attr = true;
    }
    fa_fwd_kernel<128><<<units, kThreads, Cfg<128>::kSmemBytes, stream>>>(tq, tk, tv, p);
  } else {
    static bool attr = false;
    if (!attr) {
      cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Cfg<64>::kSmemBytes);
      if (e != cudaSuccess) return e;
      attr = true;
    }
    fa_fwd_kernel<64><<<units, kThreads, Cfg<64>::kSmemBytes, stream>>>(tq, tk, tv, p);
  }
  return cudaGetLastError();
}

}  // namespace fa
