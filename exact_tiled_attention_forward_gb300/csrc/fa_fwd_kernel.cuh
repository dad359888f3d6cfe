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
// CTA layout (384 threads = three warpgroups, one CTA per SM):
//   warpgroup 0 (warps 0-3)  softmax + epilogue for query tile A (rows q0 .. q0+127)
//   warpgroup 1 (warps 4-7)  softmax + epilogue for query tile B (rows q0+128 .. q0+255)
//   warpgroup 2: warp 8 TMA producer, warp 9 TMEM allocator + tcgen05 MMA
//                issuer, warps 10-11 idle
// One thread per query row (TMEM lane). Registers: launched at 168 per
// thread; warpgroup 2 gives registers back (setmaxnreg 72) and the softmax
// warpgroups take them (216 each): 128 x (216 + 216 + 72) = 64,512 =
// 384 x 168, so the increase always fits. (Measured: 216/72 runs 1-4 % faster
// than 224/56, whose MMA-issuing warp spilled inside its loop.)
//
// Tensor memory (512 columns x 128 lanes, FP32):
//   [0,128) S_A   [128,256) S_B   [256,256+d) O_A   [384,384+d) O_B
// P (BF16, two per column) overwrites the first 64 columns of its S tile
// (all 128 scores of a row are in registers first) and is the A operand of the
// PV MMA straight from tensor memory.
// MMA issue order per key tile j (ping-pong between the two query tiles):
//   PV_A(j) keys 0..63, PV_A(j) keys 64..127, S_A(j+1), then the same for B
// The softmax hands P over in two halves (keys 0..63, then 64..127), so the
// first half of PV_X(j) runs while the second half of P is computed. The
// commit that signals S_X(j+1) also covers PV_X(j): when a softmax warp sees
// S_X(j+1) the accumulator O_X is stable and may be rescaled in place.
//
// Softmax per tile: exponentials are computed against the row's reference
// max m (log2 units). A row's reference is set from the tile max on its first
// live tile; afterwards P = 2^(s c - m) may exceed 1, and only when the first
// half's sum of P exceeds 2^tau (so some P may) or the second half's max exceeds
// m + tau is the reference raised to the tile max, O and l rescaled and the
// first half redone, all before P is handed over. tau = 16 for BF16 and 15 for
// FP16 tensors: P <= 2^tau keeps every value in range of the element type P is
// stored in, and the final O / l and LSE are exact because O and l share the
// reference. An overflowed P makes the sum infinite and takes the same path.
//
// Element type: BF16 or FP16 (Q, K, V, P and O all of one type, FP32 accumulation);
// only the instruction descriptors, the conversions and tau differ.
//
// This header holds the kernel template and its launch helpers; fa_fwd.cu
// instantiates the plain kernel for libfa. The paired-load variant (MC = true)
// needs cluster-multicast operations that only the single-GPU library
// defines (McOps<true>), so libfa never contains them.
#pragma once
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {

// Cluster-multicast operations of the paired-load variant (MC = true): a TMA
// tile load delivered to several CTAs of the cluster, and an MMA commit that
// arrives on several CTAs' barriers. Only the single-GPU library specialises
// this template; nothing here instantiates it for MC = false.
template <bool MC>
struct McOps;

namespace {

constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 216;   // per thread, warpgroups 0-1
constexpr int kRegsOther = 72;      // per thread, warpgroup 2
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
// A row's reference max may lag its true max by up to kTau (log2 units), so P
// stays <= 2^kTau: 2^16 in BF16, 2^15 in FP16 (whose largest finite value is
// 65504), 2^8 in FP8 E4M3 (largest finite value 448).
template <Elem E>
struct Lag {
  static constexpr float kTau = E == Elem::F16 ? 15.0f : (E == Elem::E4M3 ? 8.0f : 16.0f);
  static constexpr float kSumCap = E == Elem::F16 ? 32768.0f : (E == Elem::E4M3 ? 256.0f : 65536.0f);
};
// Element type of O: the input type, except BF16 for FP8 inputs.
template <Elem E>
constexpr Elem kOutElem = E == Elem::E4M3 ? Elem::BF16 : E;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, Elem E = Elem::BF16>
struct Cfg {
  static constexpr int kEsz = E == Elem::E4M3 ? 1 : 2;   // bytes per Q, K, V element
  // Q, K, V tiles: boxes of 128 rows with a 128-byte swizzle (64-byte rows,
  // and a 64-byte swizzle, for FP8 at d = 64, whose rows are 64 bytes long)
  static constexpr int kRowBytes = D * kEsz;
  static constexpr int kSwz = kRowBytes < 128 ? kRowBytes : 128;   // swizzle span = box row bytes
  static_assert(kSwz == 64 || kSwz == 128, "64- or 128-byte swizzle");
  static constexpr int kBoxCols = kSwz / kEsz;            // elements in one box row
  static constexpr int kBoxes = kRowBytes / kSwz;         // boxes per tile row
  static constexpr int kBoxBytes = 128 * kSwz;            // 128 rows x kSwz bytes
  static constexpr int kKPerBox = kSwz / 32;              // S MMAs (32 bytes of K each) per box
  static constexpr int kOBoxes = D / 64;                  // 64-column boxes of a 16-bit O row
  static constexpr int kStgBoxBytes = 128 * 128;          // staging boxes (O, partials): 128 x 128 bytes
  static constexpr int kTileBytes = 128 * D * kEsz;       // one Q, K or V tile
  static constexpr int kOTileBytes = 128 * D * 2;         // one 16-bit O tile
  static constexpr int kPartTileBytes = 128 * D * 4;      // one FP32 partial tile
  static constexpr int kStages = kTileBytes >= 32768 ? 4 : 8;   // K/V ring depth
  // MMAs per tile: S = Q K^T takes 32 bytes of d per MMA (16 BF16/FP16 or 32 FP8
  // elements); P V takes kPVKeys keys per MMA, 8 TMEM columns of P each
  static constexpr int kSKSteps = D * kEsz / 32;
  static constexpr int kPVKeys = 32 / kEsz;
  // TMEM columns of one 64-key half of P (2 BF16/FP16 or 4 FP8 values per column)
  static constexpr uint32_t kPHalfCols = 64 * kEsz / 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  // barriers
  static constexpr int kBarQ = 0;
  static constexpr int kBarFull = 1;
  static constexpr int kBarEmpty = 1 + kStages;
  static constexpr int kBarS = 1 + 2 * kStages;      // [2] S_X ready
  static constexpr int kBarP1 = 3 + 2 * kStages;     // [2] P_X keys 0..63 in TMEM
  static constexpr int kBarP2 = 5 + 2 * kStages;     // [2] P_X keys 64..127 in TMEM
  static constexpr int kBarO = 7 + 2 * kStages;
  static constexpr int kBarDrain = 8 + 2 * kStages;
  static constexpr int kNumBars = 9 + 2 * kStages;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // in-cluster merge: (m, l) of up to kCmRows partial rows received from the
  // cluster; their O rows land in [0, kOffBar) (the Q tiles and the K/V ring)
  static constexpr int kCmRows = kBlockRows;                  // (m, l) of every row, by sender
  static constexpr int kOffCm = (kOffMisc + 64 + 15) & ~15;
  static constexpr int kCmStage = kBlockRows * D * 4;         // after the FP32 receive buffer
  // + alignment slack; at least 120 KB, so that two CTAs never share an SM: each
  // allocates all 512 TMEM columns, and a second allocation on the SM would
  // wait for the first CTA to finish (FP8 tiles at d = 64 need only ~80 KB)
  static constexpr int kSmemUsed = kOffCm + kCmRows * 8 + 1024;
  static constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
  static_assert(kCmStage + 128 * D * 2 <= kOffBar, "merge buffers must fit in the Q tiles and the K/V ring");
  static_assert(2 * kPartTileBytes <= kStages * kTileBytes, "both partial tiles fit in the K/V ring");
  static_assert(kEsz == 2 || 2 * kOTileBytes <= kStages * kTileBytes, "FP8: O staged in the K/V ring");
  static constexpr uint32_t kTmemCols = 512;
  // tensor-memory column of S_X / P_X and of O_X
  __device__ static constexpr uint32_t tm_s(int X) { return X ? 128u : 0u; }
  __device__ static constexpr uint32_t tm_o(int X) { return X ? 384u : 256u; }
};

__device__ __forceinline__ int min_i(int a, int b) { return a < b ? a : b; }
// How a tile step treats the mask: never, always, or as the tile needs
// (checked at run time).
enum class MaskMode { kNone, kAlways, kCheck };
template <MaskMode M>
struct MaskTag {
  static constexpr MaskMode value = M;
};
__device__ __forceinline__ int max_i(int a, int b) { return a > b ? a : b; }

// P = 2^(s*c - mb) for 64 scores of this thread's row (FP32 pairs, one packed
// FMA per pair), packed to the P type (BF16 or FP16: 32 TMEM columns from tP;
// FP8 E4M3: 16 columns). Returns the sum of P (FP32, before rounding).
// Software-pipelined in chunks of 16: the exponentials of chunk k+1 are issued
// before chunk k is packed and stored, so the exp unit stays busy.
template <Elem E>
__device__ __forceinline__ float exp_half(const float* s, float c, float mb, uint32_t tP) {
  float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
  float pa[16], pb[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float2 e = ffma2_bc(make_float2(s[i], s[i + 1]), c, -mb);
    pa[i] = ex2_approx(e.x);
    pa[i + 1] = ex2_approx(e.y);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k + 1 < 4) {
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float2 e = ffma2_bc(make_float2(s[(k + 1) * 16 + i], s[(k + 1) * 16 + i + 1]), c, -mb);
        pb[i] = ex2_approx(e.x);
        pb[i + 1] = ex2_approx(e.y);
      }
    }
    if constexpr (E == Elem::E4M3) {
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pk[i] = pack4_e4m3(pa[4 * i], pa[4 * i + 1], pa[4 * i + 2], pa[4 * i + 3]);
      tmem_st4(tP + (uint32_t)k * 4u, pk);
    } else {
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) pk[i] = pack2<E>(pa[2 * i], pa[2 * i + 1]);
      tmem_st8(tP + (uint32_t)k * 8u, pk);
    }
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      sa = fadd2(sa, make_float2(pa[i], pa[i + 1]));
      sb = fadd2(sb, make_float2(pa[i + 2], pa[i + 3]));
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) pa[i] = pb[i];
  }
  return (sa.x + sa.y) + (sb.x + sb.y);
}

// Max of n (a multiple of 4) raw scores.
template <int N>
__device__ __forceinline__ float max_scores(const float* s) {
  float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    a0 = max3f(a0, s[i], s[i + 1]);
    a1 = max3f(a1, s[i + 2], s[i + 3]);
  }
  return fmaxf(a0, a1);
}

// O_X *= alpha for this thread's row (all lanes of the warp take part).
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
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

// Hand P (or half of it) to the MMA warp: stores complete, then arrive.
__device__ __forceinline__ void publish(uint32_t bar) {
  tmem_wait_st();
  tc_fence_before();
  mbar_arrive(bar);
}

// Bounded wait used on drain paths: ignores the abort flag, still gives up after the timeout.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, status);
}

// ---- in-cluster merge of the split partials (all query blocks split into S
// key ranges, S in {2, 4, 8}; the S CTAs of a block form one cluster). Row rr
// of the block (0..255) is finished by CTA rr / R, R = 256 / S: every CTA sends
// its unnormalised FP32 O row and (m, l) there, and the owner combines the S
// partials exactly as the merge of whole key ranges does (page 2, "The Tiling
// Algorithm"). Distributed shared memory moves ~20 B/clk per SM at best, and
// only when a warp's store covers contiguous bytes, so the receive buffer is
// laid out [sender][16-byte chunk][row]: the 32 consecutive rows of a warp
// write 512 contiguous bytes per store. Rows a CTA owns stay local.
template <int D>
__device__ __forceinline__ void cm_send(uint32_t sb, uint32_t ml_base, int S, int v, int rr, uint32_t tO,
                                        int n, float m, float l) {
  constexpr int kC = D / 4;               // 16-byte FP32 chunks per row
  const int R = kBlockRows / S;
  const int w = rr / R;                   // owner: the same for all 32 rows of a warp
  const int lr = rr - w * R;
  const uint32_t loc = sb + (uint32_t)(v * kC * R + lr) * 16u;   // chunk 0 of this row, slot v
  const bool local = (w == v);
  const uint32_t dst = local ? loc : mapa_shared(loc, (uint32_t)w);
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
    for (int g = 0; g < 8; ++g) {
      const uint32_t a = dst + (uint32_t)((cc / 4 + g) * R) * 16u;
      const uint32_t x0 = __float_as_uint(ov[4 * g]), x1 = __float_as_uint(ov[4 * g + 1]);
      const uint32_t x2 = __float_as_uint(ov[4 * g + 2]), x3 = __float_as_uint(ov[4 * g + 3]);
      if (local) st_shared_v4(a, x0, x1, x2, x3);
      else st_cluster_v4(a, x0, x1, x2, x3);
    }
  }
  const uint32_t mla = ml_base + (uint32_t)(v * R + lr) * 8u;
  st_cluster_v2f(local ? mla : mapa_shared(mla, (uint32_t)w), l > 0.f ? m : -INFINITY, l);
}

// Owner side (warps 0-7): one lane per row, each warp a group of 32 rows and a
// range of 8-column chunks, two chunks at a time with all their loads issued
// first; O is staged as BF16 in 64-column, 128-byte swizzled boxes of R rows and
// written by TMA stores (tmO has R-row boxes). S (2, 4 or 8) is a template
// parameter so the per-source arrays are exactly sized. Not inlined: it runs
// once per CTA, and compiled apart it leaves the main loop's registers alone.
template <int D, int S, Elem E>
__device__ __noinline__ void cm_reduce(uint32_t sb, uint32_t ml_base, uint32_t stage, int w, int warp,
                                       int lane, bool ok, const FwdParams& p, const CUtensorMap* tmO,
                                       int bh, int q0, float o_scale) {
  constexpr int kC = D / 4;               // FP32 chunks per row
  constexpr int kCB = D / 8;              // BF16 16-byte chunks per row
  constexpr int R = kBlockRows / S;
  constexpr int kPerWarp = (R / 32) * kCB / 8;   // BF16 chunks per warp (1 .. 8)
  const int item0 = warp * kPerWarp;
  const int lr = (item0 / kCB) * 32 + lane;
  const int row = q0 + w * R + lr;
  float ms[S], ls[S], wv[S];
  float M = -INFINITY;
#pragma unroll
  for (int v = 0; v < S; ++v) {
    const float2 ml = ld_shared_v2f(ml_base + (uint32_t)(v * R + lr) * 8u);
    ms[v] = ml.x;
    ls[v] = ml.y;
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  float L = 0.f;
#pragma unroll
  for (int v = 0; v < S; ++v) {
    wv[v] = ls[v] > 0.f ? ex2_approx(ms[v] - M) : 0.f;
    L += wv[v] * ls[v];
  }
  const float inv = L > 0.f ? o_scale / L : 0.f;
#pragma unroll
  for (int v = 0; v < S; ++v) wv[v] *= inv;
  if ((item0 % kCB) == 0 && row < p.N_q && p.lse)
    p.lse[(size_t)bh * p.N_q + row] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
  constexpr int kStep = kPerWarp >= 2 ? 2 : 1;
#pragma unroll 1
  for (int i = 0; i < kPerWarp; i += kStep) {
    float4 t[kStep][S][2];
#pragma unroll
    for (int q = 0; q < kStep; ++q) {
      const int cb = (item0 + i + q) % kCB;
#pragma unroll
      for (int v = 0; v < S; ++v) {
        const uint32_t a = sb + (uint32_t)((v * kC + 2 * cb) * R + lr) * 16u;
        t[q][v][0] = ld_shared_v4f(a);
        t[q][v][1] = ld_shared_v4f(a + (uint32_t)R * 16u);
      }
    }
#pragma unroll
    for (int q = 0; q < kStep; ++q) {
      const int cb = (item0 + i + q) % kCB;
      float acc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = 0.f;
#pragma unroll
      for (int v = 0; v < S; ++v) {
        acc[0] += wv[v] * t[q][v][0].x; acc[1] += wv[v] * t[q][v][0].y;
        acc[2] += wv[v] * t[q][v][0].z; acc[3] += wv[v] * t[q][v][0].w;
        acc[4] += wv[v] * t[q][v][1].x; acc[5] += wv[v] * t[q][v][1].y;
        acc[6] += wv[v] * t[q][v][1].z; acc[7] += wv[v] * t[q][v][1].w;
      }
      const int bx = cb >> 3, cbb = cb & 7;
      constexpr Elem OE = kOutElem<E>;
      st_shared_v4(stage + (uint32_t)(bx * R + lr) * 128u + ((uint32_t)(cbb ^ (lr & 7)) << 4),
                   pack2<OE>(acc[0], acc[1]), pack2<OE>(acc[2], acc[3]), pack2<OE>(acc[4], acc[5]),
                   pack2<OE>(acc[6], acc[7]));
    }
  }
  fence_proxy_async_smem();
  const bool all_ok = named_bar_and(1, 256, ok);
  if (all_ok && warp == 0 && lane == 0 && q0 + w * R < p.N_q) {   // rows past N_q are clipped
#pragma unroll
    for (int bx = 0; bx < D / 64; ++bx)
      tma_store_3d(tmO, stage + (uint32_t)(bx * R) * 128u, bx * 64, q0 + w * R, bh);
    bulk_commit();
    bulk_wait_read0();
  }
}

// Query block number qlin -> (b * H_q + h, query block). Non-causal: head-major,
// blocks in order. Causal: blocks differ in length, and the grid is handed
// out in order, so the heads are taken in groups of p.hgroup (as many as keep
// their K/V in L2 together); inside a group the blocks run longest first with
// the group's heads interleaved (the last block of every head, then the one
// before, ...). Head-major order would leave the longest blocks of the last
// heads to start at the very end. hgroup = 1 is head-major, longest first.
__device__ __forceinline__ void block_of(const FwdParams& p, int qlin, int& bh, int& qb) {
  if (!p.causal) {
    bh = qlin / p.n_qb;
    qb = qlin - bh * p.n_qb;
    return;
  }
  const int g = p.hgroup;
  const int per = g * p.n_qb;
  const int grp = qlin / per;
  const int w = qlin - grp * per;
  const int gh = min_i(g, p.n_bh - grp * g);   // heads in this group (the last may have fewer)
  const int rank = w / gh;
  bh = grp * g + (w - rank * gh);
  qb = p.n_qb - 1 - rank;
}

// Query block and key-tile counts of work unit u (see the kernel's unit comment).
struct UnitInfo {
  int bh, qb, split, S, slot, lo, n0, n1, nmax;
};
__device__ __forceinline__ UnitInfo unit_info(const FwdParams& p, int u) {
  UnitInfo ui;
  int qlin;
  if (u < p.u_full) {
    qlin = u; ui.split = 0; ui.S = 1; ui.slot = -1;
  } else {
    const int v = u - p.u_full;
    qlin = p.u_full + v / p.s_tail; ui.split = v % p.s_tail; ui.S = p.s_tail; ui.slot = v;
  }
  block_of(p, qlin, ui.bh, ui.qb);
  const int q0 = ui.qb * kBlockRows;
  // key tiles each query tile needs: [0, kv_hi); fully masked tiles are never visited
  int kvh[2];
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    const int first = q0 + X * kTileM;
    if (first >= p.N_q) {
      kvh[X] = 0;
    } else if (!p.causal) {
      kvh[X] = p.n_kv_tiles;
    } else {
      const int last_key = min_i(first + kTileM - 1, p.N_q - 1) + p.kv_off;
      kvh[X] = last_key < 0 ? 0 : min_i(p.n_kv_tiles, last_key / kTileN + 1);
    }
  }
  const int n_all = max_i(kvh[0], kvh[1]);
  // split * n_all < 2^29 (at most 16 splits of at most 2^24 key tiles): 32-bit division
  ui.lo = (int)(((unsigned)ui.split * (unsigned)n_all) / (unsigned)ui.S);
  const int hi = (int)(((unsigned)(ui.split + 1) * (unsigned)n_all) / (unsigned)ui.S);
  ui.n0 = max_i(0, min_i(hi, kvh[0]) - ui.lo);
  ui.n1 = max_i(0, min_i(hi, kvh[1]) - ui.lo);
  ui.nmax = max_i(ui.n0, ui.n1);
  return ui;
}

// MC (multicast): CTAs run in clusters of two (units u and u ^ 1). When both
// units belong to the same head they share every K/V tile load: each CTA
// fetches half the tile's rows once from L2 and multicasts them into both
// CTAs' shared memory, and a stage is refilled only after both CTAs' MMAs have
// released it (each MMA commit arrives on both CTAs' "empty" barriers). A
// causal pair walks the union of its key ranges (the shorter unit only
// releases the extra tiles). Single-GPU only: the tiles come from this GPU's
// own memory.
template <int D, bool MC, Elem E>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const __grid_constant__ CUtensorMap tmP, const FwdParams p) {
  using C = Cfg<D, E>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // FA_DEBUG bounds: the usable shared memory is [sb, s_hi)
  [[maybe_unused]] const uint32_t s_hi = sb + (uint32_t)(C::kSmemBytes - 1024);

  // barriers first (the plain kernel's counts do not depend on the unit), so
  // their set-up overlaps the parameter loads of the unit decode below
  if (!MC && warp == kWarpProducer && lane == 0) {
    mbar_init(bar(C::kBarQ), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    mbar_init(bar(C::kBarS + 0), 1);
    mbar_init(bar(C::kBarS + 1), 1);
    for (int X = 0; X < 2; ++X) {
      mbar_init(bar(C::kBarP1 + X), 128);
      mbar_init(bar(C::kBarP2 + X), 128);
    }
    mbar_init(bar(C::kBarO), 1);
    mbar_init(bar(C::kBarDrain), 1);
    *s_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }

  // ---- work unit. Units [0, u_full) are whole query blocks written directly;
  // the rest split the last query blocks' key ranges into s_tail parts whose
  // partial (m, l, O) go to the workspace (merged by fa_merge_kernel). Query
  // blocks are numbered head-major (a head's blocks are adjacent, so its K/V
  // stay in L2); causal blocks run longest first within groups of heads whose
  // K/V fit in L2 together (block_of).
  const int u = blockIdx.x;
  const bool idle = MC && u >= p.n_units;   // completes the last cluster only
  const UnitInfo ui = unit_info(p, idle ? 0 : u);
  const int bh = ui.bh, qb = ui.qb, slot = ui.slot, lo = ui.lo;
  const int n0 = idle ? 0 : ui.n0, n1 = idle ? 0 : ui.n1;
  const int nmax = idle ? 0 : ui.nmax;
  const int b = bh / p.H_q;
  const int h = bh - b * p.H_q;
  const int bhk = b * p.H_kv + h / (p.H_q / p.H_kv);
  const int q0 = qb * kBlockRows;
  // cluster pairing: share K/V loads with the partner unit if it is the same head
  bool share = false;
  int n_loop = nmax;        // key tiles this CTA loads and releases
  const int rank = u & 1;
  if (MC && !idle) {
    const int partner = u ^ 1;
    if (partner < p.n_units) {
      const UnitInfo pi = unit_info(p, partner);
      if (pi.bh == bh && pi.lo == lo) {
        share = true;
        n_loop = max_i(nmax, pi.nmax);
      }
    }
  }

  // ---- set-up. The producer lane initialises the barriers and starts the Q
  // loads at once, so they overlap the rest of the set-up.
  if (warp == kWarpProducer && lane == 0) {
    if (MC) {
      mbar_init(bar(C::kBarQ), 1);
      for (int s = 0; s < C::kStages; ++s) {
        mbar_init(bar(C::kBarFull + s), 1);
        mbar_init(bar(C::kBarEmpty + s), share ? 2 : 1);   // both CTAs release a shared stage
      }
      mbar_init(bar(C::kBarS + 0), 1);
      mbar_init(bar(C::kBarS + 1), 1);
      for (int X = 0; X < 2; ++X) {
        mbar_init(bar(C::kBarP1 + X), 128);   // all 128 rows of the tile
        mbar_init(bar(C::kBarP2 + X), 128);
      }
      mbar_init(bar(C::kBarO), 1);
      mbar_init(bar(C::kBarDrain), 1);
      *s_abort = 0;
      fence_mbar_init();
      fence_proxy_async_smem();
    }
    // the merge kernel (launched as a programmatic dependent) may be scheduled
    // once every CTA of this grid has started; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    // this grid may itself start before the previous kernel on the stream has
    // finished (programmatic launch): no global read before this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (n_loop > 0) {
      mbar_arrive_expect_tx(bar(C::kBarQ), 2 * C::kTileBytes);
#pragma unroll
      for (int X = 0; X < 2; ++X)
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_3d(sb + C::kOffQ + X * C::kTileBytes + bx * C::kBoxBytes, &tmQ, bar(C::kBarQ),
                      bx * C::kBoxCols, q0 + X * kTileM, bh);
    }
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (MC) cluster_sync();   // the partner's barriers exist before any multicast reaches them

  if (idle) {
    // no work: only the cluster barriers and the teardown
  } else if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (warp == kWarpProducer) {
      // ======================= TMA producer =======================
      if (lane == 0 && n_loop > 0) {
        int issued = 0;  // K/V tile loads issued (the Q loads were issued at set-up)
        const uint64_t pol = policy_evict_last();
        bool ok = true;
        for (int j = 0; j < n_loop && ok; ++j) {
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
            const void* tmap = sel ? (const void*)&tmV : (const void*)&tmK;
            const uint32_t dst = sb + C::kOffKV + st * C::kTileBytes;
            if (!FA_DBG_OK(p.status, smem_in(dst, C::kTileBytes, sb + C::kOffKV, sb + C::kOffBar) &&
                                         tile < p.n_kv_tiles)) {
              // FA_DEBUG: reported, not loaded (the consumer's bounded wait then gives up)
            } else if (!MC) {
#pragma unroll
              for (int bx = 0; bx < C::kBoxes; ++bx)
                tma_load_3d_hint(dst + bx * C::kBoxBytes, tmap, bar(C::kBarFull + st), bx * C::kBoxCols,
                                 tile * kTileN, bhk, pol);
            } else if (share) {
              // this CTA's half of the rows, into both CTAs
              if constexpr (MC) {
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx)
                  McOps<MC>::load_3d(dst + bx * C::kBoxBytes + rank * (kTileN / 2) * 128, tmap,
                                     bar(C::kBarFull + st), bx * 64, tile * kTileN + rank * (kTileN / 2),
                                     bhk, (uint16_t)0x3);
              }
            } else {
#pragma unroll
              for (int bx = 0; bx < C::kBoxes; ++bx)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                  tma_load_3d_hint(dst + bx * C::kBoxBytes + hf * (kTileN / 2) * 128, tmap,
                                   bar(C::kBarFull + st), bx * 64, tile * kTileN + hf * (kTileN / 2),
                                   bhk, pol);
            }
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
    } else if (warp == kWarpMma) {
      // ======================= tcgen05 MMA issuer =======================
      // the whole warp runs this loop converged; elected lanes issue (see mma_ss_lh_w)
      if (n_loop > 0) {
        // a stage is released to this CTA's producer, and with sharing to the partner's too
        auto release = [&](int st) {
          if constexpr (MC) {
            if (share) {
              McOps<MC>::commit_w(bar(C::kBarEmpty + st), (uint16_t)0x3);
              return;
            }
          }
          mma_commit_w(bar(C::kBarEmpty + st));
        };
        constexpr uint32_t idS = idesc_f32(128, kTileN, false, E);
        constexpr uint32_t idO = idesc_f32(128, D, true, E);
        // Descriptors are built once; each MMA adds a compile-time offset to the
        // start-address field (16-byte units) of the low word, so issuing stays
        // ahead of the tensor core.
        constexpr uint32_t kStageStep = (uint32_t)(C::kTileBytes >> 4);
        // 8-row swizzle atoms: SBO = 8 rows of the box
        constexpr uint32_t kHi = C::kSwz == 128 ? desc_sw128_hi(1024) : desc_sw64_hi(512);
        const uint32_t lq0 = desc_sw128_lo(sb + C::kOffQ, 16);
        const uint32_t lk0 = desc_sw128_lo(sb + C::kOffKV, 16);
        const uint32_t lv0 = desc_sw128_lo(sb + C::kOffKV, C::kBoxBytes);
        // MMA kk of S covers bytes 32kk .. 32kk+31 of each 128-byte box row
        auto issue_S = [&](int X, int st) {
          if (!FA_DBG_OK(p.status, st < C::kStages && tmem_in(C::tm_s(X), 128))) return;
          const uint32_t a0 = lq0 + (uint32_t)X * kStageStep;
          const uint32_t b0 = lk0 + (uint32_t)st * kStageStep;
          const uint32_t d = tmem + C::tm_s(X);
#pragma unroll
          for (int kk = 0; kk < C::kSKSteps; ++kk) {
            constexpr uint32_t kBox16 = C::kBoxBytes >> 4;
            const uint32_t off = (uint32_t)(kk / C::kKPerBox) * kBox16 + (uint32_t)(kk % C::kKPerBox) * 2u;
            if constexpr (E == Elem::E4M3)
              mma_ss_lh_w_f8(d, a0 + off, kHi, b0 + off, kHi, idS, kk > 0 ? 1u : 0u);
            else
              mma_ss_lh_w(d, a0 + off, kHi, b0 + off, kHi, idS, kk > 0 ? 1u : 0u);
          }
        };
        // MMA kk of P V takes keys kPVKeys*kk .. (P in TMEM columns 8kk .. 8kk+7,
        // V rows from kPVKeys*kk on, 128 bytes each)
        auto issue_PV = [&](int X, int st, bool acc, int h) {   // keys 64h .. 64h+63
          constexpr int kPer = 64 / C::kPVKeys;
          constexpr uint32_t kVStep = (uint32_t)(C::kPVKeys * C::kSwz) >> 4;   // kPVKeys box rows
          if (!FA_DBG_OK(p.status, st < C::kStages && tmem_in(C::tm_o(X), D) &&
                                       tmem_in(C::tm_s(X), 2 * C::kPHalfCols)))
            return;
          const uint32_t b0 = lv0 + (uint32_t)st * kStageStep;
          const uint32_t d = tmem + C::tm_o(X);
          const uint32_t a = tmem + C::tm_s(X);
#pragma unroll
          for (int kk = kPer * h; kk < kPer * h + kPer; ++kk) {
            if constexpr (E == Elem::E4M3)
              mma_ts_lh_w_f8(d, a + (uint32_t)kk * 8u, b0 + (uint32_t)kk * kVStep, kHi, idO,
                             (acc || kk > 0) ? 1u : 0u);
            else
              mma_ts_lh_w(d, a + (uint32_t)kk * 8u, b0 + (uint32_t)kk * kVStep, kHi, idO,
                          (acc || kk > 0) ? 1u : 0u);
          }
        };
        bool ok = mbar_wait_w(bar(C::kBarQ), 0, s_abort, p.status);
        if (ok) ok = mbar_wait_w(bar(C::kBarFull + 0), 0, s_abort, p.status);
        if (ok) {
          tc_fence_after();
          if (n0 > 0) { issue_S(0, 0); mma_commit_w(bar(C::kBarS + 0)); }
          if (n1 > 0) { issue_S(1, 0); mma_commit_w(bar(C::kBarS + 1)); }
          release(0);
        }
        for (int j = 0; j < n_loop && ok; ++j) {
          const int itV = 2 * j + 1, itK = 2 * j + 2;
          const int stV = itV % C::kStages, stK = itK % C::kStages;
          const uint32_t phV = (uint32_t)(itV / C::kStages) & 1u;
          const uint32_t phK = (uint32_t)(itK / C::kStages) & 1u;
          const bool next = (j + 1) < n_loop;
          if (!(ok = mbar_wait_w(bar(C::kBarFull + stV), phV, s_abort, p.status))) break;
          tc_fence_after();
          if (j < n0) {
            if (!(ok = mbar_wait_w(bar(C::kBarP1 + 0), (uint32_t)j & 1u, s_abort, p.status))) break;
            tc_fence_after();
            issue_PV(0, stV, j > 0, 0);
            if (!(ok = mbar_wait_w(bar(C::kBarP2 + 0), (uint32_t)j & 1u, s_abort, p.status))) break;
            tc_fence_after();
            issue_PV(0, stV, true, 1);
          }
          if (next) {
            if (!(ok = mbar_wait_w(bar(C::kBarFull + stK), phK, s_abort, p.status))) break;
            tc_fence_after();
            if (j + 1 < n0) { issue_S(0, stK); mma_commit_w(bar(C::kBarS + 0)); }
          }
          if (j < n1) {
            if (!(ok = mbar_wait_w(bar(C::kBarP1 + 1), (uint32_t)j & 1u, s_abort, p.status))) break;
            tc_fence_after();
            issue_PV(1, stV, j > 0, 0);
            if (!(ok = mbar_wait_w(bar(C::kBarP2 + 1), (uint32_t)j & 1u, s_abort, p.status))) break;
            tc_fence_after();
            issue_PV(1, stV, true, 1);
          }
          release(stV);
          if (next) {
            if (j + 1 < n1) { issue_S(1, stK); mma_commit_w(bar(C::kBarS + 1)); }
            release(stK);
          }
        }
        mma_commit_w(bar(C::kBarO));
        // drain: all MMAs done before tensor memory is released
        mma_commit_w(bar(C::kBarDrain));
        drain_wait(bar(C::kBarDrain), 0, p.status);
      }
      __syncwarp();
    }
    // warps 10-11: idle members of warpgroup 2
    if (p.cm) {   // the two cluster barriers of the in-cluster merge
      cluster_sync();
      cluster_sync();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ======================= softmax warpgroups =======================
    const int X = warp >> 2;                // query tile
    const int quad = warp & 3;
    const int r = quad * 32 + lane;         // row within the query tile = TMEM lane
    const int row = q0 + X * kTileM + r;    // query row within the head
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::tm_s(X);
    const uint32_t tO = tmem + lane_base + C::tm_o(X);
    const int n = X ? n1 : n0;
    const float c = p.c;
    const int tile_first_row = q0 + X * kTileM;
    float m_ref = -INFINITY;  // reference max, scaled log2 units
    float l = 0.f;
    bool ok = true;

    // One tile of the key range (j).
    auto tile_step = [&](int j, auto mask_tag) -> bool {
      constexpr MaskMode kMask = decltype(mask_tag)::value;
      if (!(ok = mbar_wait(bar(C::kBarS + X), (uint32_t)j & 1u, s_abort, p.status))) return false;
      tc_fence_after();
      float s[kTileN];
      if (!FA_DBG_OK(p.status, tmem_in(lane_base + C::tm_s(X), kTileN) &&
                                   tmem_in(lane_base + C::tm_o(X), D))) {
        ok = false;   // FA_DEBUG: reported; this tile is not processed
        return false;
      }
      tmem_ld32(tS + 0, s);
      tmem_ld32(tS + 32, s + 32);
      tmem_ld32(tS + 64, s + 64);
      tmem_ld32(tS + 96, s + 96);
      tmem_wait_ld();
      const int key0 = (lo + j) * kTileN;
      // mask: ragged key tail, and keys after the causal diagonal
      if (kMask == MaskMode::kAlways ||
          (kMask == MaskMode::kCheck &&
           (key0 + kTileN > p.N_k || (p.causal && key0 + kTileN - 1 > tile_first_row + p.kv_off)))) {
        int lim = p.N_k - key0;
        if (p.causal) lim = min_i(lim, row + p.kv_off + 1 - key0);
#pragma unroll
        for (int i = 0; i < kTileN; ++i)
          if (i >= lim) s[i] = -INFINITY;
      }
      // warp-uniform: every row of the warp has a reference max
      const bool spec = !__any_sync(0xffffffffu, m_ref == -INFINITY);
      if (!spec) {
        // some row's first live tile: references from the tile max
        const float m_tile = max_scores<kTileN>(s) * c;
        const bool need = m_tile > m_ref + Lag<E>::kTau;   // always, for a row without a reference
        if (__any_sync(0xffffffffu, need)) {
          float alpha = 1.f;
          if (need) {
            alpha = ex2_approx(m_ref - m_tile);  // 0 when the row had no reference yet
            m_ref = m_tile;
            l *= alpha;
          }
          if (j > 0) rescale_o<D>(tO, alpha);   // O_X holds PV_X(0..j-1), stable (S_X(j) commit)
        }
      }
      // The first half's P against the reference (0 for a row that has none).
      // Both paths share this code and the second half's below: one copy of each
      // in the kernel keeps its main loop small.
      // On the later tiles the second half's max then decides any rescale, while
      // O_X is stable (S_X(j) commit); a rescale redoes the first half (the same
      // copy of the code, a second pass).
      float r1;
#pragma unroll 1
      for (int pass = 0;; ++pass) {
        r1 = exp_half<E>(s, c, m_ref == -INFINITY ? 0.f : m_ref, tS);
        if (!spec || pass > 0) break;
        const float m2 = max_scores<kTileN / 2>(s + 64) * c;
        const bool need = !(r1 <= Lag<E>::kSumCap) || m2 > m_ref + Lag<E>::kTau;
        if (!__any_sync(0xffffffffu, need)) break;
        float alpha = 1.f;
        if (need) {
          const float m_new = fmaxf(m_ref, fmaxf(max_scores<kTileN / 2>(s) * c, m2));
          alpha = ex2_approx(m_ref - m_new);
          m_ref = m_new;
          l *= alpha;
        }
        rescale_o<D>(tO, alpha);
      }
      publish(bar(C::kBarP1 + X));
      // the second half's P <= 2^kTau now
      const float r2 = exp_half<E>(s + 64, c, m_ref == -INFINITY ? 0.f : m_ref, tS + C::kPHalfCols);
      publish(bar(C::kBarP2 + X));
      l += r1 + r2;
      return true;
    };
    auto masked_at = [&](int j) {
      const int key0 = (lo + j) * kTileN;
      return key0 + kTileN > p.N_k || (p.causal && key0 + kTileN - 1 > tile_first_row + p.kv_off);
    };
    if constexpr (E == Elem::E4M3) {
      // FP8 (bound by this loop): tiles that need a mask only come at the end of
      // a range, so they run in a second loop with its own copy of the step and
      // the main loop's copy has no mask code (1558 -> 1699 TFLOP/s at 32 heads x
      // 4096; the same split made the BF16 kernel 1-2.5 % slower)
      int j = 0;
      for (; j < n && !masked_at(j); ++j)
        if (!tile_step(j, MaskTag<MaskMode::kNone>{})) break;
      if (ok)
        for (; j < n; ++j)
          if (!tile_step(j, MaskTag<MaskMode::kAlways>{})) break;
    } else {
      for (int j = 0; j < n; ++j)
        if (!tile_step(j, MaskTag<MaskMode::kCheck>{})) break;
    }
    if (ok && n_loop > 0) {
      ok = mbar_wait(bar(C::kBarO), 0, s_abort, p.status);
      tc_fence_after();
    }
    // global writes only after the previous kernel on the stream has finished
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const bool valid_row = row < p.N_q;
    if (p.cm) {
      // every CTA of the cluster has finished its key range once all its
      // threads pass the first cluster barrier: the Q tiles and the K/V ring
      // are free and receive the partials (warpgroup 2 takes the same barriers)
      cluster_sync();
      // FA_DEBUG: the receive slots ([sender][16-byte chunk][row], S senders x
      // 256 / S rows each) span exactly [0, kCmStage) for S in {2, 4, 8}
      if (FA_DBG_OK(p.status, ui.split < p.s_tail && (p.s_tail == 2 || p.s_tail == 4 || p.s_tail == 8)))
        cm_send<D>(sb + C::kOffQ, sb + C::kOffCm, p.s_tail, ui.split, X * kTileM + r, tO, n, m_ref, l);
      cluster_sync();   // all partials of this CTA's rows have landed
      {
        const uint32_t rb = sb + C::kOffQ, mb2 = sb + C::kOffCm, stg = sb + C::kOffQ + C::kCmStage;
        const float os = p.o_scale;
        if (p.s_tail == 2) cm_reduce<D, 2, E>(rb, mb2, stg, ui.split, warp, lane, ok, p, &tmO, bh, q0, os);
        else if (p.s_tail == 4) cm_reduce<D, 4, E>(rb, mb2, stg, ui.split, warp, lane, ok, p, &tmO, bh, q0, os);
        else cm_reduce<D, 8, E>(rb, mb2, stg, ui.split, warp, lane, ok, p, &tmO, bh, q0, os);
      }
    } else if (slot < 0) {
      // ---- final epilogue: O / l -> BF16 into this tile's Q slot (128-byte
      // swizzled boxes, the tensor map's layout), then one TMA store; LSE direct
      // (FP8 inputs: the BF16 O tile is twice a Q tile, staged in the idle K/V ring)
      const uint32_t obase = E == Elem::E4M3 ? sb + C::kOffKV + X * C::kOTileBytes
                                             : sb + C::kOffQ + X * C::kTileBytes;
      constexpr Elem OE = kOutElem<E>;
      if (ok && !FA_DBG_OK(p.status, smem_in(obase, C::kOBoxes * C::kStgBoxBytes, sb, s_hi) && bh < p.n_bh))
        ok = false;   // FA_DEBUG: reported; nothing stored
      if (ok) {
        const float inv = l > 0.f ? p.o_scale / l : 0.f;
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
          const uint32_t rowaddr = obase + (uint32_t)(cc >> 6) * C::kStgBoxBytes + (uint32_t)r * 128u;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t ch = (uint32_t)(((cc & 63) >> 3) + g);   // 16-byte chunk in the row
            st_shared_v4(rowaddr + ((ch ^ (uint32_t)(r & 7)) << 4),
                         pack2<OE>(ov[8 * g + 0] * inv, ov[8 * g + 1] * inv),
                         pack2<OE>(ov[8 * g + 2] * inv, ov[8 * g + 3] * inv),
                         pack2<OE>(ov[8 * g + 4] * inv, ov[8 * g + 5] * inv),
                         pack2<OE>(ov[8 * g + 6] * inv, ov[8 * g + 7] * inv));
          }
        }
        if (valid_row && p.lse)
          p.lse[(size_t)bh * p.N_q + row] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      }
      fence_proxy_async_smem();
      const bool all_ok = named_bar_and(1 + X, 128, ok);
      if (all_ok && r == 0 && tile_first_row < p.N_q) {   // rows past N_q are clipped by the TMA
#pragma unroll
        for (int bx = 0; bx < C::kOBoxes; ++bx)
          tma_store_3d(&tmO, obase + bx * C::kStgBoxBytes, bx * 64, tile_first_row, bh);
        bulk_commit();
        bulk_wait_read0();
      }
    } else {
      // ---- partial: unnormalised O (FP32, 32-column swizzled boxes staged in the
      // K/V ring, one TMA store) and (m, l) of this key range to the workspace
      const uint32_t pbase = sb + C::kOffKV + X * C::kPartTileBytes;
      const int prow0 = slot * kBlockRows + X * kTileM;
      if (ok && !FA_DBG_OK(p.status, smem_in(pbase, C::kPartTileBytes, sb + C::kOffKV, sb + C::kOffBar) &&
                                         slot >= 0 && slot < p.n_tail * p.s_tail))
        ok = false;   // FA_DEBUG: reported; nothing stored
      if (ok) {
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
          const uint32_t rowaddr = pbase + (uint32_t)(cc >> 5) * C::kStgBoxBytes + (uint32_t)r * 128u;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            st_shared_v4(rowaddr + (((uint32_t)g ^ (uint32_t)(r & 7)) << 4), __float_as_uint(ov[4 * g]),
                         __float_as_uint(ov[4 * g + 1]), __float_as_uint(ov[4 * g + 2]),
                         __float_as_uint(ov[4 * g + 3]));
        }
        __stcg(reinterpret_cast<float2*>(p.part_ml) + prow0 + r,
               make_float2(l > 0.f ? m_ref : -INFINITY, l));
      }
      fence_proxy_async_smem();
      const bool all_ok = named_bar_and(1 + X, 128, ok);
      if (all_ok && r == 0) {
#pragma unroll
        for (int bx = 0; bx < D / 32; ++bx) tma_store_2d(&tmP, pbase + bx * C::kStgBoxBytes, bx * 32, prow0);
        bulk_commit();
        bulk_wait_read0();
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  // neither CTA of a cluster exits while the other may still multicast into its
  // shared memory or arrive on its barriers
  if (MC) cluster_sync();
}

// Merge of the split-key partials (the online-softmax merge of page 2, "The
// Tiling Algorithm", applied to whole key ranges): for each query row of a
// split block, M = max_s m_s, L = sum_s 2^(m_s - M) l_s, O = sum_s 2^(m_s - M)
// O_s / L, LSE = (M + log2 L) ln 2. One warp per row, lanes across columns.
// Launched as a programmatic dependent of fa_fwd_kernel: it may be resident
// early and waits (griddepcontrol.wait) until that grid has completed.
template <int D, Elem E>
__global__ void __launch_bounds__(256) fa_merge_kernel(const FwdParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kCols = D / 32;  // columns per lane
  const int lane = threadIdx.x & 31;
  const long long wrow = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int t = (int)(wrow / kBlockRows);
  const int r = (int)(wrow % kBlockRows);
  if (t >= p.n_tail) return;
  int bh, qb;
  block_of(p, p.u_full + t, bh, qb);
  const int row = qb * kBlockRows + r;
  if (row >= p.N_q) return;
  const int S = p.s_tail;
  const size_t base = (size_t)t * S * kBlockRows + r;  // partial row of split 0
  // every load of the row is independent: issue them all, then combine
  constexpr int kMaxS = 16;
  float4 va[kMaxS];
#pragma unroll
  for (int s2 = 0; s2 < kMaxS; ++s2) {
    va[s2] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (s2 < S) {
      const float* src = p.part_o + (base + (size_t)s2 * kBlockRows) * D + lane * kCols;
      if constexpr (kCols == 4) {
        va[s2] = __ldcg(reinterpret_cast<const float4*>(src));
      } else {
        const float2 t2 = __ldcg(reinterpret_cast<const float2*>(src));
        va[s2] = make_float4(t2.x, t2.y, 0.f, 0.f);
      }
    }
  }
  float m = -INFINITY, l = 0.f;
  if (lane < S) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + base + (size_t)lane * kBlockRows);
    if (ml.y > 0.f) {
      m = ml.x;
      l = ml.y;
    }
  }
  float M = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float w = (l > 0.f) ? ex2_approx(m - M) : 0.f;
  float L = w * l;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const float inv = L > 0.f ? p.o_scale / L : 0.f;
  float acc[kCols];
#pragma unroll
  for (int i = 0; i < kCols; ++i) acc[i] = 0.f;
#pragma unroll
  for (int s2 = 0; s2 < kMaxS; ++s2) {
    const float ws = __shfl_sync(0xffffffffu, w, s2) * inv;   // 0 for s2 >= S
    acc[0] += ws * va[s2].x;
    acc[1] += ws * va[s2].y;
    if constexpr (kCols == 4) {
      acc[2] += ws * va[s2].z;
      acc[3] += ws * va[s2].w;
    }
  }
  uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + ((size_t)bh * p.N_q + row) * D;   // 16-bit elements
  constexpr Elem OE = kOutElem<E>;
  if constexpr (kCols == 4) {
    uint2 v;
    v.x = pack2<OE>(acc[0], acc[1]);
    v.y = pack2<OE>(acc[2], acc[3]);
    *reinterpret_cast<uint2*>(orow + lane * 4) = v;
  } else {
    *reinterpret_cast<uint32_t*>(orow + lane * 2) = pack2<OE>(acc[0], acc[1]);
  }
  if (lane == 0 && p.lse) p.lse[(size_t)bh * p.N_q + row] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
}

// Opt in to the kernel's dynamic shared memory (once per device and kernel).
template <int D, bool MC, Elem E>
cudaError_t ensure_smem_attr() {
  static bool attr[64] = {false};  // benign race: setting the attribute twice is harmless
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (attr[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, MC, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<D, E>::kSmemBytes);
  if (e == cudaSuccess) attr[dev] = true;
  return e;
}

template <int D>
int cluster_capacity_t(int s) {
  if (ensure_smem_attr<D, false, Elem::BF16>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)s);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D, Elem::BF16>::kSmemBytes;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)s;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  // the FP16 and FP8 kernels also run one CTA per SM: one answer serves all three
  if (cudaOccupancyMaxActiveClusters(&n, fa_fwd_kernel<D, false, Elem::BF16>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int D, bool MC, Elem E>
cudaError_t launch_main_t(const FwdMaps& m, const FwdParams& p, int units, cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr<D, MC, E>();
  if (e != cudaSuccess) return e;
  // programmatic launch: set-up may overlap the previous kernel on the stream
  // (the kernel waits for it before its first global read and write)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(MC ? ((units + 1) & ~1) : units));   // MC: whole clusters of two
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D, E>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = MC ? 2 : (p.cm ? p.s_tail : 1);   // pairs, or the S splits of a block
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = (MC || p.cm) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fa_fwd_kernel<D, MC, E>, m.q, m.k, m.v, m.o, m.part, p);
}

}  // namespace
}  // namespace fa
