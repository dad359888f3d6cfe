// Decode / few-query attention forward for sm_103a ("FlashAttention HBM bytes,
// one head, 8K", "What interviewers probe next": one query against many keys
// is bandwidth-bound — K and V are read once per KV head — and "Why is
// standard attention memory-bound...", "Does FlashAttention help when
// generating one token at a time?": split the key sequence across thread
// blocks and combine).
//
// Work unit = (batch, KV head, run of cpc consecutive chunks of 128 keys). The
// rows of a unit are all query rows that read this KV head: R = G * N_q <= 16
// (G = H_q / H_kv, GQA), which is exactly the M = 16 of one mma.sync m16n8k16 —
// the contraction is a real (16 x d) x (d x keys) product, tiny next to the K/V
// stream it rides on.
//   * one thread issues the TMA loads (K tile, V tile; 128-byte swizzle) into
//     shared memory on two mbarriers, the next chunk's K as soon as every warp
//     has used the current one (overlapping this chunk's PV), its V after PV;
//     64 KB per CTA at d = 128 lets three CTAs share an SM;
//   * each of the 4 warps takes 32 keys of every chunk: S = Q K^T (Q fragments
//     from global, K fragments by ldmatrix), the online softmax over its keys
//     across the unit's chunks (running max and sum, exact rescale of its
//     accumulator in registers), P kept in registers as the A operand of
//     O += P V (V fragments by ldmatrix.trans);
//   * the 4 warps' (m, l, O) are merged in shared memory into one partial per
//     (row, unit); fa_decode_merge_kernel merges the units of each row.
// The kernel is bound by HBM bandwidth: algorithmic bytes are K and V once per
// KV head, Q read and O, LSE written once.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {

namespace {

constexpr int kDecThreads = 128;
constexpr int kDecKeys = 128;   // keys per chunk (one CTA)
constexpr float kLn2d = 0.6931471805599453f;

template <int D>
struct DecCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = kDecKeys * 128;          // 128 keys x 128 bytes
  static constexpr int kTileBytes = kDecKeys * D * 2;       // K or V chunk
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  // [4 warps][16 rows][2] f32 (m, l); later [16][8] merge weights + [16][2] (M, L)
  static constexpr int kMlFloats = 16 * 8 + 16 * 2;
  static constexpr int kOffMl = 2 * kTileBytes;
  static constexpr int kOffBar = kOffMl + kMlFloats * 4;
  static_assert(4 * 16 * 2 <= kMlFloats, "the warps' (m, l) must fit");
  static_assert(16 * D * 4 + 16 * 2 * 4 <= kTileBytes, "a CTA's partial must fit in the V tile");
  static constexpr int kSmemBytes = kOffBar + 16 + 1024;
  // merge buffer [4 warps][16 rows][D] f32 reuses the K tile (dead after S = Q K^T)
  static_assert(4 * 16 * D * 4 <= kTileBytes, "merge buffer must fit in the K tile");
};

// D (16 x 8, FP32) += A (16 x 16) B (16 x 8), A and B both BF16 or both FP16.
template <Elem E>
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (E == Elem::F16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Byte address of element row `key`, 16-byte chunk `ch16` (of d) in a TMA tile
// stored as 64-column boxes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_addr(uint32_t base, int key, int ch16) {
  const int box = ch16 >> 3, ch = ch16 & 7;
  return base + (uint32_t)(box * (kDecKeys * 128) + key * 128 + ((ch ^ (key & 7)) << 4));
}

template <int D, Elem E>
__global__ void __launch_bounds__(kDecThreads)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const DecParams p) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t barK = sb + C::kOffBar, barV = sb + C::kOffBar + 8;
  volatile int abort_flag = 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int part = blockIdx.x % p.n_parts;
  const int bhk = blockIdx.x / p.n_parts;
  const int b = bhk / p.H_kv, hk = bhk - b * p.H_kv;
  const int c_begin = part * p.cpc;
  // keys of this sequence (paged K/V: each sequence has its own length)
  int n_k = p.N_k, kv_off = p.kv_off, n_chunks = p.n_chunks;
  if (p.paged) {
    n_k = min(max(__ldg(p.seqlens + b), 0), p.max_pages * kDecKeys);
    kv_off = n_k - p.N_q;
    n_chunks = (n_k + kDecKeys - 1) / kDecKeys;
  }
  // chunks of this run; 0 only for a paged sequence shorter than the run's start
  const int nc = max(0, min(n_chunks, c_begin + p.cpc) - c_begin);

  if (threadIdx.x == 0) {
    mbar_init(barK, 1);
    mbar_init(barV, 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto load = [&](uint32_t bar, uint32_t off, const CUtensorMap* tm, int chunk) {
    mbar_arrive_expect_tx(bar, C::kTileBytes);
    // contiguous: rows chunk*128.. of (batch, KV head) slab bhk; paged: the
    // whole 128-row slab (page, KV head) (an index outside the cache reads zeros)
    int row = chunk * kDecKeys, slab = bhk;
    if (p.paged) {
      row = 0;
      slab = __ldg(p.block_table + (size_t)b * p.max_pages + chunk) * p.H_kv + hk;
    }
#pragma unroll
    for (int bx = 0; bx < C::kBoxes; ++bx)
      tma_load_3d(sb + off + bx * C::kBoxBytes, tm, bar, bx * 64, row, slab);
  };
  if (threadIdx.x == 0 && nc > 0) {
    load(barK, C::kOffK, &tmK, c_begin);
    load(barV, C::kOffV, &tmV, c_begin);
  }

  // Q fragments (A operand, rows = the R query rows of this KV head, zero-padded to 16)
  uint32_t qa[D / 16][4];
  {
    const int rows[2] = {g, g + 8};
    const uint32_t* qrow[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int m = rows[u];
      if (m < p.R) {
        const int hl = m / p.N_q, i = m - hl * p.N_q;
        const int hq = hk * p.G + hl;
        qrow[u] = reinterpret_cast<const uint32_t*>(p.q + (((size_t)b * p.H_q + hq) * p.N_q + i) * D);
      } else {
        qrow[u] = nullptr;
      }
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qa[ks][0] = qrow[0] ? __ldg(qrow[0] + ks * 8 + t) : 0u;
      qa[ks][1] = qrow[1] ? __ldg(qrow[1] + ks * 8 + t) : 0u;
      qa[ks][2] = qrow[0] ? __ldg(qrow[0] + ks * 8 + 4 + t) : 0u;
      qa[ks][3] = qrow[1] ? __ldg(qrow[1] + ks * 8 + 4 + t) : 0u;
    }
  }

  const int kw = warp * 32;  // this warp's 32 keys within each chunk
  const float c = p.c;
  // running (m, l) of rows g and g + 8 over this warp's keys (m in scaled log2 units)
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  float oacc[D / 8][4];
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[dn][e] = 0.f;
  int k_loads = nc > 0 ? 1 : 0, v_loads = k_loads;   // loads issued (thread 0), for the drain on failure
  bool ok = true;
  for (int ci = 0; ci < nc; ++ci) {
    const int key0 = (c_begin + ci) * kDecKeys;
    const uint32_t ph = (uint32_t)ci & 1u;
    // ---- S = Q K^T for 32 keys: 4 n-tiles of 8 keys
    const bool okK = mbar_wait(barK, ph, &abort_flag, p.status);
    float sacc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
    if (okK) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < 2; ++np) {   // pairs of n-tiles
          const int i = lane >> 3, rr = lane & 7;
          const int key = kw + 16 * np + 8 * (i >> 1) + rr;
          uint32_t b00, b01, b10, b11;
          ldsm_x4(sw128_addr(sb + C::kOffK, key, 2 * ks + (i & 1)), b00, b01, b10, b11);
          mma16816<E>(sacc[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
          mma16816<E>(sacc[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
        }
      }
    }
    // every warp is done with this K tile: the next chunk's may load (uniform ok)
    ok = __syncthreads_and(okK) != 0;
    if (!ok) break;
    if (threadIdx.x == 0 && ci + 1 < nc) {
      load(barK, C::kOffK, &tmK, c_begin + ci + 1);
      ++k_loads;
    }
    // ---- online softmax over this warp's 32 keys, rows g and g + 8
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int m = g + 8 * u;
      const int i = (m < p.R) ? m % p.N_q : 0;
      int lim = n_k - key0;                                    // keys of this chunk that exist
      if (p.causal) lim = min(lim, i + kv_off + 1 - key0);     // ... and that row i may see
      if (m >= p.R) lim = 0;
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = kw + 8 * nt + 2 * t + e;
          float& sv = sacc[nt][2 * u + e];
          if (key >= lim) sv = -INFINITY;
          mx = fmaxf(mx, sv);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(mrow[u], mx == -INFINITY ? -INFINITY : mx * c);
      // nothing seen yet: nothing to rescale; otherwise 2^(m_old - m_new) (0 from -inf)
      const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(mrow[u] - m_new);
      const float mb = (m_new == -INFINITY) ? 0.f : m_new;
      float l = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float& sv = sacc[nt][2 * u + e];
          sv = ex2_approx(fmaf(sv, c, -mb));
          l += sv;
        }
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      lrow[u] = lrow[u] * alpha + l;
      mrow[u] = m_new;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        oacc[dn][2 * u] *= alpha;
        oacc[dn][2 * u + 1] *= alpha;
      }
    }
    // P as the A operand of O = P V: k-step j covers keys kw + 16j .. kw + 16j + 15
    uint32_t pa[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      pa[j][0] = pack2<E>(sacc[2 * j][0], sacc[2 * j][1]);
      pa[j][1] = pack2<E>(sacc[2 * j][2], sacc[2 * j][3]);
      pa[j][2] = pack2<E>(sacc[2 * j + 1][0], sacc[2 * j + 1][1]);
      pa[j][3] = pack2<E>(sacc[2 * j + 1][2], sacc[2 * j + 1][3]);
    }
    // ---- O += P V: D/8 n-tiles of 8 columns
    const bool okV = mbar_wait(barV, ph, &abort_flag, p.status);
    if (okV) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {   // pairs of d n-tiles
          const int i = lane >> 3, rr = lane & 7;
          const int key = kw + 16 * j + 8 * (i & 1) + rr;
          uint32_t b00, b01, b10, b11;
          ldsm_x4_t(sw128_addr(sb + C::kOffV, key, 2 * dp + (i >> 1)), b00, b01, b10, b11);
          mma16816<E>(oacc[2 * dp], pa[j][0], pa[j][1], pa[j][2], pa[j][3], b00, b01);
          mma16816<E>(oacc[2 * dp + 1], pa[j][0], pa[j][1], pa[j][2], pa[j][3], b10, b11);
        }
      }
    }
    // every warp is done with this V tile: the next chunk's may load
    ok = __syncthreads_and(okV) != 0;
    if (!ok) break;
    if (threadIdx.x == 0 && ci + 1 < nc) {
      load(barV, C::kOffV, &tmV, c_begin + ci + 1);
      ++v_loads;
    }
  }
  if (!ok && threadIdx.x == 0) {
    // a wait gave up: let every load issued land (bounded) before the CTA exits
    volatile int never = 0;
    mbar_wait(barK, (uint32_t)(k_loads - 1) & 1u, &never, p.status);
    mbar_wait(barV, (uint32_t)(v_loads - 1) & 1u, &never, p.status);
  }

  // ---- merge the 4 warps' partials in shared memory (the K tile is dead now)
  __syncthreads();
  float* mo = reinterpret_cast<float*>(smem + C::kOffK);   // [4][16][D]
  float* mml = reinterpret_cast<float*>(smem + C::kOffMl); // [4][16][2]
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int m = g + 8 * u;
    float* dst = mo + ((size_t)warp * 16 + m) * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn)
      *reinterpret_cast<float2*>(dst + 8 * dn + 2 * t) = make_float2(oacc[dn][2 * u], oacc[dn][2 * u + 1]);
    if (t == 0) {
      mml[(warp * 16 + m) * 2 + 0] = mrow[u];
      mml[(warp * 16 + m) * 2 + 1] = lrow[u];
    }
  }
  __syncthreads();
  // each partial row: M = max_w m_w, L = sum_w 2^(m_w - M) l_w, O = sum_w 2^(m_w - M) O_w
  const size_t pbase = ((size_t)bhk * p.n_parts + part) * p.R;
  // this CTA's combined partial, kept in shared memory for the in-cluster merge
  // (the V tile is dead after the last PV): [16][D] O, then [16][2] (m, l)
  float* cpo = reinterpret_cast<float*>(smem + C::kOffV);
  float* cml = cpo + 16 * D;
  for (int idx = threadIdx.x; idx < p.R * D; idx += kDecThreads) {
    const int m = idx / D, dcol = idx - m * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w)
      if (mml[(w * 16 + m) * 2 + 1] > 0.f) M = fmaxf(M, mml[(w * 16 + m) * 2]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float lw = mml[(w * 16 + m) * 2 + 1];
      if (lw > 0.f) {
        const float wt = ex2_approx(mml[(w * 16 + m) * 2] - M);
        L += wt * lw;
        acc += wt * mo[((size_t)w * 16 + m) * D + dcol];
      }
    }
    if (p.cm) {
      cpo[m * D + dcol] = acc;
      if (dcol == 0) {
        cml[2 * m] = L > 0.f ? M : -INFINITY;
        cml[2 * m + 1] = L;
      }
    } else if (FA_DBG_OK(p.status, (size_t)pbase + m < (size_t)p.B * p.H_kv * p.n_parts * p.R && dcol < D)) {
      __stcg(p.part_o + (pbase + m) * D + dcol, acc);
      if (dcol == 0)
        __stcg(reinterpret_cast<float2*>(p.part_ml) + pbase + m, make_float2(L > 0.f ? M : -INFINITY, L));
    }
  }
  if (!p.cm) return;

  // ---- in-cluster merge: the n_parts CTAs of this KV head form one cluster
  // (rank = part); rank 0 combines the parts' partials from their shared memory
  // and writes O and LSE (page 2, "The Tiling Algorithm", applied to whole runs)
  cluster_sync();   // every part's partial is in its shared memory
  if (part == 0) {
    float* sw = mml;   // [16 rows][8 parts] weights 2^(m_p - M) / L (the warps' (m, l) are dead)
    float* sML = mml + 16 * 8;   // [16][2] (M, L) per row
    if (threadIdx.x < p.R) {
      const int m = threadIdx.x;
      float mp[8], lp[8];
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < 8; ++q) {   // all remote loads in flight at once
        mp[q] = -INFINITY;
        lp[q] = 0.f;
        if (q < p.n_parts) {
          const float2 v = ld_cluster_v2f(mapa_shared(smem_u32(cml + 2 * m), (uint32_t)q));
          mp[q] = v.x;
          lp[q] = v.y;
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (lp[q] > 0.f) M = fmaxf(M, mp[q]);
      float L = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float w = lp[q] > 0.f ? ex2_approx(mp[q] - M) : 0.f;
        mp[q] = w;
        L += w * lp[q];
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) sw[m * 8 + q] = mp[q] * inv;
      sML[2 * m] = M;
      sML[2 * m + 1] = L;
    }
    __syncthreads();
    // four consecutive columns per thread, one float4 from every part in flight at once
    for (int idx = threadIdx.x * 4; idx < p.R * D; idx += kDecThreads * 4) {
      const int m = idx / D, dcol = idx - m * D;
      float4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = q < p.n_parts ? ld_cluster_v4f(mapa_shared(smem_u32(cpo + m * D + dcol), (uint32_t)q))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float w = sw[m * 8 + q];   // 0 for q >= n_parts
        acc.x += w * v[q].x; acc.y += w * v[q].y; acc.z += w * v[q].z; acc.w += w * v[q].w;
      }
      const int hl = m / p.N_q, i = m - hl * p.N_q;
      const int hq = hk * p.G + hl;
      const size_t orow = ((size_t)b * p.H_q + hq) * p.N_q + i;
      if (!FA_DBG_OK(p.status, orow < (size_t)p.B * p.H_q * p.N_q && dcol + 4 <= D)) continue;
      uint2 o2;
      o2.x = pack2<E>(acc.x, acc.y);
      o2.y = pack2<E>(acc.z, acc.w);
      *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.o) + orow * D + dcol) = o2;
      if (dcol == 0 && p.lse) {
        const float L = sML[2 * m + 1];
        p.lse[orow] = L > 0.f ? (sML[2 * m] + __log2f(L)) * kLn2d : -INFINITY;
      }
    }
  }
  cluster_sync();   // rank 0 has read every part's shared memory
}

// Merge of the chunk partials of each query row (same algebra as the prefill
// merge). One CTA of D threads per row: the (m, l) of every chunk are turned
// into weights 2^(m_c - M) / L once, in shared memory; then thread t sums
// column t over the chunks with independent, coalesced loads.
constexpr int kMergeMaxChunks = 1024;   // chunks merged per pass (longer rows loop)

template <int D, Elem E>
__global__ void __launch_bounds__(D) fa_decode_merge_kernel(const DecParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float s_w[kMergeMaxChunks];
  __shared__ float s_red[D / 32];
  __shared__ float s_ML[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long wrow = blockIdx.x;
  const int bhk = (int)(wrow / p.R), m = (int)(wrow % p.R);
  const int b = bhk / p.H_kv, hk = bhk - b * p.H_kv;
  const int hl = m / p.N_q, i = m - hl * p.N_q;
  const int hq = hk * p.G + hl;
  const size_t stride = (size_t)p.R;                     // between chunks of one row
  const size_t base = (size_t)bhk * p.n_parts * p.R + m;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  // pass 1: M = max over chunks with l > 0
  float M = -INFINITY;
  for (int ch = tid; ch < p.n_parts; ch += D) {
    const float2 v = __ldcg(ml + base + ch * stride);
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) s_red[warp] = M;
  __syncthreads();
  if (tid == 0) {
    float mm = s_red[0];
    for (int w = 1; w < D / 32; ++w) mm = fmaxf(mm, s_red[w]);
    s_ML[0] = mm;
  }
  __syncthreads();
  M = s_ML[0];
  float acc = 0.f, Lpart = 0.f;
  const float* src = p.part_o + base * D + tid;
  for (int c0 = 0; c0 < p.n_parts; c0 += kMergeMaxChunks) {
    const int nc = min(kMergeMaxChunks, p.n_parts - c0);
    // pass 2: unnormalised weights of this group of chunks
    for (int ch = tid; ch < nc; ch += D) {
      const float2 v = __ldcg(ml + base + (size_t)(c0 + ch) * stride);
      const float w = (v.y > 0.f) ? ex2_approx(v.x - M) : 0.f;
      s_w[ch] = w;
      Lpart += w * v.y;
    }
    __syncthreads();
    // pass 3: column tid; 32 independent loads in flight per step
#pragma unroll 1
    for (int g0 = 0; g0 < nc; g0 += 32) {
      float v[32];
#pragma unroll
      for (int u = 0; u < 32; ++u)
        v[u] = (g0 + u < nc) ? __ldcg(src + (size_t)(c0 + g0 + u) * stride * D) : 0.f;
#pragma unroll
      for (int u = 0; u < 32; ++u)
        if (g0 + u < nc) acc += s_w[g0 + u] * v[u];
    }
    __syncthreads();
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Lpart += __shfl_xor_sync(0xffffffffu, Lpart, off);
  if (lane == 0) s_red[warp] = Lpart;
  __syncthreads();
  if (tid == 0) {
    float L = 0.f;
    for (int w = 0; w < D / 32; ++w) L += s_red[w];
    s_ML[1] = L;
  }
  __syncthreads();
  const float L = s_ML[1];
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + (((size_t)b * p.H_q + hq) * p.N_q + i) * D;
  orow[tid] = (uint16_t)(pack2<E>(acc * inv, 0.f) & 0xFFFFu);
  if (tid == 0 && p.lse)
    p.lse[((size_t)b * p.H_q + hq) * p.N_q + i] = L > 0.f ? (M + __log2f(L)) * kLn2d : -INFINITY;
}

template <int D, Elem E>
cudaError_t launch_decode_t(const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p,
                            cudaStream_t stream) {
  using C = DecCfg<D>;
  static bool attr[64] = {false};   // per device; a repeated set is harmless
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fa_decode_kernel<D, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  const long long ctas = (long long)p.B * p.H_kv * p.n_parts;
  cudaError_t e;
  if (p.cm && p.n_parts > 1) {
    // the parts of one KV head run as one cluster and merge in the kernel
    cudaLaunchConfig_t kc{};
    kc.gridDim = dim3((unsigned)ctas);
    kc.blockDim = dim3(kDecThreads);
    kc.dynamicSmemBytes = C::kSmemBytes;
    kc.stream = stream;
    cudaLaunchAttribute ka[1];
    ka[0].id = cudaLaunchAttributeClusterDimension;
    ka[0].val.clusterDim.x = (unsigned)p.n_parts;
    ka[0].val.clusterDim.y = 1;
    ka[0].val.clusterDim.z = 1;
    kc.attrs = ka;
    kc.numAttrs = 1;
    e = cudaLaunchKernelEx(&kc, fa_decode_kernel<D, E>, tk, tv, p);
  } else {
    e = launch_kernel(fa_decode_kernel<D, E>, dim3((unsigned)ctas), dim3(kDecThreads), C::kSmemBytes,
                      stream, tk, tv, p);
  }
  if (e != cudaSuccess || p.cm) return e;
  const long long rows = (long long)p.B * p.H_kv * p.R;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)rows);
  cfg.blockDim = dim3(D);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_decode_merge_kernel<D, E>, p);
}

}  // namespace

size_t decode_part_bytes(int B, int H_kv, int R, int n_parts, int d) {
  return (size_t)B * H_kv * n_parts * R * ((size_t)d * 4 + 8);
}

// (the FP16 kernel has the same resources: one answer serves both)
template <int D>
int decode_cluster_capacity_t(int parts) {
  using C = DecCfg<D>;
  if (cudaFuncSetAttribute(fa_decode_kernel<D, Elem::BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)parts);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)parts;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fa_decode_kernel<D, Elem::BF16>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

DecPlan decode_plan(long long heads, int n_chunks, int d, int sms, bool cluster_merge) {
  DecPlan pl{};
  // in-cluster merge: about 1.7 CTAs per SM in a single wave, i.e. parts per KV
  // head = 1.7 SMs / heads rounded, at least 1 and at most the head's chunks.
  // Measured on GB300 at batch 16 x 8 KV heads x 8192 keys (128 KV heads): 2
  // parts (256 CTAs) 6626 GB/s, 3: 6514, 5: 6255, 8 (two and a quarter waves of
  // three CTAs per SM): 5956, 1 (fewer CTAs than SMs): 5776. A wave that stays
  // resident to the end keeps HBM busiest; a partial last wave leaves it idle.
  // More than 8 parts would exceed a portable cluster: with few KV heads and
  // long keys the runs are merged by the merge kernel instead (below), unless a
  // head has at most 8 chunks (one part each; the GPU cannot be filled anyway).
  // One part needs no merge at all.
  if (cluster_merge) {
    const long long want = (17ll * sms + 5 * heads) / (10 * heads);   // round(1.7 sms / heads)
    int parts = 0;
    if (want <= 8) parts = (int)(want < 1 ? 1 : (want > n_chunks ? n_chunks : want));
    else if (n_chunks <= 8) parts = n_chunks;
    if (parts > 0) {
      const int cpc = (n_chunks + parts - 1) / parts;
      const int np = (n_chunks + cpc - 1) / cpc;
      if (np == 1 ||
          (d == 128 ? decode_cluster_capacity_t<128>(np) : decode_cluster_capacity_t<64>(np)) > 0) {
        pl.cpc = cpc;
        pl.n_parts = np;
        pl.cm = 1;
        return pl;
      }
    }
  }
  // otherwise (merge kernel): runs sized so that the whole grid is again about
  // 1.7 CTAs per SM in one wave. Measured on GB300 at 1 x 32 / 8 heads x 131072
  // keys (8 KV heads, 1024 chunks, 537 MB): runs of 32 chunks (256 CTAs) 6313
  // GB/s, of 64 (128 CTAs) 5507, of 16 (512) 5325, of 8 (1024) 5382, of 4 (2048,
  // the earlier four-wave rule) 4840.
  const long long want = (17ll * sms + 5 * heads) / (10 * heads);   // parts per head, rounded
  const long long parts = want < 1 ? 1 : (want > n_chunks ? n_chunks : want);
  const int cpc = (int)((n_chunks + parts - 1) / parts);
  pl.cpc = cpc;
  pl.n_parts = (n_chunks + cpc - 1) / cpc;
  pl.cm = pl.n_parts == 1 ? 1 : 0;
  return pl;
}

cudaError_t launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p,
                          cudaStream_t stream) {
  if ((long long)p.B * p.H_kv * p.n_parts <= 0) return cudaSuccess;
  if (p.elem == (int)Elem::F16)
    return d == 128 ? launch_decode_t<128, Elem::F16>(tk, tv, p, stream)
                    : launch_decode_t<64, Elem::F16>(tk, tv, p, stream);
  return d == 128 ? launch_decode_t<128, Elem::BF16>(tk, tv, p, stream)
                  : launch_decode_t<64, Elem::BF16>(tk, tv, p, stream);
}

}  // namespace fa
