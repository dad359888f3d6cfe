// Cluster-multicast operations of the paired-load forward variant. Built only
// into the single-GPU library (libfa_single_gpu.so): every tile these copy
// comes from the current GPU's own memory (the entry point rejects any other
// pointer), and the library refuses to run inside a multi-process job.
#pragma once

#include <cstdint>

namespace fa {

template <bool MC>
struct McOps;

template <>
struct McOps<true> {
  // 3-D tiled TMA load delivered to every CTA of this cluster named in
  // cta_mask: the box lands at the same shared-memory offset in each, and each
  // one's mbarrier at `bar`'s offset receives the byte count.
  static __device__ __forceinline__ void load_3d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                                 int c1, int c2, uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "h"(cta_mask)
        : "memory");
  }
  // Warp-converged MMA commit (one elected lane) that arrives once on the
  // mbarrier at `bar`'s offset in every CTA of cta_mask when this thread's
  // earlier tcgen05 MMAs have completed.
  static __device__ __forceinline__ void commit_w(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;\n\t}" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
  }
};

}  // namespace fa
