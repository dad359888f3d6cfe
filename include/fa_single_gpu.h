/* libfa_single_gpu — the single-GPU build of libfa: everything libfa exports
 * (include/fa.h), plus the forward whose CTA pairs share K/V tile loads by
 * thread-block-cluster multicast. It is a separate library so that a process
 * driving several GPUs (one rank per GPU) never loads multicast code; load it
 * only in a process that uses one GPU.
 *
 * Source: "FlashAttention HBM bytes, one head, 8K" (inferenceinterviews.com),
 * "A strong answer": when a head's K/V no longer fit in L2, the thread blocks
 * of a cluster can share each K/V tile instead of fetching it separately.
 */
#ifndef LIBFA_FA_SINGLE_GPU_H
#define LIBFA_FA_SINGLE_GPU_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* fa_forward (BF16 tensors; same arguments, layouts, results and status codes)
 * with the CTAs of the prefill kernel in clusters of two: when both CTAs of a
 * pair work on query blocks of the same head and key range, each fetches half
 * the rows of every K/V tile from L2 once and TMA multicast writes it into both
 * CTAs' shared memory, halving L2-to-SM K/V traffic. Pairs that straddle two
 * heads load privately; an odd number of blocks adds one idle CTA. Plans whose
 * key ranges are split over several CTAs (fewer query blocks than a wave, or a
 * split last wave) and decode-shaped requests run the plain kernel instead.
 * The result equals fa_forward's bit for bit (same arithmetic; only the loads
 * differ). Every tensor must be device memory of the current device
 * (FA_ERR_INVALID_ARG otherwise), as for every libfa entry point. Returns
 * FA_ERR_UNSUPPORTED without doing anything when the environment names a
 * multi-process job (WORLD_SIZE > 1). */
int fa_forward_cluster_multicast(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal,
                                 float scale, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBFA_FA_SINGLE_GPU_H */
