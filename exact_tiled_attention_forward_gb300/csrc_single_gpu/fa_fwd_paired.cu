// The paired-load forward (declared in include/fa_single_gpu.h): the fused
// kernel of fa_fwd_kernel.cuh instantiated with MC = true. CTAs run in
// clusters of two; when both units of a pair are query blocks of the same
// head, each CTA fetches half the rows of every K/V tile once and the TMA
// multicast delivers them to both CTAs ("FlashAttention HBM bytes, one head,
// 8K", "A strong answer": once K/V outgrow L2, share each tile across the
// thread blocks of a cluster). Everything else (validation, plan, tensor maps,
// the plain kernel for plans with split key ranges) is libfa's own code,
// linked into this library from the same objects.
#include "fa_mc_ops.cuh"
#include "fa_fwd_kernel.cuh"
#include "fa.h"
#include "fa_single_gpu.h"

#include <cstdlib>

namespace fa {
namespace {

cudaError_t launch_paired(int d, const FwdMaps& m, const FwdParams& p, int units, cudaStream_t stream) {
  if (units <= 0) return cudaSuccess;
  return d == 128 ? launch_main_t<128, true, Elem::BF16>(m, p, units, stream)
                  : launch_main_t<64, true, Elem::BF16>(m, p, units, stream);
}

// One rank of a job launched with several processes (torchrun and the like
// export WORLD_SIZE): each of them may drive another GPU, and this library's
// multicast belongs only in a process that uses one GPU.
bool in_multi_process_job() {
  const char* w = getenv("WORLD_SIZE");
  return w && atoi(w) > 1;
}

}  // namespace
}  // namespace fa

extern "C" int fa_forward_cluster_multicast(const void* q, const void* k, const void* v, void* o,
                                            float* lse, int B, int H_q, int H_kv, int N_q, int N_k,
                                            int d, int causal, float scale, void* stream) {
  if (fa::in_multi_process_job()) return FA_ERR_UNSUPPORTED;
  return fa::forward_impl(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, causal, scale,
                          static_cast<cudaStream_t>(stream), fa::pool_workspace(), 0, fa::launch_paired);
}
