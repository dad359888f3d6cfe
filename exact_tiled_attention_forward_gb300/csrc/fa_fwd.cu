// Fused prefill forward of libfa: instantiates the plain kernel of
// fa_fwd_kernel.cuh (BF16, FP16 and FP8 E4M3, d = 64 and 128)
// and its merge kernel.
#include "fa_fwd_kernel.cuh"

namespace fa {

namespace {

template <int D, Elem E>
cudaError_t launch_fwd_t(const FwdMaps& m, const FwdParams& p, int units, cudaStream_t stream) {
  cudaError_t e = launch_main_t<D, false, E>(m, p, units, stream);
  if (e != cudaSuccess || p.n_tail == 0 || p.cm) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(((long long)p.n_tail * kBlockRows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_merge_kernel<D, E>, p);
}

}  // namespace

int fwd_cluster_capacity(int d, int s) {
  if (s < 2 || s > 8) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  static int cache[64][2][9];   // 0 = not yet asked, else capacity + 1
  int& c = cache[dev][d == 128 ? 1 : 0][s];
  if (c == 0) c = 1 + (d == 128 ? cluster_capacity_t<128>(s) : cluster_capacity_t<64>(s));
  return c - 1;
}

size_t fwd_smem_bytes(int d) {
  return d == 128 ? (size_t)Cfg<128>::kSmemBytes : (size_t)Cfg<64>::kSmemBytes;
}

cudaError_t launch_fwd(int d, const FwdMaps& m, const FwdParams& p, int units, cudaStream_t stream) {
  if (units <= 0) return cudaSuccess;
  if (p.elem == (int)Elem::E4M3)
    return d == 128 ? launch_fwd_t<128, Elem::E4M3>(m, p, units, stream)
                    : launch_fwd_t<64, Elem::E4M3>(m, p, units, stream);
  if (p.elem == (int)Elem::F16)
    return d == 128 ? launch_fwd_t<128, Elem::F16>(m, p, units, stream)
                    : launch_fwd_t<64, Elem::F16>(m, p, units, stream);
  return d == 128 ? launch_fwd_t<128, Elem::BF16>(m, p, units, stream)
                  : launch_fwd_t<64, Elem::BF16>(m, p, units, stream);
}

}  // namespace fa
