// Instantiations and launchers of the f16/bf16 attention forward kernel.
#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <int D, Elem E>
cudaError_t launch_fwd_kernel(const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = fa_fwd_kernel<D, E>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       FwdCfg<D, E>::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, FwdCfg<D, E>::kAlloc, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(int d, bool bf16, const FwdParams& p, int grid, cudaStream_t stream) {
  if (d == 128)
    return bf16 ? launch_fwd_kernel<128, Elem::BF16>(p, grid, stream)
                : launch_fwd_kernel<128, Elem::F16>(p, grid, stream);
  if (d == 64)
    return bf16 ? launch_fwd_kernel<64, Elem::BF16>(p, grid, stream)
                : launch_fwd_kernel<64, Elem::F16>(p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
