// Instantiations and launcher of the CTA-pair (cta_group::2) attention forward kernel.
#include "fa_fwd2_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <Elem E>
cudaError_t launch_fwd2_kernel(const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = fa_fwd2_kernel<E>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Fwd2Cfg<E>::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, Fwd2Cfg<E>::kAlloc, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd2(bool bf16, const FwdParams& p, int grid, cudaStream_t stream) {
  if (grid <= 0 || (grid & 1)) return cudaErrorInvalidValue;
  return bf16 ? launch_fwd2_kernel<Elem::BF16>(p, grid, stream) : launch_fwd2_kernel<Elem::F16>(p, grid, stream);
}

}  // namespace fa
