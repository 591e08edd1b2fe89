// Instantiations and launcher of the one-tile-per-CTA forward kernel (16-bit, head dim 64).
#include "fa_fwd1_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <Elem E>
cudaError_t launch_fwd1_kernel(const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = fa_fwd1_kernel<E>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Fwd1Cfg<E>::kAlloc);
  if (e != cudaSuccess) return e;
  // two CTAs must fit an SM's shared memory: ask for the largest carveout
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads1, Fwd1Cfg<E>::kAlloc, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd1(bool bf16, const FwdParams& p, int grid, cudaStream_t stream) {
  return bf16 ? launch_fwd1_kernel<Elem::BF16>(p, grid, stream) : launch_fwd1_kernel<Elem::F16>(p, grid, stream);
}

}  // namespace fa
