// Instantiations and launcher of the f16/bf16 attention forward kernel.
#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {

namespace {
template <int D, bool BF16>
cudaError_t launch_one(const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = fa_fwd_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       FwdSmem<D>::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, FwdSmem<D>::kAlloc, stream>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_fwd(int d, bool bf16, const FwdParams& p, int grid, cudaStream_t stream) {
  if (d == 128) return bf16 ? launch_one<128, true>(p, grid, stream) : launch_one<128, false>(p, grid, stream);
  if (d == 64) return bf16 ? launch_one<64, true>(p, grid, stream) : launch_one<64, false>(p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
