// Instantiation and launcher of the E4M3 attention forward kernel (head dim 128).
#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {

cudaError_t launch_fwd_fp8(const FwdParams& p, int grid, cudaStream_t stream) {
  using Cfg = FwdCfg<128, Elem::E4M3>;
  auto kern = fa_fwd_kernel<128, Elem::E4M3>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, Cfg::kAlloc, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fa
