// Standard attention with the N x N matrix materialised in HBM (fa_fwd_naive), as the
// concept card "FlashAttention 2 + 3 — speicherbewusste Attention-Kernels" describes it
// ("Worum es geht": the whole score matrix is written to HBM and read back for the softmax
// and the weighted sum; "Begriffe auf dieser Seite", HBM: 5-10 full HBM passes a forward
// pass against about one; "Warum es zählt": 3 to 10 times the GPU hours of the tiled
// kernel at long context) and as the "Flash Attention" glossary's standard attention
// ("/01 Was ist Flash Attention?": memory quadratic in the sequence length).
// Three steps, each a full pass over an N x N matrix per head:
//   1. S = scale * Q K^T, fp32, by a library GEMM (cuBLAS, strided-batched over heads);
//   2. a row softmax kernel (below) that reads each S row once, writes P in the input
//      dtype over the first half of the same row, and writes the row's LSE;
//   3. O = P V by a second library GEMM.
// cuBLAS is loaded at the first call (dlopen of the runtime's soname); the tiled kernels
// do not depend on it.
#include <dlfcn.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_launch.h"

namespace fa {
namespace {

constexpr int kNaiveThreads = 256;
constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ float max4(float4 a) { return fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)); }

// Block-wide maximum or sum; every thread gets the result.  The partials are combined in
// warp order, so the sum is the same on every run.
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = kMax ? fmaxf(v, w) : v + w;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int k = 1; k < kNaiveThreads / 32; ++k) r = kMax ? fmaxf(r, red[k]) : r + red[k];
  __syncthreads();
  return r;
}

template <bool BF16>
__device__ __forceinline__ uint2 pack4(float a, float b, float c, float d) {
  uint2 u;
  if constexpr (BF16) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
  } else {
    const __half2 lo = __floats2half2_rn(a, b), hi = __floats2half2_rn(c, d);
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
  }
  return u;
}

// One CTA per score row r (head r / N, query row i = r % N).  S rows are `ld` floats apart
// (ld a multiple of 4, ld >= N).  Each thread keeps VPT float4 of the row in registers: the
// visible columns (0..N-1, or 0..i when causal) are read once, the row maximum and the sum of
// exp(S - max) are reduced across the block, and P = exp(S - max) / sum is written in the input
// dtype over the start of the same row (P rows are 2*ld elements apart), zeros at the masked
// columns, so the P V GEMM reads exactly softmax(S).  All reads of the row finish before the
// first block reduction returns, so the in-place write cannot overwrite a value still to be read.
template <int VPT, bool BF16>
__global__ void __launch_bounds__(kNaiveThreads) fa_naive_softmax_kernel(float* __restrict__ s,
                                                                         float* __restrict__ lse, int N,
                                                                         long long ld, int causal) {
  __shared__ float red[kNaiveThreads / 32];
  const long long r = blockIdx.x;
  const int i = static_cast<int>(r % N);
  float* row = s + r * ld;
  const int limit = causal ? i + 1 : N;
  float4 x[VPT];
  float m = -INFINITY;
#pragma unroll
  for (int t = 0; t < VPT; ++t) {
    const int c = 4 * (t * kNaiveThreads + static_cast<int>(threadIdx.x));
    x[t] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (c < limit) {
      x[t] = __ldcs(reinterpret_cast<const float4*>(row + c));
      if (c + 1 >= limit) x[t].y = -INFINITY;
      if (c + 2 >= limit) x[t].z = -INFINITY;
      if (c + 3 >= limit) x[t].w = -INFINITY;
    }
    m = fmaxf(m, max4(x[t]));
  }
  m = block_reduce<true>(m, red);
  const float mb = m * kLog2e;
  float sum = 0.f;
#pragma unroll
  for (int t = 0; t < VPT; ++t) {
    x[t].x = exp2f(fmaf(x[t].x, kLog2e, -mb));
    x[t].y = exp2f(fmaf(x[t].y, kLog2e, -mb));
    x[t].z = exp2f(fmaf(x[t].z, kLog2e, -mb));
    x[t].w = exp2f(fmaf(x[t].w, kLog2e, -mb));
    sum += (x[t].x + x[t].y) + (x[t].z + x[t].w);
  }
  sum = block_reduce<false>(sum, red);
  const float inv = 1.f / sum;
  uint2* prow = reinterpret_cast<uint2*>(row);   // 4 16-bit P values per uint2
#pragma unroll
  for (int t = 0; t < VPT; ++t) {
    const int c = 4 * (t * kNaiveThreads + static_cast<int>(threadIdx.x));
    if (c < N) prow[c / 4] = pack4<BF16>(x[t].x * inv, x[t].y * inv, x[t].z * inv, x[t].w * inv);
  }
  if (lse != nullptr && threadIdx.x == 0) lse[r] = m + logf(sum);
}

template <bool BF16>
cudaError_t launch_softmax(float* s, float* lse, long long rows, int N, long long ld, int causal,
                           cudaStream_t stream) {
  const int vecs = (N + 3) / 4;
  const int per = (vecs + kNaiveThreads - 1) / kNaiveThreads;
  const dim3 grid(static_cast<unsigned>(rows)), block(kNaiveThreads);
  if (per <= 1) fa_naive_softmax_kernel<1, BF16><<<grid, block, 0, stream>>>(s, lse, N, ld, causal);
  else if (per <= 2) fa_naive_softmax_kernel<2, BF16><<<grid, block, 0, stream>>>(s, lse, N, ld, causal);
  else if (per <= 4) fa_naive_softmax_kernel<4, BF16><<<grid, block, 0, stream>>>(s, lse, N, ld, causal);
  else if (per <= 8) fa_naive_softmax_kernel<8, BF16><<<grid, block, 0, stream>>>(s, lse, N, ld, causal);
  else if (per <= 16) fa_naive_softmax_kernel<16, BF16><<<grid, block, 0, stream>>>(s, lse, N, ld, causal);
  else fa_naive_softmax_kernel<32, BF16><<<grid, block, 0, stream>>>(s, lse, N, ld, causal);
  return cudaGetLastError();
}

// The C-linkage strided-batched GEMM with a cublasComputeType_t (the header also declares a
// C++ overload taking a cudaDataType, so the type is spelled out).
using GemmFn = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int, const void*,
                                  const void*, cudaDataType, int, long long, const void*, cudaDataType, int,
                                  long long, const void*, void*, cudaDataType, int, long long, int,
                                  cublasComputeType_t, cublasGemmAlgo_t);

// cuBLAS entry points, resolved once from the shared library the process already has loaded
// (PyTorch's), else from the runtime's soname on the loader's search path; one handle a device.
struct Blas {
  bool tried = false;
  decltype(&cublasCreate_v2) create = nullptr;
  decltype(&cublasSetStream_v2) set_stream = nullptr;
  decltype(&cublasSetWorkspace_v2) set_workspace = nullptr;
  GemmFn gemm = nullptr;
  cublasHandle_t handle[64] = {};
};

std::mutex g_blas_mu;
Blas g_blas;

bool load_blas() {
  if (g_blas.tried) return g_blas.gemm != nullptr;
  g_blas.tried = true;
  void* lib = dlopen("libcublas.so.13", RTLD_NOW | RTLD_LOCAL | RTLD_NOLOAD);
  if (lib == nullptr) lib = dlopen("libcublas.so.13", RTLD_NOW | RTLD_LOCAL);
  if (lib == nullptr) return false;
  g_blas.create = reinterpret_cast<decltype(&cublasCreate_v2)>(dlsym(lib, "cublasCreate_v2"));
  g_blas.set_stream = reinterpret_cast<decltype(&cublasSetStream_v2)>(dlsym(lib, "cublasSetStream_v2"));
  g_blas.set_workspace = reinterpret_cast<decltype(&cublasSetWorkspace_v2)>(dlsym(lib, "cublasSetWorkspace_v2"));
  g_blas.gemm = reinterpret_cast<GemmFn>(dlsym(lib, "cublasGemmStridedBatchedEx"));
  if (!g_blas.create || !g_blas.set_stream || !g_blas.set_workspace || !g_blas.gemm) {
    g_blas.gemm = nullptr;
    return false;
  }
  return true;
}

}  // namespace

int run_naive(const void* q, const void* k, const void* v, void* o, float* lse, float* s, long long ld,
              void* blas_ws, unsigned long long blas_ws_bytes, int BH, int N, int d, float scale, int causal,
              bool bf16, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_blas_mu);
  if (!load_blas()) return FA_ERR_CUDA;
  cublasHandle_t& h = g_blas.handle[dev];
  if (h == nullptr && g_blas.create(&h) != CUBLAS_STATUS_SUCCESS) {
    h = nullptr;
    return FA_ERR_CUDA;
  }
  // the GEMMs' scratch is this call's own (part of the caller's workspace), so calls that
  // share the handle but run at once on other streams, with other workspaces, do not share it
  if (g_blas.set_stream(h, stream) != CUBLAS_STATUS_SUCCESS ||
      g_blas.set_workspace(h, blas_ws, static_cast<size_t>(blas_ws_bytes)) != CUBLAS_STATUS_SUCCESS)
    return FA_ERR_CUDA;
  const cudaDataType dt = bf16 ? CUDA_R_16BF : CUDA_R_16F;
  const float zero = 0.f, one = 1.f;
  const long long nd = static_cast<long long>(N) * d, nld = static_cast<long long>(N) * ld;
  // Row-major S (N x ld) is column-major S^T = K Q^T: A = K read transposed (d x N, ld d),
  // B = Q (d x N, ld d), C = S^T (N x N, ld ld).
  if (g_blas.gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, N, N, d, &scale, k, dt, d, nd, q, dt, d, nd, &zero, s, CUDA_R_32F,
                  static_cast<int>(ld), nld, BH, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return FA_ERR_LAUNCH;
  const cudaError_t e = bf16 ? launch_softmax<true>(s, lse, static_cast<long long>(BH) * N, N, ld, causal, stream)
                             : launch_softmax<false>(s, lse, static_cast<long long>(BH) * N, N, ld, causal, stream);
  if (e != cudaSuccess) return FA_ERR_LAUNCH;
  // Row-major O (N x d) is column-major O^T = V^T P^T: A = V (d x N, ld d), B = P^T (N x N,
  // ld 2*ld 16-bit elements: P sits in the first half of each S row), C = O^T (d x N, ld d).
  if (g_blas.gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, d, N, N, &one, v, dt, d, nd, s, dt, static_cast<int>(2 * ld),
                  2 * nld, &zero, o, dt, d, nd, BH, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return FA_ERR_LAUNCH;
  return FA_OK;
}

}  // namespace fa
