// Host-side declarations shared by the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

struct FwdParams;
struct QuantParams;
struct DecodeParams;
struct BwdParams;

// Launch one forward kernel instantiation on `stream`; returns the launch status.
cudaError_t launch_fwd(int d, bool bf16, const FwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const FwdParams& p, int grid, cudaStream_t stream);
// One-tile-per-CTA forward (16-bit, head dim 64, two CTAs a SM): 128-row units.
cudaError_t launch_fwd1(bool bf16, const FwdParams& p, int grid, cudaStream_t stream);
// CTA-pair forward (16-bit, head dim 128); `grid` is even (two CTAs a cluster).
cudaError_t launch_fwd2(bool bf16, const FwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_quant_fp8(const QuantParams& p, cudaStream_t stream);
cudaError_t launch_decode(int d, bool bf16, const DecodeParams& p, cudaStream_t stream);
// Prep (D, LSE*log2e), then the dQ kernel, then the dK/dV kernel, all on `stream`.
cudaError_t launch_bwd(int d, bool bf16, const BwdParams& p, int grid, cudaStream_t stream);

// Materialising attention (fa_fwd_naive): library GEMM S = scale Q K^T into `s` (fp32 rows
// `ld` floats apart), the row softmax in place (P in the input dtype, LSE), library GEMM
// O = P V, all on `stream`; `blas_ws` is the GEMMs' scratch.  Returns an fa_status.
int run_naive(const void* q, const void* k, const void* v, void* o, float* lse, float* s, long long ld,
              void* blas_ws, unsigned long long blas_ws_bytes, int BH, int N, int d, float scale, int causal,
              bool bf16, cudaStream_t stream);

// fa_decode's shape and size checks (FA_OK, FA_ERR_SHAPE or FA_ERR_UNSUPPORTED).
int check_decode(int B, int H, int Nq, int Nk, int d);

}  // namespace fa
