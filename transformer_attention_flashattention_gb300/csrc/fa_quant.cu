// FP8 prologue for sm_103a: optional Walsh-Hadamard rotation along d, block absmax,
// E4M3 quantisation (the block-wise 8-bit storage with a Hadamard transform of the
// FlashAttention-3 news piece, "Drei technische Hebel", item 3, and the absmax
// scaling of "FlashAttention 2 + 3 — speicherbewusste Attention-Kernels",
// "Kernpunkte").  HBM-bound: one CTA reads a 64-row block once and writes it once.
//
// One CTA per (b*h, 64-row block), 8 warps x 8 rows; lane l holds elements
// [l*E, l*E + E) of a row (E = d/32).  The rotation is the fast transform in
// natural (Sylvester) order: butterflies (a, b) -> (a + b, a - b) at strides
// 1, 2, ..., d/2, the first log2(E) inside a thread, the rest across lanes by
// shuffles.  It is left unnormalised: with y = x H and a = max |y| over the
// block, the stored codes e4m3(y * 448 / a) equal e4m3((y / sqrt d) / s) for the
// normalised rotation, and the stored scale is s = a / (448 sqrt d).
//
// Variants: a sign mask negates chosen coordinates before the transform (the
// randomised rotation x D H); with one scale per head, the kernel first runs in a
// mode that only writes each block's absmax, a small kernel takes the head's
// maximum into every block entry, and a second pass quantises with it.
#include <cstdint>

#include <cuda_bf16.h>

#include "fa_launch.h"
#include "fa_params.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kQuantRows = 64;
constexpr int kQuantThreads = 256;
constexpr int kQuantWarps = kQuantThreads / 32;
constexpr int kRowsPerWarp = kQuantRows / kQuantWarps;
constexpr float kE4m3Max = 448.f;

template <int D>
__global__ void __launch_bounds__(kQuantThreads) fa_quant_fp8_kernel(const __grid_constant__ QuantParams p) {
  constexpr int E = D / 32;                       // elements per lane
  __shared__ float s_wmax[kQuantWarps];
  __shared__ float s_factor;
  __shared__ __align__(16) uint8_t s_t[D][kQuantRows + 16];   // transposed codes (+16 B pad per row)

  const int blk = blockIdx.x % p.n_sblk;
  const int bh = blockIdx.x / p.n_sblk;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int n_base = blk * kQuantRows;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x);

  float y[kRowsPerWarp][E];
  float amax = 0.f;
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int n = n_base + warp * kRowsPerWarp + rr;
    if (n < p.N) {
      const __nv_bfloat16* src = x + (static_cast<size_t>(bh) * p.N + n) * D + lane * E;
      if constexpr (E == 4) {
        const uint2 raw = *reinterpret_cast<const uint2*>(src);
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
        y[rr][0] = __low2float(lo);
        y[rr][1] = __high2float(lo);
        y[rr][2] = __low2float(hi);
        y[rr][3] = __high2float(hi);
      } else {
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(src);
        y[rr][0] = __low2float(v);
        y[rr][1] = __high2float(v);
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) y[rr][e] = 0.f;
    }
    if (p.hadamard) {
      // randomised rotation: this lane's coordinates lane*E .. lane*E+E-1 of the sign mask
      const int c0 = lane * E;
      const unsigned long long word = c0 < 64 ? p.flips_lo : p.flips_hi;
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((word >> ((c0 + e) & 63)) & 1ull) y[rr][e] = -y[rr][e];
      // strides 1 .. E/2 inside the thread
#pragma unroll
      for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & h) == 0) {
            const float a = y[rr][e], b = y[rr][e + h];
            y[rr][e] = a + b;
            y[rr][e + h] = a - b;
          }
        }
      }
      // strides E .. D/2 across lanes
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float other = __shfl_xor_sync(0xFFFFFFFFu, y[rr][e], m);
          y[rr][e] = upper ? other - y[rr][e] : y[rr][e] + other;
        }
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(y[rr][e]));
  }

  // block absmax -> quantisation factor and stored scale
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if (lane == 0) s_wmax[warp] = amax;
  __syncthreads();
  const size_t sidx = static_cast<size_t>(bh) * p.n_sblk + blk;
  if (threadIdx.x == 0) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kQuantWarps; ++w) a = fmaxf(a, s_wmax[w]);
    if (p.amax_mode == 1) {
      p.scale[sidx] = a;                 // first pass of a per-head scale: absmax only
      s_factor = 0.f;
    } else {
      if (p.amax_mode == 2) a = p.scale[sidx];   // the head's absmax
      s_factor = a > 0.f ? kE4m3Max / a : 0.f;
      float s = 1.f;
      if (a > 0.f) s = p.hadamard ? a * (1.f / (kE4m3Max * sqrtf(static_cast<float>(D)))) : a / kE4m3Max;
      p.scale[sidx] = s;
    }
  }
  __syncthreads();
  if (p.amax_mode == 1) return;
  const float f = s_factor;

#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int nl = warp * kRowsPerWarp + rr;
    const int n = n_base + nl;
    uint32_t codes;
    if constexpr (E == 4) {
      codes = ptx::pack4_e4m3(y[rr][0] * f, y[rr][1] * f, y[rr][2] * f, y[rr][3] * f);
    } else {
      codes = ptx::pack4_e4m3(y[rr][0] * f, y[rr][1] * f, 0.f, 0.f) & 0xFFFFu;
    }
    if (p.transpose_out) {
#pragma unroll
      for (int e = 0; e < E; ++e) s_t[lane * E + e][nl] = static_cast<uint8_t>(codes >> (8 * e));
    } else if (n < p.N) {
      uint8_t* dst = p.x8 + (static_cast<size_t>(bh) * p.N + n) * D + lane * E;
      if constexpr (E == 4) *reinterpret_cast<uint32_t*>(dst) = codes;
      else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(codes);
    }
  }
  if (p.transpose_out) {
    __syncthreads();
    // [d][64] codes -> rows of [d, N]: 16-byte chunks, N % 16 == 0 so a chunk is all in or all out
    const int valid = min(kQuantRows, p.N - n_base);
    for (int i = threadIdx.x; i < D * (kQuantRows / 16); i += kQuantThreads) {
      const int c = i / (kQuantRows / 16), ch = i % (kQuantRows / 16);
      if (ch * 16 < valid) {
        const uint4 v = *reinterpret_cast<const uint4*>(&s_t[c][ch * 16]);
        *reinterpret_cast<uint4*>(p.x8 + (static_cast<size_t>(bh) * D + c) * p.N + n_base + ch * 16) = v;
      }
    }
  }
}

// Per-head scale, between the two passes: the largest block absmax of each (b, h)
// into every block entry.  One warp per head.
__global__ void __launch_bounds__(256) fa_quant_head_max_kernel(const __grid_constant__ QuantParams p) {
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (w >= p.BH) return;                 // whole warps leave together
  float* row = p.scale + static_cast<size_t>(w) * p.n_sblk;
  float m = 0.f;
  for (int i = lane; i < p.n_sblk; i += 32) m = fmaxf(m, row[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  for (int i = lane; i < p.n_sblk; i += 32) row[i] = m;
}

cudaError_t launch_quant_pass(const QuantParams& p, unsigned grid, cudaStream_t stream) {
  if (p.d == 128) fa_quant_fp8_kernel<128><<<grid, kQuantThreads, 0, stream>>>(p);
  else if (p.d == 64) fa_quant_fp8_kernel<64><<<grid, kQuantThreads, 0, stream>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_fp8(const QuantParams& p, cudaStream_t stream) {
  const long long blocks = static_cast<long long>(p.n_sblk) * p.BH;
  if (blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
  const unsigned grid = static_cast<unsigned>(blocks);
  if (!p.per_head) {
    QuantParams q = p;
    q.amax_mode = 0;
    return launch_quant_pass(q, grid, stream);
  }
  QuantParams q = p;
  q.amax_mode = 1;
  cudaError_t e = launch_quant_pass(q, grid, stream);
  if (e != cudaSuccess) return e;
  const long long warps_threads = static_cast<long long>(p.BH) * 32;
  fa_quant_head_max_kernel<<<static_cast<unsigned>((warps_threads + 255) / 256), 256, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  q.amax_mode = 2;
  return launch_quant_pass(q, grid, stream);
}

}  // namespace fa
