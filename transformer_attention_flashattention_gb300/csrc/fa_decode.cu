// Split-KV attention for a few query rows against a long key cache (a decode step),
// sm_103a.  Same result as the forward pass, softmax(scale * Q K^T [+ mask]) V with
// the natural-log LSE ("FlashAttention 2 + 3 — speicherbewusste Attention-Kernels",
// "Kernpunkte"; the KV cache of "Begriffe auf dieser Seite"), for the last N_q
// positions of a sequence of N_k keys: query row i sees keys 0 .. N_k - N_q + i when
// causal (bottom-right alignment), all keys otherwise.
//
// With N_q <= 16 the work is a stream over K and V (2 * N_k * d * 2 bytes per head):
// HBM-bound, so it runs on the CUDA cores, not the tensor cores.  The key range is
// cut into `splits` chunks; one CTA per (b*h, chunk):
//   warp 8        producer: per 64-key tile, one cp.async.bulk per K and per V row into
//                 shared memory rows padded to 2d+16 bytes (conflict-free 16-byte reads),
//                 a 3-stage ring with mbarrier full/empty handoff
//   warps 0-7     scores (one key per thread, its K row in registers), online softmax
//                 per query row (running max and correction, as in the forward pass),
//                 then O += P V (two d-columns per thread)
// Each chunk writes its normalised partial O and LSE to scratch; a second kernel merges
// the chunks: LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.  With one
// chunk the first kernel writes O and LSE directly.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_launch.h"
#include "fa_params.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kDecTile = 64;                 // keys per stage
constexpr int kDecStages = 3;
constexpr int kDecCompute = 256;             // compute threads (8 warps)
constexpr int kDecThreads = kDecCompute + 32;
constexpr int kDecMaxQ = 16;
constexpr float kDecLn2 = 0.693147180559945309f;
constexpr unsigned kDecStatusTimeout = 16u;

template <int D>
struct DecCfg {
  static constexpr int kRow = 2 * D + 16;                  // padded row bytes
  static constexpr int kStageBytes = 2 * kDecTile * kRow;  // K and V of one tile
  static constexpr int kKOff = 0;
  static constexpr int kQOff = kDecStages * kStageBytes;   // q * scale * log2(e), fp32 [kDecMaxQ][D]
  static constexpr int kSOff = kQOff + kDecMaxQ * D * 4;   // scores / weights [kDecMaxQ][kDecTile]
  static constexpr int kStatOff = kSOff + kDecMaxQ * kDecTile * 4;  // m, l, alpha per row
  static constexpr int kBarOff = (kStatOff + 3 * kDecMaxQ * 4 + 7) / 8 * 8;
  static constexpr int kBytes = kBarOff + 2 * kDecStages * 8 + 16;
};

__device__ __forceinline__ void compute_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecCompute) : "memory");
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kDecThreads) fa_decode_split_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecCfg<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  auto full = [&](int s) { return sbase + C::kBarOff + 8u * s; };
  auto empty = [&](int s) { return sbase + C::kBarOff + 8u * (kDecStages + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kBarOff + 16 * kDecStages);
  float* qs = reinterpret_cast<float*>(smem + C::kQOff);
  float* sc = reinterpret_cast<float*>(smem + C::kSOff);
  float* m_run = reinterpret_cast<float*>(smem + C::kStatOff);
  float* l_run = m_run + kDecMaxQ;
  float* alpha = l_run + kDecMaxQ;

  const int bh = blockIdx.x / p.splits;
  const int split = blockIdx.x % p.splits;
  const int k0 = split * p.chunk;
  const int k1 = min(p.Nk, k0 + p.chunk);
  const int ntiles = k1 > k0 ? (k1 - k0 + kDecTile - 1) / kDecTile : 0;
  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), kDecCompute / 32);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  // q scaled into the log2 domain; running statistics
  const size_t qbase = static_cast<size_t>(bh) * p.Nq * D;
  for (int i = tid; i < p.Nq * D; i += blockDim.x) {
    const uint16_t raw = static_cast<const uint16_t*>(p.q)[qbase + i];
    float x;
    if constexpr (BF16) x = __uint_as_float(static_cast<uint32_t>(raw) << 16);
    else x = __half2float(__ushort_as_half(raw));
    qs[i] = x * p.scale_log2;
  }
  if (tid < kDecMaxQ) {
    m_run[tid] = -INFINITY;
    l_run[tid] = 0.f;
    alpha[tid] = 1.f;
  }
  __syncthreads();
  const ptx::WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp == kDecCompute / 32) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint8_t* kg = static_cast<const uint8_t*>(p.k) + static_cast<size_t>(bh) * p.Nk * D * 2;
      const uint8_t* vg = static_cast<const uint8_t*>(p.v) + static_cast<size_t>(bh) * p.Nk * D * 2;
      int issued[kDecStages] = {-1, -1, -1};
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kDecStages;
        const uint32_t fill = i / kDecStages;
        if (!ptx::mbar_wait(empty(s), (fill & 1u) ^ 1u, ctl, kDecStatusTimeout)) break;
        const int r0 = k0 + i * kDecTile;
        const int rows = min(kDecTile, k1 - r0);
        ptx::mbar_arrive_expect_tx(full(s), static_cast<uint32_t>(rows) * D * 4);
        const uint32_t kd = sbase + C::kKOff + s * C::kStageBytes;
        const uint32_t vd = kd + kDecTile * C::kRow;
        for (int r = 0; r < rows; ++r) {
          bulk_copy(kd + r * C::kRow, kg + static_cast<size_t>(r0 + r) * D * 2, D * 2, full(s));
          bulk_copy(vd + r * C::kRow, vg + static_cast<size_t>(r0 + r) * D * 2, D * 2, full(s));
        }
        issued[s] = static_cast<int>(fill);
      }
      // copies in flight land before the CTA exits
      for (int s = 0; s < kDecStages; ++s)
        if (issued[s] >= 0 && !ptx::mbar_wait_drain(full(s), static_cast<uint32_t>(issued[s]) & 1u, p.timeout_ns))
          atomicOr(p.status, kDecStatusTimeout);
    }
    return;
  }

  // ------------------------------------------------------------------ compute warps
  const int kk = tid & (kDecTile - 1);        // key of this thread in the score phase
  const int qg = tid / kDecTile;              // query group 0..3 (rows qg, qg+4, ...)
  constexpr int kCols2 = D / 2;               // column pairs
  constexpr int kQSets = kDecCompute / kCols2;   // 4 (d=128) or 8 (d=64) query sets in P.V
  const int cp = tid % kCols2;                // column pair of this thread in P.V
  const int qset = tid / kCols2;
  float2 acc[kDecMaxQ / kQSets];
#pragma unroll
  for (int i = 0; i < kDecMaxQ / kQSets; ++i) acc[i] = make_float2(0.f, 0.f);
  const int last_key_shift = p.Nk - p.Nq;     // causal: row i sees keys <= shift + i

  for (int i = 0; i < ntiles; ++i) {
    const int s = i % kDecStages;
    const bool got = ptx::mbar_wait(full(s), (i / kDecStages) & 1u, ctl, kDecStatusTimeout);
    compute_sync();
    if (!got || *abort_flag) break;               // every compute warp leaves together
    const uint8_t* ks = smem + C::kKOff + s * C::kStageBytes;
    const uint8_t* vs = ks + kDecTile * C::kRow;
    const int key = k0 + i * kDecTile + kk;
    const int valid = min(kDecTile, k1 - (k0 + i * kDecTile));   // rows loaded in this tile

    // scores: this thread's K row against its query rows
    {
      uint4 krow[D / 8];
#pragma unroll
      for (int c = 0; c < D / 8; ++c) krow[c] = *reinterpret_cast<const uint4*>(ks + kk * C::kRow + 16 * c);
      for (int qi = qg; qi < p.Nq; qi += kDecCompute / kDecTile) {
        const float* qr = qs + qi * D;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const float4 qa = *reinterpret_cast<const float4*>(qr + 8 * c);
          const float4 qb = *reinterpret_cast<const float4*>(qr + 8 * c + 4);
          const float2 x0 = unpack2<BF16>(krow[c].x), x1 = unpack2<BF16>(krow[c].y);
          const float2 x2 = unpack2<BF16>(krow[c].z), x3 = unpack2<BF16>(krow[c].w);
          a0 = fmaf(qa.x, x0.x, a0); a1 = fmaf(qa.y, x0.y, a1);
          a0 = fmaf(qa.z, x1.x, a0); a1 = fmaf(qa.w, x1.y, a1);
          a0 = fmaf(qb.x, x2.x, a0); a1 = fmaf(qb.y, x2.y, a1);
          a0 = fmaf(qb.z, x3.x, a0); a1 = fmaf(qb.w, x3.y, a1);
        }
        const bool visible = key < k1 && (!p.causal || key <= last_key_shift + qi);
        sc[qi * kDecTile + kk] = visible ? a0 + a1 : -INFINITY;
      }
    }
    compute_sync();

    // online softmax: warp w owns rows w and w + 8
    for (int qi = warp; qi < p.Nq; qi += kDecCompute / 32) {
      float* row = sc + qi * kDecTile;
      const float s0 = row[lane], s1 = row[lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      const float m_old = m_run[qi];
      const float m_new = fmaxf(m_old, mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float p0 = ptx::ex2(s0 - m_use), p1 = ptx::ex2(s1 - m_use);
      float sum = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
      row[lane] = p0;
      row[lane + 32] = p1;
      __syncwarp();
      if (lane == 0) {
        const float a = m_old == -INFINITY ? 0.f : ptx::ex2(m_old - m_use);
        alpha[qi] = a;
        l_run[qi] = l_run[qi] * a + sum;
        m_run[qi] = m_new;
      }
    }
    compute_sync();

    // O += P V: two columns per thread, rows qset, qset + kQSets, ...
#pragma unroll
    for (int a = 0; a < kDecMaxQ / kQSets; ++a) {
      const int qi = qset + a * kQSets;
      if (qi < p.Nq) {
        const float* pr = sc + qi * kDecTile;
        float2 o2 = acc[a];
        const float al = alpha[qi];
        o2.x *= al;
        o2.y *= al;
        for (int k = 0; k < valid; ++k) {             // rows past `valid` were never loaded
          const float w = pr[k];
          const float2 v2 = unpack2<BF16>(*reinterpret_cast<const uint32_t*>(vs + k * C::kRow + 4 * cp));
          o2.x = fmaf(w, v2.x, o2.x);
          o2.y = fmaf(w, v2.y, o2.y);
        }
        acc[a] = o2;
      }
    }
    // this stage may be refilled once every compute warp is past it
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty(s));
    compute_sync();
  }
  if (*abort_flag) return;

  // normalise; write the final output (one chunk) or this chunk's partial
  const bool single = p.splits == 1;
#pragma unroll
  for (int a = 0; a < kDecMaxQ / kQSets; ++a) {
    const int qi = qset + a * kQSets;
    if (qi < p.Nq) {
      const float l = l_run[qi];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float ox = acc[a].x * inv, oy = acc[a].y * inv;
      if (single) {
        uint32_t w;
        if constexpr (BF16) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(ox, oy);
          w = *reinterpret_cast<const uint32_t*>(&h);
        } else {
          const __half2 h = __floats2half2_rn(ox, oy);
          w = *reinterpret_cast<const uint32_t*>(&h);
        }
        reinterpret_cast<uint32_t*>(p.o)[(qbase + static_cast<size_t>(qi) * D) / 2 + cp] = w;
      } else {
        const size_t pb = ((static_cast<size_t>(bh) * p.splits + split) * p.Nq + qi) * D;
        reinterpret_cast<float2*>(p.part_o)[pb / 2 + cp] = make_float2(ox, oy);
      }
    }
  }
  if (tid < p.Nq) {
    const float l = l_run[tid];
    const float lse = l > 0.f ? (m_run[tid] + ptx::lg2(l)) * kDecLn2 : -INFINITY;
    if (single) {
      if (p.lse) p.lse[static_cast<size_t>(bh) * p.Nq + tid] = lse;
    } else {
      p.part_lse[(static_cast<size_t>(bh) * p.splits + split) * p.Nq + tid] = lse;
    }
  }
}

// One warp per (b*h, query row): LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_decode_merge_kernel(const __grid_constant__ DecodeParams p) {
  const int row = blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= p.BH * p.Nq) return;
  const int bh = row / p.Nq, qi = row % p.Nq;
  const float* pl = p.part_lse + static_cast<size_t>(bh) * p.splits * p.Nq + qi;
  float mx = -INFINITY;
  for (int s = lane; s < p.splits; s += 32) mx = fmaxf(mx, pl[static_cast<size_t>(s) * p.Nq]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  constexpr int E = D / 32;
  float out[E];
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] = 0.f;
  float total = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const float ls = pl[static_cast<size_t>(s) * p.Nq];
      const float w = ls == -INFINITY ? 0.f : __expf(ls - mx);
      total += w;
      const float* po = p.part_o + ((static_cast<size_t>(bh) * p.splits + s) * p.Nq + qi) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) out[e] = fmaf(w, po[e], out[e]);
    }
  }
  const float inv = total > 0.f ? 1.f / total : 0.f;
  uint16_t* orow = static_cast<uint16_t*>(p.o) + (static_cast<size_t>(bh) * p.Nq + qi) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    uint32_t w;
    if constexpr (BF16) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(out[e] * inv, out[e + 1] * inv);
      w = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const __half2 h = __floats2half2_rn(out[e] * inv, out[e + 1] * inv);
      w = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint32_t*>(orow + e) = w;
  }
  if (lane == 0 && p.lse) p.lse[static_cast<size_t>(bh) * p.Nq + qi] = total > 0.f ? mx + __logf(total) : -INFINITY;
}

template <int D, bool BF16>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  auto split = fa_decode_split_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize, DecCfg<D>::kBytes);
  if (e != cudaSuccess) return e;
  split<<<p.BH * p.splits, kDecThreads, DecCfg<D>::kBytes, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  fa_decode_merge_kernel<D, BF16><<<(p.BH * p.Nq + 7) / 8, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(int d, bool bf16, const DecodeParams& p, cudaStream_t stream) {
  if (d == 128) return bf16 ? launch_decode_t<128, true>(p, stream) : launch_decode_t<128, false>(p, stream);
  if (d == 64) return bf16 ? launch_decode_t<64, true>(p, stream) : launch_decode_t<64, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
