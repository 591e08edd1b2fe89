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
//   lane 0 of warp 0 also issues the loads: per 64-key tile, TMA loads of K and V
//                 (128-byte swizzle, which keeps the per-row reads bank-conflict free) into
//                 a 6-stage ring; a stage is refilled once all 8 warps released it
//   warps 0-7     each warp owns 8 keys of every tile: scores (lanes split d, then a
//                 9-shuffle reduce-scatter), its own online softmax per query row (running
//                 max and correction, as in the forward pass) and its own O slice; the 8
//                 warps are merged by log-sum-exp once at the end (no barrier per tile)
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
constexpr int kDecCompute = 256;             // compute threads (8 warps)
constexpr int kDecThreads = kDecCompute;
constexpr int kDecMaxQ = 16;                 // query rows a call may have
constexpr int kDecFewQ = 4;                  // bound of the few-row instantiation
constexpr float kDecLn2 = 0.693147180559945309f;
constexpr unsigned kDecStatusTimeout = 16u;

// NQ bounds the query rows (registers hold NQ rows of O and statistics per thread).  Two
// CTAs share an SM whenever their registers allow it (head dim 64, or at most kDecFewQ rows):
// the ring is then 96 KB a CTA, and one CTA's start and finish overlap the other's stream.
// Otherwise (head dim 128 with up to 16 rows, 204 registers) one CTA has a 192 KB ring.
template <int D, int NQ>
struct DecCfg {
  static constexpr int kCtasPerSm = (D == 64 || NQ <= kDecFewQ) ? 2 : 1;
  static constexpr int kBoxes = D / 64;                    // 128-byte swizzle atoms per row
  static constexpr int kBoxBytes = kDecTile * 128;         // one atom column of a tile
  static constexpr int kTileBytes = kBoxes * kBoxBytes;    // K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;       // K and V of one tile
  static constexpr int kStages = (96 * 1024 * (3 - kCtasPerSm)) / kStageBytes;   // 96 or 192 KB
  static constexpr int kKOff = 0;
  static constexpr int kQOff = kStages * kStageBytes;      // q * scale * log2(e), fp32 [NQ][D]
  static constexpr int kSOff = kQOff + NQ * D * 4;         // scores / weights [NQ][kDecTile]
  static constexpr int kStatOff = kSOff + NQ * kDecTile * 4;   // m, l, alpha per row
  static constexpr int kBarOff = (kStatOff + 3 * NQ * 4 + 7) / 8 * 8;
  static constexpr int kBytes = kBarOff + 2 * kStages * 8 + 16;
  // the final merge of the 8 warps reuses the ring: [8 warps][NQ][D] fp32, and the
  // per-warp m and l in the score area
  static_assert((kDecCompute / 32) * NQ * D * 4 <= kStages * kStageBytes, "merge buffer exceeds the ring");
  static_assert(2 * (kDecCompute / 32) * NQ <= NQ * kDecTile, "merge statistics exceed the score area");
};

__device__ __forceinline__ void compute_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecCompute) : "memory");
}

// Byte offset of 16-byte chunk c (0 .. D/8-1) of tile row r under the 128-byte swizzle.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (c / 8) * (kDecTile * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

template <int D, bool BF16, int NQ>
__global__ void __launch_bounds__(kDecThreads, DecCfg<D, NQ>::kCtasPerSm)
    fa_decode_split_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecCfg<D, NQ>;
  constexpr int kDecStages = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  auto full = [&](int s) { return sbase + C::kBarOff + 8u * s; };
  auto empty = [&](int s) { return sbase + C::kBarOff + 8u * (kDecStages + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kBarOff + 16 * kDecStages);
  float* qs = reinterpret_cast<float*>(smem + C::kQOff);
  float* sc = reinterpret_cast<float*>(smem + C::kSOff);
  float* m_run = reinterpret_cast<float*>(smem + C::kStatOff);
  float* l_run = m_run + NQ;
  float* alpha = l_run + NQ;

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
  if (tid < NQ) {
    m_run[tid] = -INFINITY;
    l_run[tid] = 0.f;
    alpha[tid] = 1.f;
  }
  __syncthreads();
  const ptx::WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  // ------------------------------------------------------------------ loads
  // issued by lane 0 of warp 0: the first stages up front, then stage s is refilled
  // with tile i + kDecStages once every warp released tile i
  const bool loader = tid == 0;
  int last_issued = -1;
  auto issue = [&](int i) {
    const int st = i % kDecStages;
    const int r0 = k0 + i * kDecTile;
    // full boxes are transferred (rows past N_k read as zero), so expect all bytes
    ptx::mbar_arrive_expect_tx(full(st), C::kStageBytes);
    const uint32_t kd = sbase + C::kKOff + st * C::kStageBytes;
    const uint32_t vd = kd + C::kTileBytes;
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b) {
      ptx::tma_load_3d(kd + b * C::kBoxBytes, &p.tm_k, full(st), b * 64, r0, bh);
      ptx::tma_load_3d(vd + b * C::kBoxBytes, &p.tm_v, full(st), b * 64, r0, bh);
    }
    last_issued = i;
  };
  if (loader) {
    ptx::prefetch_tensormap(&p.tm_k);
    ptx::prefetch_tensormap(&p.tm_v);
    for (int i = 0; i < min(ntiles, kDecStages); ++i) issue(i);
  }

  // ------------------------------------------------------------------ compute warps
  // Warp w owns keys 8w .. 8w+7 of every tile and keeps its own running max, sum and
  // O slice per query row (lane l owns d-elements E*l .. E*l+E-1); the 8 warps' partial
  // results are merged once at the end.  No CTA-wide barrier per tile.
  constexpr int E = D / 32;
  constexpr int kKeysPerWarp = kDecTile / (kDecCompute / 32);   // 8
  const int last_key_shift = p.Nk - p.Nq;                       // causal: row i sees keys <= shift + i
  float acc[NQ][E];
  float m_w[NQ], l_w[NQ];
#pragma unroll
  for (int qi = 0; qi < NQ; ++qi) {
#pragma unroll
    for (int e = 0; e < E; ++e) acc[qi][e] = 0.f;
    m_w[qi] = -INFINITY;
    l_w[qi] = 0.f;
  }
  // key of this lane after the reduce-scatter: lane bits 4, 3, 2 -> key bits 2, 1, 0
  const int my_key = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);

  bool ok = true;
  for (int i = 0; i < ntiles; ++i) {
    const int s = i % kDecStages;
    if (!ptx::mbar_wait(full(s), (i / kDecStages) & 1u, ctl, kDecStatusTimeout)) { ok = false; break; }
    const uint8_t* ks = smem + C::kKOff + s * C::kStageBytes;
    const uint8_t* vs = ks + C::kTileBytes;
    const int kbase = warp * kKeysPerWarp;               // first key of this warp in the tile
    const int key0 = k0 + i * kDecTile + kbase;
    // this lane's d-slice of the warp's 8 K rows (E bf16/f16 values = E*2 bytes)
    float kv[kKeysPerWarp][E];
    uint32_t roff[kKeysPerWarp];
#pragma unroll
    for (int r = 0; r < kKeysPerWarp; ++r) {
      roff[r] = swz<D>(kbase + r, (E * lane) / 8) + ((E * lane) % 8) * 2;
      if constexpr (E == 4) {
        const uint2 kw = *reinterpret_cast<const uint2*>(ks + roff[r]);
        const float2 k01 = unpack2<BF16>(kw.x), k23 = unpack2<BF16>(kw.y);
        kv[r][0] = k01.x; kv[r][1] = k01.y; kv[r][2] = k23.x; kv[r][3] = k23.y;
      } else {
        const float2 k01 = unpack2<BF16>(*reinterpret_cast<const uint32_t*>(ks + roff[r]));
        kv[r][0] = k01.x; kv[r][1] = k01.y;
      }
    }

#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
      if (qi >= p.Nq) break;
      // partial dot products over this lane's slice, then a reduce-scatter across lanes
      float qv[E];
      if constexpr (E == 4) {
        const float4 q4 = *reinterpret_cast<const float4*>(qs + qi * D + E * lane);
        qv[0] = q4.x; qv[1] = q4.y; qv[2] = q4.z; qv[3] = q4.w;
      } else {
        const float2 q2 = *reinterpret_cast<const float2*>(qs + qi * D + E * lane);
        qv[0] = q2.x; qv[1] = q2.y;
      }
      float t8[kKeysPerWarp];
#pragma unroll
      for (int r = 0; r < kKeysPerWarp; ++r) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) a = fmaf(qv[e], kv[r][e], a);
        t8[r] = a;
      }
      float t4[4], t2[2];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const bool hi = lane & 16;
        const float send = hi ? t8[r] : t8[r + 4];
        const float keep = hi ? t8[r + 4] : t8[r];
        t4[r] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const bool hi = lane & 8;
        const float send = hi ? t4[r] : t4[r + 2];
        const float keep = hi ? t4[r + 2] : t4[r];
        t2[r] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
      }
      float sc1;
      {
        const bool hi = lane & 4;
        const float send = hi ? t2[0] : t2[1];
        const float keep = hi ? t2[1] : t2[0];
        sc1 = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
      }
      sc1 += __shfl_xor_sync(0xFFFFFFFFu, sc1, 2);
      sc1 += __shfl_xor_sync(0xFFFFFFFFu, sc1, 1);
      const int key = key0 + my_key;
      const bool visible = key < k1 && (!p.causal || key <= last_key_shift + qi);
      if (!visible) sc1 = -INFINITY;
      // online softmax over the warp's 8 keys
      float mx = sc1;
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
      const float m_new = fmaxf(m_w[qi], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float pk = ptx::ex2(sc1 - m_use);
      float sum = pk;
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 8);
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 16);
      const float corr = m_w[qi] == -INFINITY ? 0.f : ptx::ex2(m_w[qi] - m_use);
      l_w[qi] = l_w[qi] * corr + sum;
      m_w[qi] = m_new;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[qi][e] *= corr;
#pragma unroll
      for (int r = 0; r < kKeysPerWarp; ++r) {
        // weight of key r lives in the lanes whose bits 4,3,2 spell r
        const float w = __shfl_sync(0xFFFFFFFFu, pk, ((r >> 2) & 1) * 16 + ((r >> 1) & 1) * 8 + (r & 1) * 4);
        float vv[E];
        if constexpr (E == 4) {
          const uint2 vw = *reinterpret_cast<const uint2*>(vs + roff[r]);
          const float2 v01 = unpack2<BF16>(vw.x), v23 = unpack2<BF16>(vw.y);
          vv[0] = v01.x; vv[1] = v01.y; vv[2] = v23.x; vv[3] = v23.y;
        } else {
          const float2 v01 = unpack2<BF16>(*reinterpret_cast<const uint32_t*>(vs + roff[r]));
          vv[0] = v01.x; vv[1] = v01.y;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) acc[qi][e] = fmaf(w, vv[e], acc[qi][e]);
      }
    }
    // this warp's rows are read: the stage may be refilled once all 8 warps are here
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty(s));
    if (loader && i + kDecStages < ntiles) {
      if (!ptx::mbar_wait(empty(s), (i / kDecStages) & 1u, ctl, kDecStatusTimeout)) { ok = false; break; }
      issue(i + kDecStages);
    }
  }
  // copies in flight land before the CTA exits (immediate on the normal path)
  if (loader) {
    // tiles are issued in order, so the last fill of stage st is the largest tile
    // index <= last_issued that maps to st
    for (int st = 0; st < kDecStages && st <= last_issued; ++st) {
      const int i = last_issued - (last_issued - st) % kDecStages;
      if (!ptx::mbar_wait_drain(full(st), static_cast<uint32_t>(i / kDecStages) & 1u, p.timeout_ns))
        atomicOr(p.status, kDecStatusTimeout);
    }
  }
  // leave together if any warp gave up
  compute_sync();
  if (!ok || *abort_flag) return;

  // merge the 8 warps: M = max m_w, L = sum l_w 2^(m_w - M), O = sum acc_w 2^(m_w - M) / L
  float* red_o = reinterpret_cast<float*>(smem + C::kKOff);     // the ring is idle now
  float* red_m = sc;                                            // [8 warps][NQ]
  float* red_l = sc + (kDecCompute / 32) * NQ;
#pragma unroll
  for (int qi = 0; qi < NQ; ++qi) {
    if (qi >= p.Nq) break;
#pragma unroll
    for (int e = 0; e < E; ++e) red_o[(warp * NQ + qi) * D + E * lane + e] = acc[qi][e];
    if (lane == 0) {
      red_m[warp * NQ + qi] = m_w[qi];
      red_l[warp * NQ + qi] = l_w[qi];
    }
  }
  compute_sync();
  const bool single = p.splits == 1;
  for (int idx = tid; idx < p.Nq * (D / 2); idx += kDecCompute) {
    const int qi = idx / (D / 2), cpair = idx % (D / 2);
    float M = -INFINITY;
    for (int w = 0; w < kDecCompute / 32; ++w) M = fmaxf(M, red_m[w * NQ + qi]);
    float L = 0.f, ox = 0.f, oy = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kDecCompute / 32; ++w) {
        const float mw = red_m[w * NQ + qi];
        const float f = mw == -INFINITY ? 0.f : ptx::ex2(mw - M);
        L = fmaf(red_l[w * NQ + qi], f, L);
        ox = fmaf(red_o[(w * NQ + qi) * D + 2 * cpair], f, ox);
        oy = fmaf(red_o[(w * NQ + qi) * D + 2 * cpair + 1], f, oy);
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    ox *= inv;
    oy *= inv;
    if (single) {
      uint32_t wv;
      if constexpr (BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(ox, oy);
        wv = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __half2 h = __floats2half2_rn(ox, oy);
        wv = *reinterpret_cast<const uint32_t*>(&h);
      }
      reinterpret_cast<uint32_t*>(p.o)[(qbase + static_cast<size_t>(qi) * D) / 2 + cpair] = wv;
    } else {
      const size_t pb = ((static_cast<size_t>(bh) * p.splits + split) * p.Nq + qi) * D;
      reinterpret_cast<float2*>(p.part_o)[pb / 2 + cpair] = make_float2(ox, oy);
    }
    if (cpair == 0) {
      const float lse = L > 0.f ? (M + ptx::lg2(L)) * kDecLn2 : -INFINITY;
      if (single) {
        if (p.lse) p.lse[static_cast<size_t>(bh) * p.Nq + qi] = lse;
      } else {
        p.part_lse[(static_cast<size_t>(bh) * p.splits + split) * p.Nq + qi] = lse;
      }
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

template <int D, bool BF16, int NQ>
cudaError_t launch_split(const DecodeParams& p, cudaStream_t stream) {
  auto split = fa_decode_split_kernel<D, BF16, NQ>;
  constexpr int kSmem = DecCfg<D, NQ>::kBytes + 1024;      // room to align the base to 1 KB
  cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if (DecCfg<D, NQ>::kCtasPerSm > 1) {
    e = cudaFuncSetAttribute(split, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  split<<<p.BH * p.splits, kDecThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t e = p.Nq <= kDecFewQ ? launch_split<D, BF16, kDecFewQ>(p, stream)
                                   : launch_split<D, BF16, kDecMaxQ>(p, stream);
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
