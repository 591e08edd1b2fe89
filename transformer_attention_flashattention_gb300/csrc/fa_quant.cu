// FP8 prologue for sm_103a: optional Walsh-Hadamard rotation along d, block absmax,
// E4M3 quantisation (the block-wise 8-bit storage with a Hadamard transform of the
// FlashAttention-3 news piece, "Drei technische Hebel", item 3, and the absmax
// scaling of "FlashAttention 2 + 3 — speicherbewusste Attention-Kernels",
// "Kernpunkte").  HBM-bound: every 64-row block is read once and written once.
//
// A persistent grid of 4 CTAs per SM walks the (b*h, 64-row block) blocks.  Each
// block is contiguous in HBM; one bulk copy streams it into a shared-memory stage
// while the CTA works on the previous one, so the stream of loads never stops.
// 8 warps x 8 rows, four lanes per row.  The rotation is the fast transform in
// natural (Sylvester) order: butterflies (a, b) -> (a + b, a - b) at strides 1, 2,
// ..., d/2, all but the last two inside a thread, those two across the row's lanes
// by shuffles.  It is left unnormalised: with y = x H and a = max |y| over the
// block, the stored codes e4m3(y * 448 / a) equal e4m3((y / sqrt d) / s) for the
// normalised rotation, and the stored scale is s = a / (448 sqrt d).
//
// Variants: a sign mask negates chosen coordinates before the transform (the
// randomised rotation x D H); with one scale per head, the kernel first runs in a
// mode that only writes each block's absmax, a small kernel takes the head's
// maximum into every block entry, and a second pass quantises with it.  One launch
// can take up to three tensors of the same shape (Q and K rotated, V transposed):
// their blocks form one sequence, so the grid has one ramp and one tail, not three.
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
constexpr int kRowsPerWarp = 8;                    // four lanes per row
constexpr int kQuantCtasPerSm = 4;
constexpr float kE4m3Max = 448.f;
constexpr unsigned kQuantStatusLoadTimeout = 1u;    // a wait for a block's copy gave up
constexpr unsigned kQuantStatusDrainTimeout = 8u;   // a copy in flight had not landed at exit
static_assert(kRowsPerWarp * kQuantWarps == kQuantRows, "one row per four lanes");

// Packed fp32 pairs with IEEE rounding and subnormals kept, like the scalar float
// arithmetic around them: each lane's result is bitwise the scalar a + b, a * b + c, a * b.
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Shared memory of one CTA: two input stages, the staged codes, control words.
template <int D>
struct QuantSmem {
  static constexpr int kPitch = D + 4;   // bytes per row of staged codes (conflict-free transpose reads)
  __nv_bfloat16 in[2][kQuantRows * D];   // one 64-row block per stage, rows of D elements
  uint8_t t[kQuantRows * kPitch];       // the block's codes, row-major, for the transposed output
  uint64_t full[2];                     // stage s holds its block once its phase completes
  float wmax[kQuantWarps];
  float factor;
  int abort;
};

// Four lanes share a row: lane l holds the quarter q = l & 3 of row 8 * warp + (l >> 2),
// E = d/4 coordinates, read from shared memory in 16-byte chunks.  The lane reads
// chunk k ^ a at step k, a = (q ^ row) & (E/8 - 1), which spreads a quarter-warp's
// reads over all banks; selects on the raw words then put the chunks back in order.
// The rotation runs its strides 1 .. E/2 inside the thread and E, 2E across the four
// lanes, in the same order and with the same operations as a one-thread transform.
template <int D>
__global__ void __launch_bounds__(kQuantThreads, kQuantCtasPerSm) fa_quant_fp8_kernel(const __grid_constant__ QuantParams p) {
  using S = QuantSmem<D>;
  constexpr int E = D / 4;                        // coordinates per lane
  constexpr int NC = E / 8;                       // 16-byte chunks per lane
  constexpr uint32_t kRowBytes = D * 2;
  __shared__ __align__(128) S sm;

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int q = lane & 3;
  const int nl = warp * kRowsPerWarp + (lane >> 2);     // row within the block
  const int a = (q ^ (lane >> 2)) & (NC - 1);
  // blocks of one tensor, and of the launch (below 2^31, checked on the host)
  const int per = p.BH * p.n_sblk;
  const long long total = static_cast<long long>(per) * p.ntens;
  const long long G = gridDim.x;
  // the tensor of a block (selects, not a dynamic index into parameter space)
  auto pick = [](int ti, auto a0, auto a1, auto a2) { return ti == 0 ? a0 : (ti == 1 ? a1 : a2); };
  const uint32_t full0 = ptx::smem_u32(&sm.full[0]);
  const ptx::WaitCtl ctl{&sm.abort, p.status, p.timeout_ns};

  // copy of block b (only its rows inside the head) into stage s
  auto issue = [&](long long b, int s) {
    const int ti = static_cast<int>(b) / per;
    const int lb = static_cast<int>(b) - ti * per;
    const int bh = lb / p.n_sblk, blk = lb % p.n_sblk;
    const uint32_t rows = static_cast<uint32_t>(min(kQuantRows, p.N - blk * kQuantRows));
    const uint32_t bar = full0 + 8u * static_cast<uint32_t>(s);
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(pick(ti, p.x[0], p.x[1], p.x[2]));
    ptx::mbar_arrive_expect_tx(bar, rows * kRowBytes);
    ptx::bulk_load(ptx::smem_u32(sm.in[s]), x + (static_cast<size_t>(bh) * p.N + blk * kQuantRows) * D,
                   rows * kRowBytes, bar);
  };

  if (threadIdx.x == 0) {
    sm.abort = 0;
    ptx::mbar_init(full0, 1);
    ptx::mbar_init(full0 + 8u, 1);
    ptx::fence_barrier_init();
    if (blockIdx.x < total) issue(blockIdx.x, 0);
  }
  __syncthreads();

  int it = 0;
  for (long long b = blockIdx.x; b < total; b += G, ++it) {
    const int s = it & 1;
    // The other stage was last read before the first barrier of the previous block.
    if (threadIdx.x == 0 && b + G < total) issue(b + G, s ^ 1);
    const bool landed = ptx::mbar_wait(full0 + 8u * s, static_cast<uint32_t>(it >> 1) & 1u, ctl,
                                       kQuantStatusLoadTimeout);
    if (__syncthreads_or(!landed)) {
      // leave only after the copies in flight (this stage's, and the next one's) have landed
      if (threadIdx.x == 0) {
        bool drained = ptx::mbar_wait_drain(full0 + 8u * s, static_cast<uint32_t>(it >> 1) & 1u, p.timeout_ns);
        if (b + G < total)
          drained = ptx::mbar_wait_drain(full0 + 8u * (s ^ 1), static_cast<uint32_t>((it + 1) >> 1) & 1u,
                                         p.timeout_ns) && drained;
        if (!drained) atomicOr(p.status, kQuantStatusDrainTimeout);
      }
      return;
    }

    const int ti = static_cast<int>(b) / per;
    const int lb = static_cast<int>(b) - ti * per;
    const int bh = lb / p.n_sblk, blk = lb % p.n_sblk;
    const int n_base = blk * kQuantRows;
    const int valid = min(kQuantRows, p.N - n_base);
    float y[E];
    if (nl < valid) {
      const uint4* src = reinterpret_cast<const uint4*>(sm.in[s] + nl * D + q * E);
      uint4 c[NC];
#pragma unroll
      for (int k = 0; k < NC; ++k) c[k] = src[k ^ a];          // c[k] = chunk k ^ a
#pragma unroll
      for (int bit = 1; bit < NC; bit <<= 1) {                  // swap back, one bit of a at a time
        const bool sw = (a & bit) != 0;
#pragma unroll
        for (int k = 0; k < NC; ++k) {
          if ((k & bit) == 0) {
            const uint4 lo = c[k], hi = c[k + bit];
            c[k] = sw ? hi : lo;
            c[k + bit] = sw ? lo : hi;
          }
        }
      }
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        const uint32_t w[4] = {c[k].x, c[k].y, c[k].z, c[k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
          y[8 * k + 2 * i] = __low2float(v);
          y[8 * k + 2 * i + 1] = __high2float(v);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) y[e] = 0.f;
    }

    if (pick(ti, p.hadamard[0], p.hadamard[1], p.hadamard[2])) {
      if ((p.flips_lo | p.flips_hi) != 0) {
        // randomised rotation: bit e of m negates this lane's coordinate q*E + e
        const int c0 = q * E;
        const unsigned long long word = c0 < 64 ? p.flips_lo : p.flips_hi;
        const uint32_t m = static_cast<uint32_t>(word >> (c0 & 63));
#pragma unroll
        for (int e = 0; e < E; ++e)
          if ((m >> e) & 1u) y[e] = -y[e];
      }
      // stride 1 inside each register pair
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float u = y[e], v = y[e + 1];
        y[e] = u + v;
        y[e + 1] = u - v;
      }
      // strides 2 .. E/2 on packed pairs: u + v as an add, u - v as v * -1 + u (exact product)
      const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
      for (int h = 2; h < E; h <<= 1) {
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          if ((e & h) == 0) {
            const float2 u = make_float2(y[e], y[e + 1]), v = make_float2(y[e + h], y[e + h + 1]);
            const float2 sum = add2_rn(u, v), dif = fma2_rn(v, neg1, u);
            y[e] = sum.x;
            y[e + 1] = sum.y;
            y[e + h] = dif.x;
            y[e + h + 1] = dif.y;
          }
        }
      }
      // strides E and 2E across the row's four lanes: the lower lane keeps u + v, the
      // upper u - v, both as y * sign + other
#pragma unroll
      for (int m = 1; m < 4; m <<= 1) {
        const float sg = (q & m) != 0 ? -1.f : 1.f;
        const float2 s2 = make_float2(sg, sg);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 other = make_float2(__shfl_xor_sync(0xFFFFFFFFu, y[e], m),
                                           __shfl_xor_sync(0xFFFFFFFFu, y[e + 1], m));
          const float2 r = fma2_rn(make_float2(y[e], y[e + 1]), s2, other);
          y[e] = r.x;
          y[e + 1] = r.y;
        }
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(y[e]));

    // block absmax -> quantisation factor and stored scale
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) sm.wmax[warp] = amax;
    __syncthreads();   // every row of stage s has been read, and every warp's maximum written
    if (threadIdx.x == 0) {
      float* const scale = pick(ti, p.scale[0], p.scale[1], p.scale[2]);
      const int hadamard = pick(ti, p.hadamard[0], p.hadamard[1], p.hadamard[2]);
      float am = 0.f;
#pragma unroll
      for (int w = 0; w < kQuantWarps; ++w) am = fmaxf(am, sm.wmax[w]);
      if (p.amax_mode == 1) {
        scale[lb] = am;                  // first pass of a per-head scale: absmax only
        sm.factor = 0.f;
      } else {
        if (p.amax_mode == 2) am = scale[lb];   // the head's absmax
        sm.factor = am > 0.f ? kE4m3Max / am : 0.f;
        float sc = 1.f;
        if (am > 0.f) sc = hadamard ? am * (1.f / (kE4m3Max * sqrtf(static_cast<float>(D)))) : am / kE4m3Max;
        scale[lb] = sc;
      }
    }
    __syncthreads();
    if (p.amax_mode == 1) continue;
    const float f = sm.factor;

    uint32_t codes[E / 4];
    const float2 f2 = make_float2(f, f);
#pragma unroll
    for (int w = 0; w < E / 4; ++w) {
      const float2 p01 = mul2_rn(make_float2(y[4 * w], y[4 * w + 1]), f2);
      const float2 p23 = mul2_rn(make_float2(y[4 * w + 2], y[4 * w + 3]), f2);
      codes[w] = ptx::pack4_e4m3(p01.x, p01.y, p23.x, p23.y);
    }
    uint8_t* const x8 = pick(ti, p.x8[0], p.x8[1], p.x8[2]);
    if (!pick(ti, p.transpose_out[0], p.transpose_out[1], p.transpose_out[2])) {
      if (nl < valid) {
        uint8_t* dst = x8 + (static_cast<size_t>(bh) * p.N + n_base + nl) * D + q * E;
#pragma unroll
        for (int k = 0; k < E / 16; ++k)
          *reinterpret_cast<uint4*>(dst + 16 * k) =
              make_uint4(codes[4 * k], codes[4 * k + 1], codes[4 * k + 2], codes[4 * k + 3]);
      }
      continue;
    }
    // Transposed output: stage the codes row-major, then each thread moves a 4-row x
    // 4-coordinate tile, transposed by byte permutes, into four rows of [d, N].
    {
      uint32_t* row = reinterpret_cast<uint32_t*>(sm.t + nl * S::kPitch + q * E);
#pragma unroll
      for (int w = 0; w < E / 4; ++w) row[w] = codes[w];
    }
    __syncthreads();
    // tile i: rows 4 * rg .. 4 * rg + 3, coordinates 4 * cg .. 4 * cg + 3; a warp takes 8 row
    // groups of 4 coordinate groups (distinct banks); N % 16 == 0, so a group is all in or out
    for (int i = threadIdx.x; i < (D / 4) * (kQuantRows / 4); i += kQuantThreads) {
      const int rg = ((i >> 3) / (D / 4)) * 8 + (i & 7);
      const int cg = (i >> 3) % (D / 4);
      if (rg * 4 < valid) {
        const uint8_t* src = sm.t + rg * 4 * S::kPitch + cg * 4;
        const uint32_t r0 = *reinterpret_cast<const uint32_t*>(src);
        const uint32_t r1 = *reinterpret_cast<const uint32_t*>(src + S::kPitch);
        const uint32_t r2 = *reinterpret_cast<const uint32_t*>(src + 2 * S::kPitch);
        const uint32_t r3 = *reinterpret_cast<const uint32_t*>(src + 3 * S::kPitch);
        const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r0, r1, 0x7362);
        const uint32_t t2 = __byte_perm(r2, r3, 0x5140), t3 = __byte_perm(r2, r3, 0x7362);
        const uint32_t col[4] = {__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632),
                                 __byte_perm(t1, t3, 0x5410), __byte_perm(t1, t3, 0x7632)};
        uint8_t* dst = x8 + (static_cast<size_t>(bh) * D + cg * 4) * p.N + n_base + rg * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(e) * p.N) = col[e];
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
  float* row = p.scale[0] + static_cast<size_t>(w) * p.n_sblk;
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
  if (p.ntens < 1 || p.ntens > 3 || (p.per_head && p.ntens != 1)) return cudaErrorInvalidValue;
  const long long blocks = static_cast<long long>(p.n_sblk) * p.BH * p.ntens;
  if (blocks >= (1ll << 31) || p.sm_count < 1) return cudaErrorInvalidConfiguration;
  const long long ctas = static_cast<long long>(p.sm_count) * kQuantCtasPerSm;
  const unsigned grid = static_cast<unsigned>(blocks < ctas ? blocks : ctas);
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
