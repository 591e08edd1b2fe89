// Attention backward for sm_103a (f16/bf16, head dim 64 or 128): dQ, dK, dV of
// O = softmax(scale * Q K^T [+ causal mask]) V for an upstream gradient dO, from the
// forward pass's O and natural-log LSE.
//
// The pages name the backward pass as the place FlashAttention-2 parallelises better
// (concept card "FlashAttention 2 + 3 — speicherbewusste Attention-Kernels", section
// "Kernpunkte") but print no formula; the gradient is the calculus of the forward
// definition, recomputing P tile by tile from the saved LSE so that no N x N matrix
// reaches HBM:
//   P = 2^(scale*log2(e) * Q K^T - LSE*log2(e)),  D_i = sum_c dO_ic O_ic,
//   dS = P * (dO V^T - D),  dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Three kernels on the caller's stream, no atomics (results are deterministic):
//   prep   -D and -LSE*log2(e) into a workspace padded to 128 rows per head (padding:
//          0 and -inf, so padded queries get P = 0); negated so that both enter the
//          packed-pair arithmetic below as addends
//   dq     Q-stationary: per 128-row Q tile (Q and dO copied into TMEM once per tile),
//          stream K_j, V_j; S = Q K^T and dP = dO V^T (TS MMAs), P and dS in
//          registers, dS packed into TMEM over the dP columns, then dQ += dS K (TS
//          MMA, K as an MN-major operand)
//   dkdv   K/V-stationary: per 128-key tile, stream Q_i, dO_i (+ their LSE, D);
//          S^T = K Q^T and dP^T = V dO^T (SS), then P^T and dS^T per key row (packed
//          into TMEM), then dV += P^T dO and dK += dS^T Q (TS)
// S and dP are computed twice (once per kernel) in exchange for no dQ reduction.
//
// Each main kernel is a persistent grid with these roles (320 threads):
//   warps 0-7  compute: warp w takes TMEM lanes 32*(w%4).. (Q rows, or key rows) and
//              column half w/4, so every row is shared by two threads
//   warp 8     TMA producer (the warp runs the loop, one elected lane issues): the
//              unit's two stationary tiles, then the streamed tiles
//              (dq: K in a 3-slot ring and V in a 2-slot ring; dkdv: Q and dO in
//              2-slot rings)
//   warp 9     MMA issuer (the warp runs the loop converged, one elected lane issues)
//              and TMEM owner
// dq kernel: whole 128-key tiles, S and dP with N = 128, in the tensor-pipe order
//   ... S(j)  dP(j)  S(j+1)  dQ(j)  dP(j+1)  S(j+2)  dQ(j+1) ...
// The unit's Q and dO tiles are copied from shared memory into TMEM once (tcgen05.cp, issued
// by the MMA thread in order before the unit's products), so all three
// products take their A operand from TMEM and read only B (K or V) from shared memory.
// The compute threads form P(j) as soon as S(j) is in, and signal once S(j) is in their
// registers so that S(j+1) can follow; once dP(j) is in, they form dS(j) and pack it over
// the dP columns they have read.  dP(j+1) follows dQ(j) in the in-order pipe.  24 MMA
// instructions a key tile (d = 128).
// TMEM: Q | dO (64 columns each, two 16-bit values a column) | S | dP, then dS (128 each) |
// dQ (D).
// dkdv kernel: whole 128-query tiles, S^T and dP^T with N = 128, in the tensor-pipe order
//   ... S^T(i)  dP^T(i)  dV(i)  S^T(i+1)  dK(i)  dP^T(i+1)  dV(i+1) ...
// The compute threads form P^T(i) as soon as S^T(i) is in, packed over the S^T columns
// they have read (queries 0-63 at columns 0-31, 64-127 at 64-95), for dV += P^T dO; then,
// once dP^T(i) is in, dS^T(i) from the P values they kept in registers, packed the same
// way over the dP^T columns, for dK += dS^T Q.  So each half of their work overlaps two
// products of the pipe.  The pipe runs its MMAs in order: S^T(i+1) overwrites P^T(i) only
// after dV(i) has read it, dP^T(i+1) overwrites dS^T(i) only after dK(i).  Both A operands
// come from TMEM, which keeps shared memory (the operand feed of the S^T and dP^T MMAs)
// for the B operands and the loads.  32 MMA instructions a Q tile (d = 128).
// TMEM (512 columns at d = 128): S^T | dP^T (128 columns each) | dV | dK.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

constexpr int kBwdComputeWarps = 8;
constexpr int kBwdThreads = kBwdComputeWarps * 32 + 64;
constexpr int kBwdLoadWarp = 8;
constexpr int kBwdMmaWarp = 9;
constexpr int kBwdStages = 2;                                      // dkdv: Q and dO ring slots
constexpr uint32_t kTmS = 0, kTmDP = 128, kTmAcc = 256;            // dkdv: S^T | dP^T | dV | dK
constexpr uint32_t kQQ = 0, kQDO = 64, kQS = 128, kQDP = 256, kQAcc = 384;   // dq: Q | dO | S | dP | dQ
constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct BwdCfg {
  using L = FwdCfg<D, Elem::BF16>;                    // tile geometry (same for f16)
  static constexpr int kTile = L::kTileBytes;         // 128 rows x D, 128-byte swizzle atoms
  static constexpr int kStatOff = 0;                  // the unit's two stationary tiles
  static constexpr int kVecBytes = 128 * 4;           // one tile's -LSE*log2(e) (or -D) values
  // dq kernel: the stationary Q and dO tiles, then K in a ring of kDqKSlots tiles and V in
  // one of kDqVSlots.  V_j is free once dP(j) has run, K_j only after dQ += dS(j) K_j, so
  // the two rings release at different points and K needs the deeper one.
  static constexpr int kDqKSlots = 3, kDqVSlots = 2;
  static constexpr int kDqKOff = 2 * kTile;
  static constexpr int kDqVOff = kDqKOff + kDqKSlots * kTile;
  static constexpr int kDqEnd = kDqVOff + kDqVSlots * kTile;
  // dkdv kernel: the stationary K and V tiles, Q and dO in rings of kBwdStages slots (Q_i is
  // free after dK += dS^T Q_i, dO_i after dV += P^T dO_i), and each Q slot's -LSE*log2(e)
  // and -D vectors
  static constexpr int kKvQOff = 2 * kTile;
  static constexpr int kKvDoOff = kKvQOff + kBwdStages * kTile;
  static constexpr int kKvVecOff = kKvDoOff + kBwdStages * kTile;
  static constexpr int kDkdvEnd = kKvVecOff + kBwdStages * 2 * kVecBytes;
  static constexpr int kBarOff = kDqEnd > kDkdvEnd ? kDqEnd : kDkdvEnd;
  // barriers
  static constexpr int kStFull = 0, kStEmpty = 1, kReady = 2, kDone = kReady + kBwdStages;
  static constexpr int kSdpFull = kDone + kBwdStages, kDsFull = kSdpFull + 2, kAccFull = kDsFull + 2;   // per half
  static constexpr int kMmaDone = kAccFull + 1;
  // dq kernel only: S read into registers (compute arrives); Q and dO's TMEM columns free
  // again (commit after the unit's last S and dP); the K and V rings' full / free
  // barriers per slot.  It takes kSdpFull / kSdpFull + 1 as "S in" / "dP in" (commits) and
  // kStEmpty as "stationary tiles copied into TMEM" (commit after the copies).
  static constexpr int kSdpFree = kMmaDone + 1, kQtFree = kSdpFree + 1;
  static constexpr int kKFull = kQtFree + 1, kKFree = kKFull + kDqKSlots;
  static constexpr int kVFull = kKFree + kDqKSlots, kVFree = kVFull + kDqVSlots;
  // dkdv kernel only: its dO slots' full / free barriers.  It also takes kReady / kDone as
  // its Q slots' full / free barriers, kSdpFull / kSdpFull + 1 as "S^T in" / "dP^T in"
  // (commits), and kDsFull / kDsFull + 1 as "dS^T written" / "P^T written" (compute arrives).
  static constexpr int kDoFull = kVFree + kDqVSlots, kDoFree = kDoFull + kBwdStages;
  // dkdv kernel only: the stationary V tile's full / empty barriers (kStFull / kStEmpty are
  // its K tile's), so that each is reloaded as soon as the unit's last product using it ran
  static constexpr int kVsFull = kDoFree + kBwdStages, kVsEmpty = kVsFull + 1;
  // d = 128, both kernels: unit u's epilogue has staged its accumulators in the ring slots of
  // its last tile and its TMA stores have read them (compute arrives on kEpiFree + u % 3);
  // the producer refills those slots only then.  Three barriers in turn, so that no barrier
  // completes twice before the producer has waited for it (a unit can finish while the
  // producer waits for an earlier unit's epilogue: at most two, with the dq kernel's three
  // K slots and units of one tile)
  static constexpr int kEpiFree = kVsEmpty + 1;
  static constexpr int kNumBars = kEpiFree + 3;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;        // slack to align the base to 1 KB
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// The k-th unit of this CTA of the persistent grid, (b*h, tile blk); false once it
// has none left.  The dq kernel's units are Q tiles, the dkdv kernel's K/V tiles.
//  - Non-causal: head-major, dealt round-robin, so concurrent CTAs share a few heads
//    and the streamed tiles hit L2.
//  - Causal: a unit's cost grows with its Q tile (dq: tile i sees i + 1 key tiles) or
//    shrinks with its K/V tile (dkdv: tile j is seen by n - j Q tiles); causal_unit pairs
//    tiles b and n-1-b of one head and levels the grid's last wave.
__device__ __forceinline__ bool bwd_unit_at(const BwdParams& p, int k, bool cost_grows, int& bh, int& blk) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  if (!p.causal) {
    const int u = c + k * G;
    if (u >= p.num_units) return false;
    bh = u / p.n_blk;
    blk = u % p.n_blk;
    return true;
  }
  return causal_unit(G, c, p.BH, p.n_blk, k, cost_grows, bh, blk);
}

// ---------------------------------------------------------------------------- prep

// -D_i = -sum_c dO_ic O_ic and -LSE_i * log2(e), one row per group of D/8 lanes.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __grid_constant__ BwdParams p) {
  constexpr int kLanes = D / 8;                      // 8 elements (16 bytes) per lane
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long grow = t / kLanes;                 // row over [B*H, n_pad]
  const int part = static_cast<int>(t % kLanes);
  // no early exit: every lane takes part in the shuffles below
  const bool valid = grow < static_cast<long long>(p.BH) * p.n_pad;
  const int bh = valid ? static_cast<int>(grow / p.n_pad) : 0;
  const int row = valid ? static_cast<int>(grow % p.n_pad) : p.n_pad;
  float acc = 0.f;
  if (row < p.N) {
    const size_t off = (static_cast<size_t>(bh) * p.N + row) * D + part * 8;
    const uint4 ov = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + off);
    const uint4 dv = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + off);
    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 a, b;
      if constexpr (BF16) {
        a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
        b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[e]));
      } else {
        a = __half22float2(*reinterpret_cast<const __half2*>(&ow[e]));
        b = __half22float2(*reinterpret_cast<const __half2*>(&dw[e]));
      }
      acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
    }
  }
#pragma unroll
  for (int m = kLanes / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, m);
  if (valid && part == 0) {
    const size_t w = static_cast<size_t>(bh) * p.n_pad + row;
    p.ndelta[w] = row < p.N ? -acc : 0.f;
    p.nlse2[w] = row < p.N ? -(p.lse[static_cast<size_t>(bh) * p.N + row] * kLog2e) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------- shared pieces

template <int D, Elem E>
__device__ __forceinline__ void load_tile(const CUtensorMap* map, uint32_t dst, uint32_t bar, int row0, int bh) {
  using L = FwdCfg<D, E>;
#pragma unroll
  for (int a = 0; a < L::kAtoms; ++a)
    ptx::tma_load_3d(dst + a * L::kAtomBytes, map, bar, a * L::kAtomElems, row0, bh);
}

// P^T of one key row against 32 queries: P = 2^(s * c + nl) with the queries'
// -LSE*log2(e) as pairs from shared memory; with MASK, queries x < first get P = 0.  The
// values stay in pv for dS; w gets them packed.
template <bool BF16, bool MASK>
__device__ __forceinline__ void dkdv_p32(const uint32_t (&sr)[32], float2 cc, const float4* nl, int first,
                                         float2 (&pv)[16], uint32_t (&w)[16]) {
#pragma unroll
  for (int x = 0; x < 16; ++x) {
    const float4 n4 = nl[x / 2];                   // 16-byte broadcast loads: two pairs each
    const float2 n = (x & 1) ? make_float2(n4.z, n4.w) : make_float2(n4.x, n4.y);
    const float2 t = ptx::fma2(make_float2(__uint_as_float(sr[2 * x]), __uint_as_float(sr[2 * x + 1])), cc, n);
    float2 v = make_float2(ptx::ex2(t.x), ptx::ex2(t.y));
    if constexpr (MASK) {
      if (2 * x < first) v.x = 0.f;
      if (2 * x + 1 < first) v.y = 0.f;
    }
    pv[x] = v;
    w[x] = ptx::pack2<BF16>(v.x, v.y);
  }
}

// dS^T = P (dP - D) of one key row against 32 queries, packed (nd: the queries' -D pairs).
template <bool BF16>
__device__ __forceinline__ void dkdv_ds32(const uint32_t (&dr)[32], const float2 (&pv)[16], const float4* nd,
                                          uint32_t (&w)[16]) {
#pragma unroll
  for (int x = 0; x < 16; ++x) {
    const float4 n4 = nd[x / 2];
    const float2 n = (x & 1) ? make_float2(n4.z, n4.w) : make_float2(n4.x, n4.y);
    const float2 ds =
        ptx::mul2(pv[x], ptx::add2(make_float2(__uint_as_float(dr[2 * x]), __uint_as_float(dr[2 * x + 1])), n));
    w[x] = ptx::pack2<BF16>(ds.x, ds.y);
  }
}

// Writes COLS accumulator columns of one row, times `mul`, as 16-bit values at
// element offset `off` of `out`.
template <int COLS, bool BF16>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, float mul, void* out, size_t off, bool live) {
  uint32_t r[COLS / 32][32];
#pragma unroll
  for (int c = 0; c < COLS / 32; ++c) ptx::tmem_ld32(taddr + 32 * c, r[c]);
  ptx::tmem_wait_ld();
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + off);
#pragma unroll
  for (int c = 0; c < COLS / 32; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = ptx::pack2<BF16>(__uint_as_float(r[c][2 * i]) * mul, __uint_as_float(r[c][2 * i + 1]) * mul);
    if (live) {
      if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
        // 32-byte stores fill whole sectors: half as many scattered row writes, and
        // those slow the MMA issue of the steps they overlap
#pragma unroll
        for (int i = 0; i < 2; ++i) ptx::st_global_v8(dst + c * 4 + 2 * i, pk + 8 * i);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[c * 4 + i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  }
}

// The epilogue slice of one compute warp at d = 128: its 32 accumulator rows (TMEM lanes)
// x 64 columns from taddr, times `mul`, packed to 16 bits into 4 KB of a free ring slot
// laid out like a loaded tile (128-byte rows, 16-byte chunk c of row r at c ^ (r % 8)),
// which is the 128-byte swizzle of the store's tensor map.  Each lane writes its own row.
template <bool BF16>
__device__ __forceinline__ void stage_slice(uint32_t taddr, float mul, uint8_t* slice, int lane) {
  uint32_t r[2][32];
  ptx::tmem_ld32(taddr, r[0]);
  ptx::tmem_ld32(taddr + 32, r[1]);
  ptx::tmem_wait_ld();
  uint8_t* row = slice + lane * 128;
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {               // chunk 4c + kk: columns 32c + 8kk .. +7
      const uint32_t* x = r[c] + 8 * kk;
      const uint4 v = make_uint4(ptx::pack2<BF16>(__uint_as_float(x[0]) * mul, __uint_as_float(x[1]) * mul),
                                 ptx::pack2<BF16>(__uint_as_float(x[2]) * mul, __uint_as_float(x[3]) * mul),
                                 ptx::pack2<BF16>(__uint_as_float(x[4]) * mul, __uint_as_float(x[5]) * mul),
                                 ptx::pack2<BF16>(__uint_as_float(x[6]) * mul, __uint_as_float(x[7]) * mul));
      *reinterpret_cast<uint4*>(row + (((4 * c + kk) ^ (lane & 7)) << 4)) = v;
    }
  ptx::fence_proxy_async();
}

// Two such slices (dV and dK: the first unscaled, the second times `mul2`) with their
// four TMEM loads in flight at once.
template <bool BF16>
__device__ __forceinline__ void stage_slices(uint32_t ta1, uint32_t ta2, float mul2, uint8_t* s1, uint8_t* s2,
                                             int lane) {
  uint32_t r[4][32];
  ptx::tmem_ld32(ta1, r[0]);
  ptx::tmem_ld32(ta1 + 32, r[1]);
  ptx::tmem_ld32(ta2, r[2]);
  ptx::tmem_ld32(ta2 + 32, r[3]);
  ptx::tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint8_t* row = (c < 2 ? s1 : s2) + lane * 128;
    const float mul = c < 2 ? 1.f : mul2;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {               // chunk 4(c % 2) + kk: columns 32(c % 2) + 8kk .. +7
      const uint32_t* x = r[c] + 8 * kk;
      const uint4 v = make_uint4(ptx::pack2<BF16>(__uint_as_float(x[0]) * mul, __uint_as_float(x[1]) * mul),
                                 ptx::pack2<BF16>(__uint_as_float(x[2]) * mul, __uint_as_float(x[3]) * mul),
                                 ptx::pack2<BF16>(__uint_as_float(x[4]) * mul, __uint_as_float(x[5]) * mul),
                                 ptx::pack2<BF16>(__uint_as_float(x[6]) * mul, __uint_as_float(x[7]) * mul));
      *reinterpret_cast<uint4*>(row + (((4 * (c & 1) + kk) ^ (lane & 7)) << 4)) = v;
    }
  }
  ptx::fence_proxy_async();
}

// dV += P^T dO or dK += dS^T Q over a tile's 128 queries: A = P^T or dS^T packed in TMEM by
// the two compute threads of each key row (queries 0-63 at columns 0-31, 64-127 at columns
// 64-95), B = dO or Q as an MN-major operand (16 query rows, 2 KB, a step).
template <int D, Elem E, bool ACC, int KK = 0>
__device__ __forceinline__ void issue_t128(uint32_t tD, uint32_t tA, uint32_t b_lo, uint32_t lead) {
  using L = FwdCfg<D, E>;
  static_assert(!L::kFp8, "16-bit operands");
  if constexpr (KK < 8) {
    constexpr uint32_t idesc = ptx::idesc_make(kBlockM, D, L::kAbType, false, true);
    constexpr uint32_t desc_hi = ptx::sdesc_hi(1024);
    constexpr int kAcc = (ACC || KK > 0) ? 1 : 0;
    constexpr uint32_t kOt = 8 * KK + (KK >= 4 ? 32 : 0);
    constexpr uint32_t kOb = (KK * 16 * 128) >> 4;
    ptx::mma_f16_ts_oe<kAcc, kOt, kOb>(lead, tD, tA, b_lo, desc_hi, idesc);
    issue_t128<D, E, ACC, KK + 1>(tD, tA, b_lo, lead);
  }
}

// S = Q K^T or dP = dO V^T with A (Q or dO) packed in TMEM (16 elements of d, 8 columns, a
// step) and B a K-major K or V tile (N = 128 keys).
template <int D, Elem E, int KK = 0>
__device__ __forceinline__ void issue_ts_s(uint32_t tD, uint32_t tA, uint32_t b_lo, uint32_t lead) {
  using L = FwdCfg<D, E>;
  static_assert(!L::kFp8, "16-bit operands");
  if constexpr (KK < D / 16) {
    constexpr uint32_t idesc = ptx::idesc_make(kBlockM, kBlockN, L::kAbType, false, false);
    constexpr uint32_t desc_hi = ptx::sdesc_hi(1024);
    constexpr uint32_t kOb = ((KK * 32 / 128) * L::kAtomBytes + (KK * 32) % 128) >> 4;
    ptx::mma_f16_ts_oe<KK ? 1 : 0, 8 * KK, kOb>(lead, tD, tA, b_lo, desc_hi, idesc);
    issue_ts_s<D, E, KK + 1>(tD, tA, b_lo, lead);
  }
}

// A 128-row tile of shared memory (D elements a row, 128-byte swizzle atoms) into TMEM as an
// A operand (two 16-bit values a column, D / 2 columns at tD), by tcgen05.cp: one 32-byte
// K step (8 columns) a copy, in order before the MMAs issued after it.
template <int D, Elem E, int KK = 0>
__device__ __forceinline__ void copy_tile_tmem(uint32_t tD, uint32_t lo, uint32_t lead) {
  using L = FwdCfg<D, E>;
  if constexpr (KK < D / 16) {
    constexpr uint32_t desc_hi = ptx::sdesc_hi(1024);
    constexpr uint32_t kOb = ((KK * 32 / 128) * L::kAtomBytes + (KK * 32) % 128) >> 4;
    ptx::cp_128x256b_oe<kOb>(lead, tD + 8 * KK, lo, desc_hi);
    copy_tile_tmem<D, E, KK + 1>(tD, lo, lead);
  }
}

// ---------------------------------------------------------------------------- dq kernel

template <int D, Elem E>
__device__ __noinline__ void dq_producer(const BwdParams& p, uint32_t sbase, const ptx::WaitCtl& ctl) {
  using C = BwdCfg<D>;
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * i; };
  uint32_t nk = 0, nv = 0, units = 0;     // K and V loads issued so far, stationary fills
  // d = 128: bit b of `last` says K fill nk-1-b was its unit's last tile, whose slot then
  // holds that unit's epilogue staging; `epi` counts the epilogues waited for
  uint32_t last = 0, epi = 0;
  // the whole warp runs this loop converged (its waits included); one lane issues
  const bool lead = ptx::elect_one() != 0;
  int bh, i;
  for (int k = 0; bwd_unit_at(p, k, true, bh, i); ++k) {
    const int n = p.causal ? i + 1 : p.n_blk;
    if (!ptx::mbar_wait(bar(C::kStEmpty), (units & 1u) ^ 1u, ctl, 1u)) goto drain;
    if (lead) {
      ptx::mbar_arrive_expect_tx(bar(C::kStFull), 2 * C::kTile);
      load_tile<D, E>(&p.tm_q, sbase + C::kStatOff, bar(C::kStFull), i * 128, bh);
      load_tile<D, E>(&p.tm_do, sbase + C::kStatOff + C::kTile, bar(C::kStFull), i * 128, bh);
    }
    ++units;
    for (int j = 0; j < n; ++j) {
      const uint32_t ks = nk % C::kDqKSlots, kf = nk / C::kDqKSlots;
      static_assert(C::kDqKSlots == 3, "the history below spans three K fills");
      if (D == 128 && (last & 4u)) {
        if (!ptx::mbar_wait(bar(C::kEpiFree + epi % 3u), (epi / 3u) & 1u, ctl, 1u)) goto drain;
        ++epi;
      }
      last = ((last << 1) | (j + 1 == n ? 1u : 0u)) & 7u;
      if (!ptx::mbar_wait(bar(C::kKFree + ks), (kf & 1u) ^ 1u, ctl, 1u)) goto drain;
      if (lead) {
        ptx::mbar_arrive_expect_tx(bar(C::kKFull + ks), C::kTile);
        load_tile<D, E>(&p.tm_k, sbase + C::kDqKOff + ks * C::kTile, bar(C::kKFull + ks), j * 128, bh);
      }
      ++nk;
      const uint32_t vs = nv % C::kDqVSlots, vf = nv / C::kDqVSlots;
      if (!ptx::mbar_wait(bar(C::kVFree + vs), (vf & 1u) ^ 1u, ctl, 1u)) goto drain;
      if (lead) {
        ptx::mbar_arrive_expect_tx(bar(C::kVFull + vs), C::kTile);
        load_tile<D, E>(&p.tm_v, sbase + C::kDqVOff + vs * C::kTile, bar(C::kVFull + vs), j * 128, bh);
      }
      ++nv;
    }
  }
drain:
  // Copies still in flight must land before the CTA may exit: the last fill of every slot
  // issued so far (immediate on the normal path).
  for (uint32_t t = nk > static_cast<uint32_t>(C::kDqKSlots) ? nk - C::kDqKSlots : 0; t < nk; ++t)
    if (!ptx::mbar_wait_drain(bar(C::kKFull + t % C::kDqKSlots), (t / C::kDqKSlots) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, 8u);
  for (uint32_t t = nv > static_cast<uint32_t>(C::kDqVSlots) ? nv - C::kDqVSlots : 0; t < nv; ++t)
    if (!ptx::mbar_wait_drain(bar(C::kVFull + t % C::kDqVSlots), (t / C::kDqVSlots) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, 8u);
  if (units > 0 && !ptx::mbar_wait_drain(bar(C::kStFull), (units - 1u) & 1u, ctl.timeout_ns))
    atomicOr(ctl.status, 8u);
}

template <int D, Elem E>
__device__ __noinline__ void dq_mma(const BwdParams& p, uint32_t sbase, uint32_t tmem, const ptx::WaitCtl& ctl) {
  using C = BwdCfg<D>;
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * i; };
  const uint32_t lead = ptx::elect_one();   // the whole warp runs this loop, one lane issues
  constexpr uint32_t kTileDesc = C::kTile >> 4;
  const uint32_t k_lo0 = ptx::sdesc_lo(sbase + C::kDqKOff, 16);                 // K as K-major B of S
  const uint32_t kmn_lo0 = ptx::sdesc_lo(sbase + C::kDqKOff, v_lbo<D, E>());    // K as MN-major B of dQ
  const uint32_t v_lo0 = ptx::sdesc_lo(sbase + C::kDqVOff, 16);                 // V as K-major B of dP
  const uint32_t tQ = tmem + kQQ, tDO = tmem + kQDO, tS = tmem + kQS, tDP = tmem + kQDP, tAcc = tmem + kQAcc;
  const uint32_t q_lo = ptx::sdesc_lo(sbase + C::kStatOff, 16);                 // stationary Q
  const uint32_t do_lo = ptx::sdesc_lo(sbase + C::kStatOff + C::kTile, 16);     // stationary dO
  // S = Q K^T and dP = dO V^T for global tile number t, each with its commit; V's slot is
  // free once dP has run
  auto s_ = [&](uint32_t t) -> bool {
    const uint32_t ks = t % C::kDqKSlots;
    if (!ptx::mbar_wait(bar(C::kKFull + ks), (t / C::kDqKSlots) & 1u, ctl, 2u)) return false;
    ptx::tc_fence_after();
    issue_ts_s<D, E>(tS, tQ, k_lo0 + ks * kTileDesc, lead);
    ptx::mma_commit_e(lead, bar(C::kSdpFull));
    return true;
  };
  auto dp_ = [&](uint32_t t) -> bool {
    const uint32_t vs = t % C::kDqVSlots;
    if (!ptx::mbar_wait(bar(C::kVFull + vs), (t / C::kDqVSlots) & 1u, ctl, 2u)) return false;
    ptx::tc_fence_after();
    issue_ts_s<D, E>(tDP, tDO, v_lo0 + vs * kTileDesc, lead);
    ptx::mma_commit_e(lead, bar(C::kSdpFull + 1));
    ptx::mma_commit_e(lead, bar(C::kVFree + vs));
    return true;
  };
  // unit u's Q and dO into TMEM once they have landed in shared memory and unit u-1's
  // last S and dP (which read those columns) have completed; the copies run in order
  // before the products issued after them, and their commit frees the shared memory for
  // unit u+1's tiles
  auto copy_in = [&](uint32_t u) -> bool {
    if (!ptx::mbar_wait(bar(C::kStFull), u & 1u, ctl, 2u)) return false;
    if (u > 0 && !ptx::mbar_wait(bar(C::kQtFree), (u - 1u) & 1u, ctl, 2u)) return false;
    ptx::tc_fence_after();
    copy_tile_tmem<D, E>(tQ, q_lo, lead);
    copy_tile_tmem<D, E>(tDO, do_lo, lead);
    ptx::mma_commit_e(lead, bar(C::kStEmpty));
    return true;
  };
  uint32_t tile = 0, units = 0;
  int bh = 0, i = 0;
  bool have = bwd_unit_at(p, 0, true, bh, i);
  if (have && !copy_in(0)) goto done;
  for (int k = 0; have; ++k) {
    const int n = p.causal ? i + 1 : p.n_blk;
    if (!s_(tile) || !dp_(tile)) goto done;
    // Q and dO are free once the unit's last S and dP have run
    if (n == 1) ptx::mma_commit_e(lead, bar(C::kQtFree));
    // the next unit, worked out while these products run
    int bhn = 0, inext = 0;
    const bool more_units = bwd_unit_at(p, k + 1, true, bhn, inext);
    for (int j = 0; j < n; ++j, ++tile) {
      const bool more = j + 1 < n;
      // S(j) is in the compute threads' registers: S(j+1) goes into its columns
      if (!ptx::mbar_wait(bar(C::kSdpFree), tile & 1u, ctl, 2u)) goto done;
      if (more && !s_(tile + 1)) goto done;
      // the next unit's Q and dO go in as soon as this unit's last S and dP have completed,
      // ahead of its last dQ: the copies then overlap the compute threads' last dS
      if (!more && more_units && !copy_in(units + 1)) goto done;
      // dS(j) packed over the dP(j) columns: dQ += dS K_j, after which K_j's slot is free
      if (!ptx::mbar_wait(bar(C::kDsFull), tile & 1u, ctl, 2u)) goto done;
      ptx::tc_fence_after();
      const uint32_t ks = tile % C::kDqKSlots;
      if (j == 0) issue_t128<D, E, false>(tAcc, tDP, kmn_lo0 + ks * kTileDesc, lead);
      else issue_t128<D, E, true>(tAcc, tDP, kmn_lo0 + ks * kTileDesc, lead);
      ptx::mma_commit_e(lead, bar(C::kKFree + ks));
      // dP(j+1) into the columns dQ has just read
      if (more) {
        if (!dp_(tile + 1)) goto done;
        if (j + 2 == n) ptx::mma_commit_e(lead, bar(C::kQtFree));
      }
    }
    ptx::mma_commit_e(lead, bar(C::kAccFull));
    ++units;
    bh = bhn;
    i = inext;
    have = more_units;
  }
done:
  ptx::mma_commit_e(lead, bar(C::kMmaDone));
  if (!ptx::mbar_wait_drain(bar(C::kMmaDone), 0, ctl.timeout_ns)) atomicOr(ctl.status, 8u);
}

// P of 32 scores of one dq row: P = 2^(s * c + nl) with the row's nl = -LSE*log2(e); with
// MASK, keys x >= visible get P = 0.
template <bool MASK>
__device__ __forceinline__ void dq_p32(const uint32_t (&sr)[32], float2 cc, float2 nl, int visible, float2 (&pv)[16]) {
#pragma unroll
  for (int x = 0; x < 16; ++x) {
    const float2 t = ptx::fma2(make_float2(__uint_as_float(sr[2 * x]), __uint_as_float(sr[2 * x + 1])), cc, nl);
    float2 v = make_float2(ptx::ex2(t.x), ptx::ex2(t.y));
    if constexpr (MASK) {
      if (2 * x >= visible) v.x = 0.f;
      if (2 * x + 1 >= visible) v.y = 0.f;
    }
    pv[x] = v;
  }
}

// dS = P (dP - D) of 32 keys of one dq row, packed (nd = the row's -D in both halves).
template <bool BF16>
__device__ __forceinline__ void dq_ds32(const uint32_t (&dr)[32], const float2 (&pv)[16], float2 nd, uint32_t (&w)[16]) {
#pragma unroll
  for (int x = 0; x < 16; ++x) {
    const float2 ds =
        ptx::mul2(pv[x], ptx::add2(make_float2(__uint_as_float(dr[2 * x]), __uint_as_float(dr[2 * x + 1])), nd));
    w[x] = ptx::pack2<BF16>(ds.x, ds.y);
  }
}

template <int D, Elem E>
__device__ __forceinline__ void dq_compute(const BwdParams& p, uint32_t sbase, uint8_t* smem, uint32_t tmem,
                                           const ptx::WaitCtl& ctl) {
  using C = BwdCfg<D>;
  using L = FwdCfg<D, E>;
  constexpr bool kBf16 = E == Elem::BF16;
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * i; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int r = (warp & 3) * 32 + lane;                        // row in the Q tile = TMEM lane
  const int sub = warp >> 2;                                   // keys 64*sub .. +63 of each tile
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_base + kQS + 64 * sub, tDP = tmem + lane_base + kQDP + 64 * sub;
  const uint32_t tAcc = tmem + lane_base + kQAcc + (D / 2) * sub;
  const float2 cc = make_float2(p.scale_log2, p.scale_log2);
  uint32_t tile = 0, units = 0;
  uint32_t pend = 0;   // d = 128: 1 + the unit whose epilogue store may still read its staging
  int bh = 0, i = 0;
  float nl = 0.f, nd = 0.f;   // this row's -LSE*log2(e) and -D, loaded a unit ahead
  bool have = bwd_unit_at(p, 0, true, bh, i);
  if (have) {
    const size_t w0 = static_cast<size_t>(bh) * p.n_pad + i * 128 + r;
    nl = p.nlse2[w0];
    nd = p.ndelta[w0];
  }
  for (int k = 0; have; ++k) {
    const int n = p.causal ? i + 1 : p.n_blk;
    const int row = i * 128 + r;
    const float2 nl2 = make_float2(nl, nl), nd2 = make_float2(nd, nd);
    const int limit = min(p.N, p.causal ? row + 1 : p.N);      // keys >= limit get P = 0
    for (int j = 0; j < n; ++j, ++tile) {
      // P(j) as soon as S(j) is in
      bool got = ptx::mbar_wait(bar(C::kSdpFull), tile & 1u, ctl, 4u);
      if (!__all_sync(0xFFFFFFFFu, got)) return;
      ptx::tc_fence_after();
      uint32_t sr[2][32];
      ptx::tmem_ld32(tS, sr[0]);
      ptx::tmem_ld32(tS + 32, sr[1]);
      ptx::tmem_wait_ld();
      // S is read: the MMA thread may overwrite it with the next tile's
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::kSdpFree));
      const int visible = limit - (j * 128 + 64 * sub);
      float2 pv[2][16];
      if (visible >= 64) {
        dq_p32<false>(sr[0], cc, nl2, 0, pv[0]);
        dq_p32<false>(sr[1], cc, nl2, 0, pv[1]);
      } else {
        dq_p32<true>(sr[0], cc, nl2, visible, pv[0]);
        dq_p32<true>(sr[1], cc, nl2, visible - 32, pv[1]);
      }
      // dS(j) once dP(j) is in, packed over the dP columns this thread has read
      got = ptx::mbar_wait(bar(C::kSdpFull + 1), tile & 1u, ctl, 4u);
      if (!__all_sync(0xFFFFFFFFu, got)) return;
      ptx::tc_fence_after();
      uint32_t dr[2][32];
      ptx::tmem_ld32(tDP, dr[0]);
      ptx::tmem_ld32(tDP + 32, dr[1]);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[16];
        dq_ds32<kBf16>(dr[c], pv[c], nd2, w);
        ptx::tmem_st16(tDP + 16 * c, w);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::kDsFull));
      // the previous unit's epilogue store has long read its staging by now: hand the slot
      // back to the producer (it refills it for this unit's third tile at the earliest)
      if (D == 128 && pend != 0) {
        if (lane == 0) {
          ptx::bulk_wait_read<0>();
          ptx::mbar_arrive(bar(C::kEpiFree + (pend - 1) % 3u));
        }
        pend = 0;
      }
    }
    // the next unit's rows' -LSE*log2(e) and -D, loaded while the last dQ product runs
    int bhn = 0, inext = 0;
    const bool more = bwd_unit_at(p, k + 1, true, bhn, inext);
    if (more) {
      const size_t wn = static_cast<size_t>(bhn) * p.n_pad + inext * 128 + r;
      nl = p.nlse2[wn];
      nd = p.ndelta[wn];
    }
    const bool got = ptx::mbar_wait(bar(C::kAccFull), units & 1u, ctl, 4u);
    if (!__all_sync(0xFFFFFFFFu, got)) return;
    ptx::tc_fence_after();
    if constexpr (D == 128) {
      // dQ staged in the K slot of the unit's last tile (its products have run; the producer
      // refills it once the store below has read it), then one TMA store, and no wait here
      const uint32_t at = C::kDqKOff + ((tile - 1) % C::kDqKSlots) * C::kTile + sub * L::kAtomBytes +
                          (warp & 3) * 32 * 128;
      stage_slice<kBf16>(tAcc, p.scale, smem + at, lane);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const int row0 = i * 128 + (warp & 3) * 32;
        if (row0 < p.N) ptx::tma_store_3d(&p.tm_dq, sbase + at, 64 * sub, row0, bh);
        ptx::bulk_commit();
      }
      pend = units + 1;
      __syncwarp();
    } else {
      store_acc_row<D / 2, kBf16>(tAcc, p.scale, p.dq,
                                  (static_cast<size_t>(bh) * p.N + (row < p.N ? row : 0)) * D + (D / 2) * sub,
                                  row < p.N);
      ptx::tc_fence_before();
    }
    ++units;
    bh = bhn;
    i = inext;
    have = more;
  }
}

// ---------------------------------------------------------------------------- dkdv kernel

template <int D, Elem E>
__device__ __noinline__ void dkdv_producer(const BwdParams& p, uint32_t sbase, const ptx::WaitCtl& ctl) {
  using C = BwdCfg<D>;
  using L = FwdCfg<D, E>;
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * i; };
  uint32_t nd = 0, nq = 0, units = 0, vunits = 0;   // dO, Q, K and V fills issued so far
  // d = 128: bit b of `last` says fill nq-1-b was its unit's last tile, whose slots then hold
  // that unit's epilogue staging; `epi` counts the epilogues waited for
  uint32_t last = 0, epi = 0;
  // the whole warp runs this loop converged (its waits included); one lane issues
  const bool lead = ptx::elect_one() != 0;
  int bh, j;
  for (int k = 0; bwd_unit_at(p, k, false, bh, j); ++k) {
    const int i0 = p.causal ? j : 0;
    // the next unit's stationary tiles into L2 while this unit runs
    int bhn, jn;
    if (lead && bwd_unit_at(p, k + 1, false, bhn, jn)) {
#pragma unroll
      for (int a = 0; a < L::kAtoms; ++a) {
        ptx::tma_prefetch_3d(&p.tm_k, a * L::kAtomElems, jn * 128, bhn);
        ptx::tma_prefetch_3d(&p.tm_v, a * L::kAtomElems, jn * 128, bhn);
      }
    }
    // K once the previous unit's last S^T has run, V once its last dP^T has
    if (!ptx::mbar_wait(bar(C::kStEmpty), (units & 1u) ^ 1u, ctl, 1u)) goto drain;
    if (lead) {
      ptx::mbar_arrive_expect_tx(bar(C::kStFull), C::kTile);
      load_tile<D, E>(&p.tm_k, sbase + C::kStatOff, bar(C::kStFull), j * 128, bh);
    }
    ++units;
    if (!ptx::mbar_wait(bar(C::kVsEmpty), (vunits & 1u) ^ 1u, ctl, 1u)) goto drain;
    if (lead) {
      ptx::mbar_arrive_expect_tx(bar(C::kVsFull), C::kTile);
      load_tile<D, E>(&p.tm_v, sbase + C::kStatOff + C::kTile, bar(C::kVsFull), j * 128, bh);
    }
    ++vunits;
    for (int i = i0; i < p.n_blk; ++i) {
      // tile number nq == nd: its ring slot and the slot's fill count
      const uint32_t s = nq % kBwdStages, f = nq / kBwdStages;
      if (D == 128 && (last & 2u)) {
        if (!ptx::mbar_wait(bar(C::kEpiFree + epi % 3u), (epi / 3u) & 1u, ctl, 1u)) goto drain;
        ++epi;
      }
      last = ((last << 1) | (i + 1 == p.n_blk ? 1u : 0u)) & 3u;
      // Q first: S^T is the first product of a tile
      if (!ptx::mbar_wait(bar(C::kDone + s), (f & 1u) ^ 1u, ctl, 1u)) goto drain;
      if (lead) {
        ptx::mbar_arrive_expect_tx(bar(C::kReady + s), C::kTile + 2 * C::kVecBytes);
        load_tile<D, E>(&p.tm_q, sbase + C::kKvQOff + s * C::kTile, bar(C::kReady + s), i * 128, bh);
        const size_t w = static_cast<size_t>(bh) * p.n_pad + i * 128;
        const uint32_t vec = sbase + C::kKvVecOff + s * 2 * C::kVecBytes;
        ptx::bulk_load(vec, p.nlse2 + w, C::kVecBytes, bar(C::kReady + s));
        ptx::bulk_load(vec + C::kVecBytes, p.ndelta + w, C::kVecBytes, bar(C::kReady + s));
      }
      ++nq;
      if (!ptx::mbar_wait(bar(C::kDoFree + s), (f & 1u) ^ 1u, ctl, 1u)) goto drain;
      if (lead) {
        ptx::mbar_arrive_expect_tx(bar(C::kDoFull + s), C::kTile);
        load_tile<D, E>(&p.tm_do, sbase + C::kKvDoOff + s * C::kTile, bar(C::kDoFull + s), i * 128, bh);
      }
      ++nd;
    }
  }
drain:
  // Copies still in flight must land before the CTA may exit: the last fill of every slot
  // issued so far (immediate on the normal path)
  for (uint32_t t = nd > static_cast<uint32_t>(kBwdStages) ? nd - kBwdStages : 0; t < nd; ++t)
    if (!ptx::mbar_wait_drain(bar(C::kDoFull + t % kBwdStages), (t / kBwdStages) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, 8u);
  for (uint32_t t = nq > static_cast<uint32_t>(kBwdStages) ? nq - kBwdStages : 0; t < nq; ++t)
    if (!ptx::mbar_wait_drain(bar(C::kReady + t % kBwdStages), (t / kBwdStages) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, 8u);
  if (units > 0 && !ptx::mbar_wait_drain(bar(C::kStFull), (units - 1u) & 1u, ctl.timeout_ns))
    atomicOr(ctl.status, 8u);
  if (vunits > 0 && !ptx::mbar_wait_drain(bar(C::kVsFull), (vunits - 1u) & 1u, ctl.timeout_ns))
    atomicOr(ctl.status, 8u);
}

template <int D, Elem E>
__device__ __noinline__ void dkdv_mma(const BwdParams& p, uint32_t sbase, uint32_t tmem, const ptx::WaitCtl& ctl) {
  using C = BwdCfg<D>;
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * i; };
  const uint32_t lead = ptx::elect_one();   // the whole warp runs this loop, one lane issues
  constexpr uint32_t kTileDesc = C::kTile >> 4;
  const uint32_t k_lo = ptx::sdesc_lo(sbase + C::kStatOff, 16);                  // K as K-major A of S^T
  const uint32_t v_lo = ptx::sdesc_lo(sbase + C::kStatOff + C::kTile, 16);       // V as K-major A of dP^T
  const uint32_t q_lo0 = ptx::sdesc_lo(sbase + C::kKvQOff, 16);                  // Q as K-major B of S^T
  const uint32_t do_lo0 = ptx::sdesc_lo(sbase + C::kKvDoOff, 16);                // dO as K-major B of dP^T
  const uint32_t qmn_lo0 = ptx::sdesc_lo(sbase + C::kKvQOff, v_lbo<D, E>());     // Q as MN-major B of dK
  const uint32_t domn_lo0 = ptx::sdesc_lo(sbase + C::kKvDoOff, v_lbo<D, E>());   // dO as MN-major B of dV
  const uint32_t tS = tmem + kTmS, tDP = tmem + kTmDP, tDV = tmem + kTmAcc, tDK = tmem + kTmAcc + D;
  // S^T = K Q^T and dP^T = V dO^T of streamed tile t (N = 128), each with its commit
  auto st = [&](uint32_t t) -> bool {
    const uint32_t s = t % kBwdStages;
    if (!ptx::mbar_wait(bar(C::kReady + s), (t / kBwdStages) & 1u, ctl, 2u)) return false;
    ptx::tc_fence_after();
    issue_s<D, E>(tS, k_lo, q_lo0 + s * kTileDesc, lead);
    ptx::mma_commit_e(lead, bar(C::kSdpFull));
    return true;
  };
  auto dp = [&](uint32_t t) -> bool {
    const uint32_t s = t % kBwdStages;
    if (!ptx::mbar_wait(bar(C::kDoFull + s), (t / kBwdStages) & 1u, ctl, 2u)) return false;
    ptx::tc_fence_after();
    issue_s<D, E>(tDP, v_lo, do_lo0 + s * kTileDesc, lead);
    ptx::mma_commit_e(lead, bar(C::kSdpFull + 1));
    return true;
  };
  uint32_t tile = 0, units = 0;
  int bh = 0, j = 0;
  bool have = bwd_unit_at(p, 0, false, bh, j);
  for (int k = 0; have; ++k) {
    const int i0 = p.causal ? j : 0;
    // K is free once the unit's last S^T has run, V once its last dP^T has: the next
    // unit's loads overlap this unit's last products
    const bool one = i0 + 1 == p.n_blk;
    if (!ptx::mbar_wait(bar(C::kStFull), units & 1u, ctl, 2u)) goto done;
    if (!st(tile)) goto done;
    if (one) ptx::mma_commit_e(lead, bar(C::kStEmpty));
    if (!ptx::mbar_wait(bar(C::kVsFull), units & 1u, ctl, 2u)) goto done;
    if (!dp(tile)) goto done;
    if (one) ptx::mma_commit_e(lead, bar(C::kVsEmpty));
    // the next unit, worked out while these products run
    int bhn = 0, jn = 0;
    const bool more_units = bwd_unit_at(p, k + 1, false, bhn, jn);
    for (int i = i0; i < p.n_blk; ++i, ++tile) {
      const uint32_t s = tile % kBwdStages;
      const bool more = i + 1 < p.n_blk;
      // P^T(i) in TMEM: dV += P^T dO, then S^T(i+1) into the columns dV has just read
      if (!ptx::mbar_wait(bar(C::kDsFull + 1), tile & 1u, ctl, 2u)) goto done;
      ptx::tc_fence_after();
      if (i == i0) issue_t128<D, E, false>(tDV, tS, domn_lo0 + s * kTileDesc, lead);
      else issue_t128<D, E, true>(tDV, tS, domn_lo0 + s * kTileDesc, lead);
      ptx::mma_commit_e(lead, bar(C::kDoFree + s));
      if (more) {
        if (!st(tile + 1)) goto done;
        if (i + 2 == p.n_blk) ptx::mma_commit_e(lead, bar(C::kStEmpty));
      }
      // dS^T(i) in TMEM: dK += dS^T Q, then dP^T(i+1) into the columns dK has just read
      if (!ptx::mbar_wait(bar(C::kDsFull), tile & 1u, ctl, 2u)) goto done;
      ptx::tc_fence_after();
      if (i == i0) issue_t128<D, E, false>(tDK, tDP, qmn_lo0 + s * kTileDesc, lead);
      else issue_t128<D, E, true>(tDK, tDP, qmn_lo0 + s * kTileDesc, lead);
      ptx::mma_commit_e(lead, bar(C::kDone + s));
      if (more) {
        if (!dp(tile + 1)) goto done;
        if (i + 2 == p.n_blk) ptx::mma_commit_e(lead, bar(C::kVsEmpty));
      }
    }
    ptx::mma_commit_e(lead, bar(C::kAccFull));
    ++units;
    bh = bhn;
    j = jn;
    have = more_units;
  }
done:
  ptx::mma_commit_e(lead, bar(C::kMmaDone));
  if (!ptx::mbar_wait_drain(bar(C::kMmaDone), 0, ctl.timeout_ns)) atomicOr(ctl.status, 8u);
}

template <int D, Elem E>
__device__ __forceinline__ void dkdv_compute(const BwdParams& p, uint32_t sbase, uint8_t* smem, uint32_t tmem,
                                             const ptx::WaitCtl& ctl) {
  using C = BwdCfg<D>;
  using L = FwdCfg<D, E>;
  constexpr bool kBf16 = E == Elem::BF16;
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * i; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int kr = (warp & 3) * 32 + lane;                       // key row in the K/V tile = TMEM lane
  const int sub = warp >> 2;                                   // queries 64*sub .. +63 of each tile
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_base + kTmS + 64 * sub, tDP = tmem + lane_base + kTmDP + 64 * sub;
  const uint32_t tDV = tmem + lane_base + kTmAcc + (D / 2) * sub, tDK = tDV + D;
  const float2 cc = make_float2(p.scale_log2, p.scale_log2);
  uint32_t tile = 0, units = 0;
  uint32_t pend = 0;   // d = 128: 1 + the unit whose epilogue stores may still read its staging
  int bh = 0, j = 0;
  bool have = bwd_unit_at(p, 0, false, bh, j);
  for (int k = 0; have; ++k) {
    const int i0 = p.causal ? j : 0;
    const int key = j * 128 + kr;
    for (int i = i0; i < p.n_blk; ++i, ++tile) {
      const uint32_t s = tile % kBwdStages;
      // P^T(i) as soon as S^T(i) is in
      bool got = ptx::mbar_wait(bar(C::kSdpFull), tile & 1u, ctl, 4u);
      if (!__all_sync(0xFFFFFFFFu, got)) return;
      // the Q slot's vectors landed with Q itself, before S^T(i) could run (an
      // already-completed phase: this only orders the reads below after the copy)
      got = ptx::mbar_wait(bar(C::kReady + s), (tile / kBwdStages) & 1u, ctl, 4u);
      if (!__all_sync(0xFFFFFFFFu, got)) return;
      ptx::tc_fence_after();
      uint32_t sr[2][32];
      ptx::tmem_ld32(tS, sr[0]);
      ptx::tmem_ld32(tS + 32, sr[1]);
      const float* vec = reinterpret_cast<const float*>(smem + C::kKvVecOff + s * 2 * C::kVecBytes);
      const bool diag = p.causal && i == j;
      ptx::tmem_wait_ld();
      float2 pv[2][16];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int q0 = 64 * sub + 32 * c;                      // first query of this chunk
        const float4* nl = reinterpret_cast<const float4*>(vec + q0);   // 128-byte aligned
        uint32_t wp[16];
        // causal diagonal tile: query i*128 + q0 + x sees this key iff q0 + x >= kr (padded
        // queries have -LSE*log2(e) = -inf and so P = 0 already)
        if (diag) dkdv_p32<kBf16, true>(sr[c], cc, nl, kr - q0, pv[c], wp);
        else dkdv_p32<kBf16, false>(sr[c], cc, nl, 0, pv[c], wp);
        ptx::tmem_st16(tS + 16 * c, wp);                       // over S^T columns already read
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::kDsFull + 1));
      // the previous unit's epilogue stores have long read their staging by now: hand the
      // slots back to the producer (it refills them for this unit's second tile at the earliest)
      if (D == 128 && pend != 0) {
        if (lane == 0) {
          ptx::bulk_wait_read<0>();
          ptx::mbar_arrive(bar(C::kEpiFree + (pend - 1) % 3u));
        }
        pend = 0;
      }
      // dS^T(i) once dP^T(i) is in
      got = ptx::mbar_wait(bar(C::kSdpFull + 1), tile & 1u, ctl, 4u);
      if (!__all_sync(0xFFFFFFFFu, got)) return;
      ptx::tc_fence_after();
      uint32_t dr[2][32];
      ptx::tmem_ld32(tDP, dr[0]);
      ptx::tmem_ld32(tDP + 32, dr[1]);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int q0 = 64 * sub + 32 * c;
        const float4* nd = reinterpret_cast<const float4*>(vec + 128 + q0);
        uint32_t wd[16];
        dkdv_ds32<kBf16>(dr[c], pv[c], nd, wd);
        ptx::tmem_st16(tDP + 16 * c, wd);                      // over dP^T columns already read
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::kDsFull));
    }
    // the next unit, worked out while the last dK product runs (not after the epilogue)
    int bhn = 0, jn = 0;
    const bool more = bwd_unit_at(p, k + 1, false, bhn, jn);
    const bool got = ptx::mbar_wait(bar(C::kAccFull), units & 1u, ctl, 4u);
    if (!__all_sync(0xFFFFFFFFu, got)) return;
    ptx::tc_fence_after();
    if constexpr (D == 128) {
      // dV staged in the dO slot and dK in the Q slot of the unit's last tile (its products
      // have run; the producer refills the slots once the stores below have read them),
      // then one TMA store per accumulator: no scattered row stores, and no wait here
      const uint32_t sl = (tile - 1) % kBwdStages;
      const uint32_t slice = sub * L::kAtomBytes + (warp & 3) * 32 * 128;
      const uint32_t dv_at = C::kKvDoOff + sl * C::kTile + slice, dk_at = C::kKvQOff + sl * C::kTile + slice;
      stage_slices<kBf16>(tDV, tDK, p.scale, smem + dv_at, smem + dk_at, lane);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const int row0 = j * 128 + (warp & 3) * 32;
        if (row0 < p.N) {
          ptx::tma_store_3d(&p.tm_dv, sbase + dv_at, 64 * sub, row0, bh);
          ptx::tma_store_3d(&p.tm_dk, sbase + dk_at, 64 * sub, row0, bh);
        }
        ptx::bulk_commit();
      }
      pend = units + 1;
      __syncwarp();
    } else {
      const size_t off = (static_cast<size_t>(bh) * p.N + (key < p.N ? key : 0)) * D + (D / 2) * sub;
      store_acc_row<D / 2, kBf16>(tDV, 1.f, p.dv, off, key < p.N);
      store_acc_row<D / 2, kBf16>(tDK, p.scale, p.dk, off, key < p.N);
      ptx::tc_fence_before();
    }
    ++units;
    bh = bhn;
    j = jn;
    have = more;
  }
}

// ---------------------------------------------------------------------------- kernels

template <int D, Elem E, bool DKDV>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * i; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i)
      ptx::mbar_init(bar(i), (i == C::kDsFull || i == C::kDsFull + 1 || i == C::kSdpFree ||
                              (i >= C::kEpiFree && i < C::kEpiFree + 3))
                                 ? kBwdComputeWarps : 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == kBwdLoadWarp && lane == 0) {
    ptx::prefetch_tensormap(&p.tm_q);
    ptx::prefetch_tensormap(&p.tm_k);
    ptx::prefetch_tensormap(&p.tm_v);
    ptx::prefetch_tensormap(&p.tm_do);
  }
  if (warp == kBwdMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp == kBwdLoadWarp) {
    if constexpr (DKDV) dkdv_producer<D, E>(p, sbase, ctl);
    else dq_producer<D, E>(p, sbase, ctl);
  } else if (warp == kBwdMmaWarp) {
    if constexpr (DKDV) dkdv_mma<D, E>(p, sbase, tmem, ctl);
    else dq_mma<D, E>(p, sbase, tmem, ctl);
  } else {
    if constexpr (DKDV) dkdv_compute<D, E>(p, sbase, smem, tmem, ctl);
    else dq_compute<D, E>(p, sbase, smem, tmem, ctl);
    // the epilogues' TMA stores (issued by lane 0) complete before the CTA leaves
    if (D == 128 && lane == 0) ptx::bulk_wait<0>();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, Elem E>
cudaError_t launch_bwd_kernels(const BwdParams& p, int grid, cudaStream_t stream) {
  using C = BwdCfg<D>;
  constexpr bool kBf16 = E == Elem::BF16;
  const long long rows = static_cast<long long>(p.BH) * p.n_pad;
  const long long threads = rows * (D / 8);
  fa_bwd_prep_kernel<D, kBf16><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto dq = fa_bwd_kernel<D, E, false>;
  auto dkdv = fa_bwd_kernel<D, E, true>;
  for (auto k : {dq, dkdv}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc);
    if (e != cudaSuccess) return e;
  }
  dq<<<grid, kBwdThreads, C::kAlloc, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dkdv<<<grid, kBwdThreads, C::kAlloc, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(int d, bool bf16, const BwdParams& p, int grid, cudaStream_t stream) {
  if (d == 128)
    return bf16 ? launch_bwd_kernels<128, Elem::BF16>(p, grid, stream)
                : launch_bwd_kernels<128, Elem::F16>(p, grid, stream);
  return bf16 ? launch_bwd_kernels<64, Elem::BF16>(p, grid, stream)
              : launch_bwd_kernels<64, Elem::F16>(p, grid, stream);
}

}  // namespace fa
