// Attention forward with one 128-row Q tile per CTA and two CTAs per SM: f16/bf16,
// head dimension 64.
//
// The same computation as fa_fwd_kernel.cuh (tiling with an online softmax, the method
// of "FlashAttention 2 + 3 — speicherbewusste Attention-Kernels", "Kernpunkte" and
// "Begriffe auf dieser Seite"; asynchronous tile movement and a tensor pipe kept busy,
// the FlashAttention-3 news piece, "Drei technische Hebel").  At head dimension 64 a
// key step's MMAs take half as long as at 128, so the two-tile kernel waits on its
// softmax chain: S_t(j) -> softmax -> P_t(j) -> O_t += P_t V_j -> S_t(j+1), with both
// tiles' MMAs in one thread's issue order.  Here:
//   - each CTA holds one Q tile, and P has TMEM columns of its own, so S(j+1) is issued
//     as soon as the softmax has read S(j) into registers: the next scores are ready
//     when the softmax finishes P(j);
//   - two CTAs share each SM (256 TMEM columns each), so the tensor pipe interleaves two
//     chains whose issue orders do not wait on each other.
//
// TMEM (256 columns): S (128 fp32 columns) | P (64: 128 keys as 16-bit pairs) | O (64).
// Roles (192 threads): warps 0-3 softmax (thread = row of the Q tile = TMEM lane), warp 4
// TMA producer, warp 5 MMA issuer and TMEM owner; the producer and issuer run their loops
// on the whole warp, one elected lane issuing.
// Shared memory: two Q buffers (the next unit's Q lands while this one runs) and a ring
// of K/V tiles, loaded in the order K_0, K_1, V_0, K_2, V_1, ... in which the MMAs use
// them.  Every wait is bounded, as in the two-tile kernel.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kThreads1 = 192;
constexpr int kLoadWarp1 = 4;
constexpr int kMmaWarp1 = 5;

template <Elem E>
struct Fwd1Cfg {
  static_assert(E != Elem::E4M3, "16-bit inputs");
  static constexpr int D = 64;
  static constexpr bool kBf16Out = E != Elem::F16;
  static constexpr int kTileBytes = kBlockM * D * 2;       // one 128-byte swizzle atom: 16 KB
  static constexpr int kStages = 4;                        // K/V ring slots (two key steps)
  static constexpr int kQOff = 0;                          // two Q buffers
  static constexpr int kKVOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  // Q buffers full / free; K/V slots full / free; S in (commit); S read into registers
  // (softmax arrives); P written (softmax arrives); O += P V done (commit); all MMAs done
  static constexpr int kQFull = 0, kQEmpty = 2, kFull = 4, kEmpty = 4 + kStages;
  static constexpr int kSFull = 4 + 2 * kStages, kSFree = kSFull + 1, kPFull = kSFree + 1;
  static constexpr int kPvDone = kPFull + 1, kMmaDone = kPvDone + 1;
  static constexpr int kNumBars = kMmaDone + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM base slot, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;             // room to align the base to 1 KB
  // two CTAs a SM, and never three (three would wait on each other's TMEM)
  static_assert(2 * kAlloc <= 233472 && 3 * kAlloc > 233472, "two CTAs per SM");
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kTmS = 0, kTmP = 128, kTmO = 192;
};

// Key tiles the 128-row Q tile qb attends to.
__device__ __forceinline__ int tile_nkv1(const FwdParams& p, int qb) {
  const int nkv = (p.N + kBlockN - 1) / kBlockN;
  return p.causal ? min(nkv, qb + 1) : nkv;
}

// Load i of a unit with n key tiles: K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}
// (the inverse of k_pos / v_pos).
__device__ __forceinline__ void kv_load(int i, int n, bool& is_k, int& jj) {
  if (i == 0) {
    is_k = true;
    jj = 0;
  } else if ((i & 1) && (i + 1) / 2 < n) {
    is_k = true;
    jj = (i + 1) / 2;
  } else if (i & 1) {
    is_k = false;
    jj = n - 1;
  } else {
    is_k = false;
    jj = (i - 2) / 2;
  }
}

// ---------------------------------------------------------------------------- producer

template <Elem E>
__device__ __noinline__ void fwd1_producer(const FwdParams& p, uint32_t sbase, const ptx::WaitCtl& ctl) {
  using L = Fwd1Cfg<E>;
  auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
  const bool lead = ptx::elect_one() != 0;   // the whole warp runs the loop; one lane issues
  uint32_t nl = 0;                           // K/V loads so far: ring position
  uint32_t units = 0;                        // Q loads so far
  int bh, qb;
  for (int k = 0; unit_at(p, k, bh, qb); ++k) {
    const int n = tile_nkv1(p, qb);
    // Q into buffer units % 2, once the unit two back has run its last S
    const uint32_t qbuf = units & 1u;
    if (!ptx::mbar_wait(bar(L::kQEmpty + qbuf), ((units >> 1) & 1u) ^ 1u, ctl, kStatusLoadTimeout)) goto drain;
    if (lead) {
      ptx::mbar_arrive_expect_tx(bar(L::kQFull + qbuf), L::kTileBytes);
      ptx::tma_load_3d(sbase + L::kQOff + qbuf * L::kTileBytes, &p.tm_q, bar(L::kQFull + qbuf), 0,
                       qb * kBlockM, bh);
    }
    ++units;
    {
      // Q is read once: start the next unit's on its way into L2 a unit ahead
      int bhn, qbn;
      if (lead && unit_at(p, k + 1, bhn, qbn)) ptx::tma_prefetch_3d(&p.tm_q, 0, qbn * kBlockM, bhn);
    }
    for (int i = 0; i < 2 * n; ++i, ++nl) {
      bool is_k;
      int jj;
      kv_load(i, n, is_k, jj);
      const uint32_t s = nl % L::kStages, f = nl / L::kStages;
      if (!ptx::mbar_wait(bar(L::kEmpty + s), (f & 1u) ^ 1u, ctl, kStatusLoadTimeout)) goto drain;
      // test hook: load number dbg_skip_load is left out (its consumer's wait runs out)
      const bool skip = p.dbg_skip_load >= 0 && static_cast<uint32_t>(p.dbg_skip_load) == nl;
      if (lead && !skip) {
        ptx::mbar_arrive_expect_tx(bar(L::kFull + s), L::kTileBytes);
        ptx::tma_load_3d(sbase + L::kKVOff + s * L::kTileBytes, is_k ? &p.tm_k : &p.tm_v, bar(L::kFull + s), 0,
                         jj * kBlockN, bh);
      }
    }
  }
drain:
  // Copies in flight must land before the CTA may exit: the last load of every slot and
  // of both Q buffers (immediate on the normal path)
  for (uint32_t t = nl > static_cast<uint32_t>(L::kStages) ? nl - L::kStages : 0; t < nl; ++t) {
    if (p.dbg_skip_load >= 0 && static_cast<uint32_t>(p.dbg_skip_load) == t) continue;
    if (!ptx::mbar_wait_drain(bar(L::kFull + t % L::kStages), (t / L::kStages) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, kStatusDrainTimeout);
  }
  for (uint32_t u = units > 2u ? units - 2u : 0u; u < units; ++u)
    if (!ptx::mbar_wait_drain(bar(L::kQFull + (u & 1u)), (u >> 1) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, kStatusDrainTimeout);
}

// ---------------------------------------------------------------------------- MMA issuer

// Over all the CTA's key steps g in order (unit by unit): S(g+1) as soon as the softmax has
// read S(g) (the next unit's first S after a unit's last), then O += P(g) V once the
// softmax has written P(g).  S(g+1) thus runs while the softmax works on S(g), and the
// P.V of step g while it works on S(g+1).
template <Elem E>
__device__ __noinline__ void fwd1_mma(const FwdParams& p, uint32_t sbase, uint32_t tmem, const ptx::WaitCtl& ctl) {
  using L = Fwd1Cfg<E>;
  auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
  const uint32_t lead = ptx::elect_one();    // the whole warp runs the loop; one lane issues
  constexpr uint32_t kSlotDesc = L::kTileBytes >> 4;
  const uint32_t q_lo0 = ptx::sdesc_lo(sbase + L::kQOff, 16);
  const uint32_t k_lo0 = ptx::sdesc_lo(sbase + L::kKVOff, 16);
  const uint32_t v_lo0 = ptx::sdesc_lo(sbase + L::kKVOff, v_lbo<64, E>());
  const uint32_t tS = tmem + L::kTmS, tP = tmem + L::kTmP, tO = tmem + L::kTmO;
  // S = Q K^T from Q buffer qbuf and the K tile of ring load `load`, with its commits
  auto s_mma = [&](uint32_t qbuf, uint32_t load) -> bool {
    const uint32_t s = load % L::kStages;
    if (!ptx::mbar_wait(bar(L::kFull + s), (load / L::kStages) & 1u, ctl, kStatusMmaTimeout)) return false;
    ptx::tc_fence_after();
    issue_s<64, E>(tS, q_lo0 + qbuf * kSlotDesc, k_lo0 + s * kSlotDesc, lead);
    ptx::mma_commit_e(lead, bar(L::kSFull));
    ptx::mma_commit_e(lead, bar(L::kEmpty + s));
    return true;
  };
  uint32_t g = 0;        // key steps issued so far (S and P.V alike)
  uint32_t base = 0;     // ring position of the current unit's first load
  uint32_t units = 0;
  int bh = 0, qb = 0;
  bool have = unit_at(p, 0, bh, qb);
  int n = have ? tile_nkv1(p, qb) : 0;
  if (have) {
    if (!ptx::mbar_wait(bar(L::kQFull), 0u, ctl, kStatusMmaTimeout)) goto done;
    if (!s_mma(0u, 0u)) goto done;
    if (n == 1) ptx::mma_commit_e(lead, bar(L::kQEmpty));
  }
  for (int k = 0; have; ++k) {
    const uint32_t qbuf = units & 1u;
    int bhn = 0, qbn = 0;
    const bool has_next = unit_at(p, k + 1, bhn, qbn);
    const int nn = has_next ? tile_nkv1(p, qbn) : 0;
    for (int j = 0; j < n; ++j, ++g) {
      // the next S, into the columns the softmax has just read
      if (j + 1 < n || has_next) {
        if (!ptx::mbar_wait(bar(L::kSFree), g & 1u, ctl, kStatusMmaTimeout)) goto done;
        if (j + 1 < n) {
          if (!s_mma(qbuf, base + k_pos(j + 1))) goto done;
          if (j + 2 == n) ptx::mma_commit_e(lead, bar(L::kQEmpty + qbuf));   // its last S
        } else {
          const uint32_t nbuf = qbuf ^ 1u;
          if (!ptx::mbar_wait(bar(L::kQFull + nbuf), ((units + 1u) >> 1) & 1u, ctl, kStatusMmaTimeout)) goto done;
          if (!s_mma(nbuf, base + 2u * n)) goto done;
          if (nn == 1) ptx::mma_commit_e(lead, bar(L::kQEmpty + nbuf));
        }
      }
      // O += P(g) V_j once P(g) is in TMEM
      if (!ptx::mbar_wait(bar(L::kPFull), g & 1u, ctl, kStatusMmaTimeout)) goto done;
      const uint32_t vl = base + v_pos(j, n), vs = vl % L::kStages;
      if (!ptx::mbar_wait(bar(L::kFull + vs), (vl / L::kStages) & 1u, ctl, kStatusMmaTimeout)) goto done;
      ptx::tc_fence_after();
      if (j == 0) issue_pv<64, E, false>(tO, tP, v_lo0 + vs * kSlotDesc, lead);
      else issue_pv<64, E, true>(tO, tP, v_lo0 + vs * kSlotDesc, lead);
      ptx::mma_commit_e(lead, bar(L::kPvDone));
      ptx::mma_commit_e(lead, bar(L::kEmpty + vs));
    }
    base += 2u * n;
    ++units;
    have = has_next;
    bh = bhn;
    qb = qbn;
    n = nn;
  }
done:
  // Every MMA issued so far must finish before TMEM is released.
  ptx::mma_commit_e(lead, bar(L::kMmaDone));
  if (!ptx::mbar_wait_drain(bar(L::kMmaDone), 0, ctl.timeout_ns)) atomicOr(ctl.status, kStatusDrainTimeout);
}

// ---------------------------------------------------------------------------- softmax

// Warps 0-3: thread r owns row r of the CTA's Q tile (TMEM lane r).  Per key step it reads
// S into registers and hands the columns back at once, forms P with the online softmax
// (the running maximum moves only when it grows past kRescaleThreshold), waits for the
// previous P.V before writing P and rescaling O, and at the end of a unit writes
// O / l and the LSE.
template <Elem E>
__device__ __forceinline__ void fwd1_softmax(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                             const ptx::WaitCtl& ctl) {
  using L = Fwd1Cfg<E>;
  auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
  const int r = threadIdx.x;
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = static_cast<uint32_t>(threadIdx.x / 32) * 32u;
  const uint32_t tS = tmem + (lane_base << 16) + L::kTmS;
  const uint32_t tP = tmem + (lane_base << 16) + L::kTmP;
  const uint32_t tO = tmem + (lane_base << 16) + L::kTmO;
  const float sl2 = p.scale_log2;
  const float2 f2 = make_float2(sl2, sl2);
  const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
  uint32_t g = 0;    // key steps so far
  int bh, qb;
  for (int k = 0; unit_at(p, k, bh, qb); ++k) {
    const int n = tile_nkv1(p, qb);
    const int r0 = qb * kBlockM;
    const int row = r0 + r;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < n; ++j, ++g) {
      bool got = ptx::mbar_wait(bar(L::kSFull), g & 1u, ctl, kStatusSoftmaxTimeout);
      if (!__all_sync(0xFFFFFFFFu, got)) return;
      ptx::tc_fence_after();
      uint32_t sr[4][32];
#define S_(c) __uint_as_float(sr[(c) / 32][(c) % 32])
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + 32 * c, sr[c]);
      ptx::tmem_wait_ld();
      // S is in registers: the MMA thread may issue the next S into its columns
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(L::kSFree));

      const int col0 = j * kBlockN;
      if (col0 + kBlockN > p.N || (p.causal && col0 + kBlockN - 1 > r0)) {
        // columns c >= visible are masked (past N, or past the diagonal)
        const int visible = (p.causal ? min(p.N, row + 1) : p.N) - col0;
#pragma unroll
        for (int c = 0; c < kBlockN; ++c)
          if (c >= visible) sr[c / 32][c % 32] = __float_as_uint(-INFINITY);
      }
      // row maximum: 3-input max trees, four chains per 64-column half
      float mh[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float acc[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int b = 64 * h + 16 * a;
          float x = ptx::max3(S_(b), S_(b + 1), S_(b + 2));
#pragma unroll
          for (int i = 3; i < 15; i += 2) x = ptx::max3(x, S_(b + i), S_(b + i + 1));
          acc[a] = fmaxf(x, S_(b + 15));
        }
        mh[h] = ptx::max3(acc[0], acc[1], fmaxf(acc[2], acc[3]));
      }
      const float m_new = fmaxf(m, fmaxf(mh[0], mh[1]) * sl2);
      float m_use, alpha = 1.f;
      bool rescale_o = false;
      if (j == 0) {
        m_use = (m_new == -INFINITY) ? 0.f : m_new;
      } else {
        const bool need = m_new > m + kRescaleThreshold;
        m_use = need ? m_new : m;
        alpha = need ? ptx::ex2(m - m_new) : 1.f;
        rescale_o = __any_sync(0xFFFFFFFFu, need);
      }
      // P = 2^(s * scale * log2(e) - m) in packed pairs, packed to 16 bits over the scores
      // already consumed; row sums in four packed accumulators per half
      const float2 nb = make_float2(-m_use, -m_use);
      float sum = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int c = 64 * h + 4 * q;
          const float2 x01 = ptx::fma2(make_float2(S_(c), S_(c + 1)), f2, nb);
          const float2 x23 = ptx::fma2(make_float2(S_(c + 2), S_(c + 3)), f2, nb);
          const float2 p01 = make_float2(ptx::ex2(x01.x), ptx::ex2(x01.y));
          const float2 p23 = make_float2(ptx::ex2(x23.x), ptx::ex2(x23.y));
          acc[q & 3] = ptx::add2(acc[q & 3], ptx::add2(p01, p23));
          sr[(c / 2) / 32][(c / 2) % 32] = ptx::pack2<L::kBf16Out>(p01.x, p01.y);
          sr[(c / 2 + 1) / 32][(c / 2 + 1) % 32] = ptx::pack2<L::kBf16Out>(p23.x, p23.y);
        }
        const float2 t = ptx::add2(ptx::add2(acc[0], acc[1]), ptx::add2(acc[2], acc[3]));
        sum += t.x + t.y;
      }
#undef S_
      l = l * alpha + sum;
      if (j > 0) {
        // the previous P.V has read P and added into O: both may change now
        got = ptx::mbar_wait(bar(L::kPvDone), (g - 1u) & 1u, ctl, kStatusSoftmaxTimeout);
        if (!__all_sync(0xFFFFFFFFu, got)) return;
        ptx::tc_fence_after();
      }
      if (rescale_o) {
        // both 32-column chunks of O in one TMEM round trip
        uint32_t orr[2][32];
        ptx::tmem_ld32(tO, orr[0]);
        ptx::tmem_ld32(tO + 32, orr[1]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 v = ptx::mul2(make_float2(__uint_as_float(orr[h][i]), __uint_as_float(orr[h][i + 1])),
                                       make_float2(alpha, alpha));
            orr[h][i] = __float_as_uint(v.x);
            orr[h][i + 1] = __float_as_uint(v.y);
          }
        ptx::tmem_st32(tO, orr[0]);
        ptx::tmem_st32(tO + 32, orr[1]);
      }
      ptx::tmem_st32(tP, sr[0]);
      ptx::tmem_st32(tP + 32, sr[1]);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(L::kPFull));
      m = m_use;
    }

    // epilogue, once the unit's last P.V is done: O = O_acc / l, LSE = ln 2 * (m + log2 l)
    const bool got = ptx::mbar_wait(bar(L::kPvDone), (g - 1u) & 1u, ctl, kStatusSoftmaxTimeout);
    if (!__all_sync(0xFFFFFFFFu, got)) return;
    ptx::tc_fence_after();
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    const bool live = row < p.N;
    uint32_t pk[32];
    {
      uint32_t orr[2][32];
      ptx::tmem_ld32(tO, orr[0]);
      ptx::tmem_ld32(tO + 32, orr[1]);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 v = ptx::mul2(
            make_float2(__uint_as_float(orr[i / 16][(2 * i) % 32]), __uint_as_float(orr[i / 16][(2 * i + 1) % 32])),
            make_float2(inv_l, inv_l));
        pk[i] = ptx::pack2<L::kBf16Out>(v.x, v.y);
      }
    }
    // O is read: the next unit's first P.V may overwrite it (it waits for the next P)
    ptx::tc_fence_before();
    if (live) {
      uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + (static_cast<size_t>(bh) * p.N + row) * 64);
      if (o_v8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ptx::st_global_v8(orow + 2 * i, pk + 8 * i);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) orow[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
      if (p.lse != nullptr)
        p.lse[static_cast<size_t>(bh) * p.N + row] = l > 0.f ? (m + ptx::lg2(l)) * kLn2 : -INFINITY;
    }
  }
}

// ---------------------------------------------------------------------------- kernel

template <Elem E>
__global__ void __launch_bounds__(kThreads1, 2) fa_fwd1_kernel(const __grid_constant__ FwdParams p) {
  using L = Fwd1Cfg<E>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i) ptx::mbar_init(bar(i), (i == L::kSFree || i == L::kPFull) ? 4 : 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == kLoadWarp1 && lane == 0) {
    ptx::prefetch_tensormap(&p.tm_q);
    ptx::prefetch_tensormap(&p.tm_k);
    ptx::prefetch_tensormap(&p.tm_v);
  }
  if (warp == kMmaWarp1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), L::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp == kLoadWarp1) fwd1_producer<E>(p, sbase, ctl);
  else if (warp == kMmaWarp1) fwd1_mma<E>(p, sbase, tmem, ctl);
  else fwd1_softmax<E>(p, sbase, tmem, ctl);

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace fa
