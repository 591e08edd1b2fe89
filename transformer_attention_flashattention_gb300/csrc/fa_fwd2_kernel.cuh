// Attention forward on CTA pairs (tcgen05 cta_group::2), f16/bf16, head dim 128.
//
// The same computation as fa_fwd_kernel.cuh (tiling with an online softmax, the method
// of "FlashAttention 2 + 3 — speicherbewusste Attention-Kernels", "Kernpunkte" and
// "Begriffe auf dieser Seite"), with the larger MMA tile the FlashAttention-3 news
// piece's levers point at ("Drei technische Hebel", items 1-2: asynchronous tile
// movement, keeping the tensor cores busy): a cluster of two CTAs on two SMs computes
// each 256-row Q tile with M = 256 MMAs issued by one thread of the even CTA.
//
// Split of the operands between the pair (rank r = 0 leader, 1 follower):
//   Q     each CTA holds its own 128 rows of the pair's 256-row tile (the A operand);
//   K_j   each CTA holds 64 of the tile's 128 keys (B of S = Q K^T is split along N);
//   V_j   each CTA holds 64 of the d = 128 columns (B of O += P V is split along N);
//   S, O  each CTA's TMEM holds its 128 rows x all columns; P is written to the
//         follower's TMEM by its own softmax warps and read from there by the MMA.
// Per SM that halves the K/V shared memory of a tile (16 KB of each instead of 32), so
// the ring holds ten 16 KB slots.
//
// Synchronisation between the two CTAs (every wait bounded, as in the 1-CTA kernel):
//   - each CTA loads its halves with TMA against its own barriers; the follower's MMA
//     warp, idle otherwise, relays each landed step and Q tile to the leader's barrier
//     (remote mbarrier arrive), so every copy is drained by the CTA it writes to;
//   - the follower's softmax warps arrive on the leader's P barrier remotely;
//   - the leader's commits multicast to both CTAs (S ready, O ready, slots free);
//   - TMEM is allocated and freed by one warp of each CTA together (cta_group::2).
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kPairRows = 2 * kBlockM;            // rows of one M = 256 tile of the pair
constexpr int kUnitRows2 = kQTiles * kPairRows;   // rows of one work unit of the pair

template <Elem E>
struct Fwd2Cfg {
  static_assert(E != Elem::E4M3, "16-bit inputs");
  static constexpr int D = 128;
  static constexpr uint32_t kAbType = (E == Elem::BF16) ? 1u : 0u;
  static constexpr bool kBf16Out = E != Elem::F16;
  static constexpr int kQTileBytes = kBlockM * D * 2;     // this CTA's 128 Q rows: 32 KB, 2 atoms
  static constexpr int kQAtomBytes = kBlockM * 128;       // 16 KB
  static constexpr int kSlotBytes = 16384;                // half a K tile or half a V tile
  static constexpr int kKAtomBytes = 64 * 128;            // 64 keys x 128 bytes of d
  static constexpr int kStages = 10;
  static constexpr int kSteps = 16;
  static_assert(kSteps > kStages, "step ring must outlast the load ring");
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQTiles * kQTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kSlotBytes;
  static constexpr int kQFull = 0, kQEmpty = 2, kReady = 4, kDone = 4 + kSteps;
  static constexpr int kSFull = 4 + 2 * kSteps, kPFull = kSFull + 2, kOFull = kPFull + 2;
  static constexpr int kMmaDone = kOFull + 2;
  static constexpr int kNumBars = kMmaDone + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemS = 0, kTmemO = 256;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// The k-th (b*h, 512-row q-block) unit of this CTA pair (cluster); the same sequence as
// unit_at, dealt over clusters instead of CTAs.
__device__ __forceinline__ bool unit_at2(const FwdParams& p, int k, int& bh, int& qb) {
  const int G = static_cast<int>(gridDim.x) >> 1, c = static_cast<int>(blockIdx.x) >> 1;
  if (!p.causal) {
    const int u = c + k * G;
    if (u >= p.num_units) return false;
    bh = u / p.n_qblk;
    qb = u % p.n_qblk;
    return true;
  }
  return causal_unit(G, c, p.BH, p.n_qblk, k, true, bh, qb);
}

// Key tiles the pair's 256-row tile t of q-block qb needs (0 if it lies past N).  Both
// CTAs take this many S tiles; under the causal mask the leader's rows see the last one
// fully masked.
__device__ __forceinline__ int tile_nkv2(const FwdParams& p, int qb, int t) {
  const int r0 = qb * kUnitRows2 + t * kPairRows;
  if (r0 >= p.N) return 0;
  const int nkv = (p.N + kBlockN - 1) / kBlockN;
  return p.causal ? min(nkv, min(p.N - 1, r0 + kPairRows - 1) / kBlockN + 1) : nkv;
}

// ---------------------------------------------------------------------------- producer

// Both CTAs: this CTA's halves of K_j and V_{j-1} per step, and its Q rows, against its
// own barriers (the loads of a step complete on that step's ready barrier).
template <Elem E>
__device__ __noinline__ void fwd2_producer(const FwdParams& p, uint32_t sbase, uint32_t rank,
                                           const ptx::WaitCtl& ctl) {
  using L = Fwd2Cfg<E>;
  auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
  uint32_t load_idx = 0, step = 0;
  uint32_t q_fills[kQTiles] = {0, 0};
  uint32_t slot_step[L::kStages];
#pragma unroll
  for (int s = 0; s < L::kStages; ++s) slot_step[s] = 0;
  uint32_t armed = 0;
  const int qrow = static_cast<int>(rank) * kBlockM;

  int bh, qb;
  for (int k = 0; unit_at2(p, k, bh, qb); ++k) {
    const int n0 = tile_nkv2(p, qb, 0), n1 = tile_nkv2(p, qb, 1);
    const int n = max(n0, n1);
    {
      int bhn, qbn;
      if (unit_at2(p, k + 1, bhn, qbn)) {
#pragma unroll
        for (int t = 0; t < kQTiles; ++t)
          if (tile_nkv2(p, qbn, t) > 0)
#pragma unroll
            for (int a = 0; a < 2; ++a)
              ptx::tma_prefetch_3d(&p.tm_q, a * 64, qbn * kUnitRows2 + t * kPairRows + qrow, bhn);
      }
    }
    for (int j = 0; j <= n; ++j, ++step) {
      const uint32_t cnt = (j < n ? 1u : 0u) + (j >= 1 ? 1u : 0u);
      const uint32_t bit = 1u << (step % L::kSteps);
      const uint32_t rb = bar(L::kReady + step % L::kSteps);
      armed &= ~bit;
      for (uint32_t i = 0; i < cnt; ++i) {
        const uint32_t slot = (load_idx + i) % L::kStages;
        const uint32_t prev = slot_step[slot];
        if (prev != 0 && !ptx::mbar_wait(bar(L::kDone + (prev - 1) % L::kSteps),
                                         ((prev - 1) / L::kSteps) & 1u, ctl, kStatusLoadTimeout)) {
          if (i > 0) {
            ptx::mbar_arrive(rb);
            armed |= bit;
          }
          goto drain;
        }
        if (i + 1 < cnt) ptx::mbar_expect_tx(rb, L::kSlotBytes);
        else ptx::mbar_arrive_expect_tx(rb, L::kSlotBytes);
        const bool is_k = i == 0 && j < n;
        const uint32_t dst = sbase + L::kKVOff + slot * L::kSlotBytes;
        if (is_k) {
          // keys 128 j + 64 r .. +63, both 64-wide d atoms
#pragma unroll
          for (int a = 0; a < 2; ++a)
            ptx::tma_load_3d(dst + a * L::kKAtomBytes, &p.tm_kh, rb, a * 64, j * kBlockN + 64 * static_cast<int>(rank),
                             bh);
        } else {
          // d columns 64 r .. +63 of all 128 keys of V_{j-1}
          ptx::tma_load_3d(dst, &p.tm_v, rb, 64 * static_cast<int>(rank), (j - 1) * kBlockN, bh);
        }
        slot_step[slot] = step + 1;
      }
      armed |= bit;
      load_idx += cnt;
      if (j == 0) {
#pragma unroll
        for (int t = 0; t < kQTiles; ++t) {
          if ((t == 0 ? n0 : n1) == 0) continue;
          if (!ptx::mbar_wait(bar(L::kQEmpty + t), (q_fills[t] & 1u) ^ 1u, ctl, kStatusLoadTimeout)) goto drain;
          ptx::mbar_arrive_expect_tx(bar(L::kQFull + t), L::kQTileBytes);
#pragma unroll
          for (int a = 0; a < 2; ++a)
            ptx::tma_load_3d(sbase + L::kQOff + t * L::kQTileBytes + a * L::kQAtomBytes, &p.tm_q, bar(L::kQFull + t),
                             a * 64, qb * kUnitRows2 + t * kPairRows + qrow, bh);
          ++q_fills[t];
        }
      }
    }
  }
drain:
  for (uint32_t g = step > static_cast<uint32_t>(L::kSteps) ? step - L::kSteps : 0; g < step; ++g)
    if (((armed >> (g % L::kSteps)) & 1u) &&
        !ptx::mbar_wait_drain(bar(L::kReady + g % L::kSteps), (g / L::kSteps) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, kStatusDrainTimeout);
  for (int t = 0; t < kQTiles; ++t)
    if (q_fills[t] > 0 &&
        !ptx::mbar_wait_drain(bar(L::kQFull + t), (q_fills[t] - 1u) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, kStatusDrainTimeout);
}

// Follower only: forwards each landed step and Q tile to the leader's barrier, in the
// producer's order.
template <Elem E>
__device__ __noinline__ void fwd2_relay(const FwdParams& p, uint32_t sbase, const ptx::WaitCtl& ctl) {
  using L = Fwd2Cfg<E>;
  auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
  uint32_t step = 0;
  uint32_t q_fills[kQTiles] = {0, 0};
  int bh, qb;
  for (int k = 0; unit_at2(p, k, bh, qb); ++k) {
    const int nt[kQTiles] = {tile_nkv2(p, qb, 0), tile_nkv2(p, qb, 1)};
    const int n = max(nt[0], nt[1]);
    for (int j = 0; j <= n; ++j, ++step) {
      const uint32_t rb = bar(L::kReady + step % L::kSteps);
      if (!ptx::mbar_wait(rb, (step / L::kSteps) & 1u, ctl, kStatusLoadTimeout)) return;
      ptx::mbar_arrive_cluster(ptx::mapa_shared(rb, 0));
      if (j == 0) {
#pragma unroll
        for (int t = 0; t < kQTiles; ++t) {
          if (nt[t] == 0) continue;
          if (!ptx::mbar_wait(bar(L::kQFull + t), q_fills[t] & 1u, ctl, kStatusLoadTimeout)) return;
          ptx::mbar_arrive_cluster(ptx::mapa_shared(bar(L::kQFull + t), 0));
          ++q_fills[t];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------- MMA issuer

template <Elem E, bool ACC, int KK = 0>
__device__ __forceinline__ void issue_pv2(uint32_t tO, uint32_t tS, uint32_t v_lo) {
  using L = Fwd2Cfg<E>;
  if constexpr (KK < kBlockN / 16) {
    constexpr uint32_t idesc = ptx::idesc_make(kPairRows, L::D, L::kAbType, false, true);
    constexpr uint32_t desc_hi = ptx::sdesc_hi(1024);
    constexpr int kAcc = (ACC || KK > 0) ? 1 : 0;
    // P: 8 TMEM columns per step (16 keys); V half: 16 key rows (2 KB) per step
    constexpr uint32_t kOb = (KK * 16 * 128) >> 4;
    ptx::mma2_f16_ts_o<kAcc, KK * 8, kOb>(tO, tS, v_lo, desc_hi, idesc);
    issue_pv2<E, ACC, KK + 1>(tO, tS, v_lo);
  }
}

template <Elem E, int KK = 0>
__device__ __forceinline__ void issue_s2(uint32_t tS, uint32_t q_lo, uint32_t k_lo) {
  using L = Fwd2Cfg<E>;
  if constexpr (KK < L::D / 16) {
    constexpr uint32_t idesc = ptx::idesc_make(kPairRows, kBlockN, L::kAbType, false, false);
    constexpr uint32_t desc_hi = ptx::sdesc_hi(1024);
    // 32 bytes of d per step: Q atoms are 128 rows (16 KB) apart, the K half's 64 rows (8 KB)
    constexpr uint32_t kOa = ((KK * 32 / 128) * L::kQAtomBytes + (KK * 32) % 128) >> 4;
    constexpr uint32_t kOk = ((KK * 32 / 128) * L::kKAtomBytes + (KK * 32) % 128) >> 4;
    ptx::mma2_f16_ss_o<KK ? 1 : 0, kOa, kOk>(tS, q_lo, k_lo, desc_hi, idesc);
    issue_s2<E, KK + 1>(tS, q_lo, k_lo);
  }
}

// Leader only: the same schedule as fwd_mma, with the pair's M = 256 MMAs and commits
// multicast to both CTAs (bit r = rank r).
template <Elem E>
__device__ __noinline__ void fwd2_mma(const FwdParams& p, uint32_t sbase, uint32_t tmem, const ptx::WaitCtl& ctl) {
  using L = Fwd2Cfg<E>;
  const uint32_t bar0 = sbase + L::kBarOff;
  auto bar = [bar0](int i) { return bar0 + 8u * i; };
  constexpr uint16_t kBoth = 3;
  constexpr uint32_t kSlotDesc = L::kSlotBytes >> 4;
  const uint32_t q_lo0 = ptx::sdesc_lo(sbase + L::kQOff, 16);
  const uint32_t q_lo1 = ptx::sdesc_lo(sbase + L::kQOff + L::kQTileBytes, 16);
  const uint32_t k_lo0 = ptx::sdesc_lo(sbase + L::kKVOff, 16);
  const uint32_t v_lo0 = ptx::sdesc_lo(sbase + L::kKVOff, L::kSlotBytes);
  const uint32_t tS0 = tmem + L::kTmemS, tS1 = tS0 + kBlockN;
  const uint32_t tO0 = tmem + L::kTmemO, tO1 = tO0 + L::D;
  const uint32_t ready0 = bar(L::kReady), done0 = bar(L::kDone);
  uint32_t load_idx = 0, step = 0;
  uint32_t q_uses[kQTiles] = {0, 0};
  uint32_t p_uses[kQTiles] = {0, 0};

  int bh, qb;
  bool have = unit_at2(p, 0, bh, qb);
  int j0 = 0;
  for (int k = 0; have; ++k) {
    const int nt[kQTiles] = {tile_nkv2(p, qb, 0), tile_nkv2(p, qb, 1)};
    const int n = max(nt[0], nt[1]);
    const int steady_end = min(nt[0], nt[1]) - 1;
    int bhn = 0, qbn = 0;
    const bool has_next = unit_at2(p, k + 1, bhn, qbn);
    const int ntn[kQTiles] = {has_next ? tile_nkv2(p, qbn, 0) : 0, has_next ? tile_nkv2(p, qbn, 1) : 0};
    bool next_ready = false;
    for (int j = j0; j <= n; ++j, ++step) {
      if (j == 2 && steady_end > 2) {
        uint32_t ks = (load_idx + 2u * j - 1u) % L::kStages;
        uint32_t pp0 = p_uses[0] & 1u, pp1 = p_uses[1] & 1u;
        for (; j < steady_end; ++j, ++step) {
          const uint32_t vs = ks + 1 == L::kStages ? 0u : ks + 1;
          const uint32_t v_lo = v_lo0 + vs * kSlotDesc, k_lo = k_lo0 + ks * kSlotDesc;
          const uint32_t si = step % L::kSteps, sph = (step / L::kSteps) & 1u;
          if (!ptx::mbar_wait(ready0 + 8u * si, sph, ctl, kStatusMmaTimeout)) goto done;
          if (!ptx::mbar_wait(bar(L::kPFull), pp0, ctl, kStatusMmaTimeout)) goto done;
          ptx::tc_fence_after();
          issue_pv2<E, true>(tO0, tS0, v_lo);
          issue_s2<E>(tS0, q_lo0, k_lo);
          ptx::mma2_commit_mc(bar(L::kSFull), kBoth);
          if (!ptx::mbar_wait(bar(L::kPFull + 1), pp1, ctl, kStatusMmaTimeout)) goto done;
          ptx::tc_fence_after();
          issue_pv2<E, true>(tO1, tS1, v_lo);
          issue_s2<E>(tS1, q_lo1, k_lo);
          ptx::mma2_commit_mc(bar(L::kSFull + 1), kBoth);
          ptx::mma2_commit_mc(done0 + 8u * si, kBoth);
          pp0 ^= 1u;
          pp1 ^= 1u;
          ks = vs + 1 == L::kStages ? 0u : vs + 1;
        }
        p_uses[0] += steady_end - 2;
        p_uses[1] += steady_end - 2;
      }
      if (!ptx::mbar_wait(ready0 + 8u * (step % L::kSteps), (step / L::kSteps) & 1u, ctl, kStatusMmaTimeout))
        goto done;
      const uint32_t vslot = j >= 1 ? (load_idx + v_pos(j - 1, n)) % L::kStages : 0u;
      const uint32_t kslot = j < n ? (load_idx + k_pos(j)) % L::kStages : 0u;
      const uint32_t next0 = step - j + n + 1;
      const uint32_t kslot_next = (load_idx + 2u * n) % L::kStages;
#pragma unroll
      for (int t = 0; t < kQTiles; ++t) {
        const uint32_t tS = t ? tS1 : tS0;
        if (j >= 1 && j - 1 < nt[t]) {
          if (!ptx::mbar_wait(bar(L::kPFull + t), p_uses[t] & 1u, ctl, kStatusMmaTimeout)) goto done;
          ++p_uses[t];
          ptx::tc_fence_after();
          const uint32_t v_lo = v_lo0 + vslot * kSlotDesc;
          if (j - 1 > 0) issue_pv2<E, true>(t ? tO1 : tO0, tS, v_lo);
          else issue_pv2<E, false>(t ? tO1 : tO0, tS, v_lo);
          if (j - 1 == nt[t] - 1) ptx::mma2_commit_mc(bar(L::kOFull + t), kBoth);
        }
        if (j < nt[t]) {
          if (j == 0) {
            if (!ptx::mbar_wait(bar(L::kQFull + t), q_uses[t] & 1u, ctl, kStatusMmaTimeout)) goto done;
            ++q_uses[t];
          }
          issue_s2<E>(tS, t == 0 ? q_lo0 : q_lo1, k_lo0 + kslot * kSlotDesc);
          ptx::mma2_commit_mc(bar(L::kSFull + t), kBoth);
          if (j == nt[t] - 1) ptx::mma2_commit_mc(bar(L::kQEmpty + t), kBoth);
        }
        if (has_next && ntn[t] > 0 && j == (nt[t] > 0 ? nt[t] : n)) {
          if (!next_ready) {
            if (!ptx::mbar_wait(ready0 + 8u * (next0 % L::kSteps), (next0 / L::kSteps) & 1u, ctl,
                                kStatusMmaTimeout))
              goto done;
            next_ready = true;
          }
          if (!ptx::mbar_wait(bar(L::kQFull + t), q_uses[t] & 1u, ctl, kStatusMmaTimeout)) goto done;
          ++q_uses[t];
          issue_s2<E>(tS, t == 0 ? q_lo0 : q_lo1, k_lo0 + kslot_next * kSlotDesc);
          ptx::mma2_commit_mc(bar(L::kSFull + t), kBoth);
          if (ntn[t] == 1) ptx::mma2_commit_mc(bar(L::kQEmpty + t), kBoth);
        }
      }
      ptx::mma2_commit_mc(done0 + 8u * (step % L::kSteps), kBoth);
      if (j == n && has_next) ptx::mma2_commit_mc(done0 + 8u * (next0 % L::kSteps), kBoth);
    }
    load_idx += 2u * n;
    if (has_next) ++step;
    j0 = has_next ? 1 : 0;
    have = has_next;
    bh = bhn;
    qb = qbn;
  }
done:
  // Every MMA issued so far must finish before TMEM is released.
  ptx::mma2_commit(bar(L::kMmaDone));
  if (!ptx::mbar_wait_drain(bar(L::kMmaDone), 0, ctl.timeout_ns)) atomicOr(ctl.status, kStatusDrainTimeout);
}

// ---------------------------------------------------------------------------- softmax

// Both CTAs: thread i of softmax warpgroup t owns row i of this CTA's 128 rows of the
// pair's tile t (TMEM lane i).  The leader's warps signal P locally, the follower's on
// the leader's barrier.
template <Elem E>
__device__ __forceinline__ void fwd2_softmax(const FwdParams& p, int t, uint32_t sbase, uint32_t tmem,
                                             uint32_t rank, const ptx::WaitCtl& ctl) {
  using L = Fwd2Cfg<E>;
  constexpr int D = L::D;
  auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
  const int r = threadIdx.x - t * kBlockM;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x / 32) & 3) * 32u;
  const uint32_t tS = tmem + (lane_base << 16) + L::kTmemS + t * kBlockN;
  const uint32_t tO = tmem + (lane_base << 16) + L::kTmemO + t * D;
  const uint32_t p_bar = rank == 0 ? bar(L::kPFull + t) : ptx::mapa_shared(bar(L::kPFull + t), 0);
  const float sl2 = p.scale_log2;
  uint32_t s_uses = 0, o_uses = 0;
  const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
  const int lane = threadIdx.x & 31;

  int bh, qb;
  for (int k = 0; unit_at2(p, k, bh, qb); ++k) {
    const int ntile = tile_nkv2(p, qb, t);
    if (ntile == 0) continue;
    const int r0 = qb * kUnitRows2 + t * kPairRows + static_cast<int>(rank) * kBlockM;
    const int row = r0 + r;
    float m = -INFINITY, l = 0.f;

    for (int j = 0; j < ntile; ++j) {
      const bool got = ptx::mbar_wait(bar(L::kSFull + t), s_uses & 1u, ctl, kStatusSoftmaxTimeout);
      if (!__all_sync(0xFFFFFFFFu, got)) return;
      ++s_uses;
      ptx::tc_fence_after();

      uint32_t sr[4][32];
#define S_(c) __uint_as_float(sr[(c) / 32][(c) % 32])
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + 32 * c, sr[c]);
      ptx::tmem_wait_ld();

      const int col0 = j * kBlockN;
      if (col0 + kBlockN > p.N || (p.causal && col0 + kBlockN - 1 > r0)) {
        // columns c >= visible are masked (past N, or past the diagonal); under the causal
        // mask the leader's rows can see none of the pair's last tile
        const int visible = (p.causal ? min(p.N, row + 1) : p.N) - col0;
#pragma unroll
        for (int c = 0; c < kBlockN; ++c)
          if (c >= visible) sr[c / 32][c % 32] = __float_as_uint(-INFINITY);
      }
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

      const float2 f2 = make_float2(sl2, sl2);
      const float2 nb = make_float2(-m_use, -m_use);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int c = 4 * q;
        const float2 x01 = ptx::fma2(make_float2(S_(c), S_(c + 1)), f2, nb);
        const float2 x23 = ptx::fma2(make_float2(S_(c + 2), S_(c + 3)), f2, nb);
        const float2 p01 = make_float2(ptx::ex2(x01.x), ptx::ex2(x01.y));
        const float2 p23 = make_float2(ptx::ex2(x23.x), ptx::ex2(x23.y));
        acc[q & 3] = ptx::add2(acc[q & 3], ptx::add2(p01, p23));
        sr[(c / 2) / 32][(c / 2) % 32] = ptx::pack2<L::kBf16Out>(p01.x, p01.y);
        sr[(c / 2 + 1) / 32][(c / 2 + 1) % 32] = ptx::pack2<L::kBf16Out>(p23.x, p23.y);
      }
      const float2 hs = ptx::add2(ptx::add2(acc[0], acc[1]), ptx::add2(acc[2], acc[3]));
      l = l * alpha + (hs.x + hs.y);

      if (rescale_o) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          ptx::tmem_ld32(tO + 32 * c, orr);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 v = ptx::mul2(make_float2(__uint_as_float(orr[i]), __uint_as_float(orr[i + 1])),
                                       make_float2(alpha, alpha));
            orr[i] = __float_as_uint(v.x);
            orr[i + 1] = __float_as_uint(v.y);
          }
          ptx::tmem_st32(tO + 32 * c, orr);
        }
      }
#undef S_
      ptx::tmem_st32(tS + 0, sr[0]);
      ptx::tmem_st32(tS + 32, sr[1]);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) ptx::mbar_arrive(p_bar);
        else ptx::mbar_arrive_cluster(p_bar);
      }
      m = m_use;
    }

    const bool got = ptx::mbar_wait(bar(L::kOFull + t), o_uses & 1u, ctl, kStatusSoftmaxTimeout);
    if (!__all_sync(0xFFFFFFFFu, got)) return;
    ++o_uses;
    ptx::tc_fence_after();
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    const bool live = row < p.N;
    uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                           (static_cast<size_t>(bh) * p.N + (live ? row : 0)) * D);
    uint32_t pk[D / 2];
    {
      uint32_t orr[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(tO + 32 * c, orr[c]);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < D / 2; ++i) {
        const float2 v = ptx::mul2(
            make_float2(__uint_as_float(orr[i / 16][(2 * i) % 32]), __uint_as_float(orr[i / 16][(2 * i + 1) % 32])),
            make_float2(inv_l, inv_l));
        pk[i] = ptx::pack2<L::kBf16Out>(v.x, v.y);
      }
    }
    if (live) {
      if (o_v8) {
#pragma unroll
        for (int i = 0; i < D / 16; ++i) ptx::st_global_v8(orow + 2 * i, pk + 8 * i);
      } else {
#pragma unroll
        for (int i = 0; i < D / 8; ++i) orow[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
    if (live && p.lse != nullptr)
      p.lse[static_cast<size_t>(bh) * p.N + row] = l > 0.f ? (m + ptx::lg2(l)) * kLn2 : -INFINITY;
    ptx::tc_fence_before();
  }
}

// ---------------------------------------------------------------------------- kernel

template <Elem E>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fa_fwd2_kernel(const __grid_constant__ FwdParams p) {
  using L = Fwd2Cfg<E>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  if (threadIdx.x == 0) {
    auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
    // the leader's ready and Q barriers also take the follower's relayed arrivals
    const uint32_t relayed = rank == 0 ? 2u : 1u;
    for (int t = 0; t < kQTiles; ++t) {
      ptx::mbar_init(bar(L::kQFull + t), relayed);
      ptx::mbar_init(bar(L::kQEmpty + t), 1);
      ptx::mbar_init(bar(L::kSFull + t), 1);
      ptx::mbar_init(bar(L::kPFull + t), 8);   // 4 softmax warps in each CTA (used in the leader)
      ptx::mbar_init(bar(L::kOFull + t), 1);
    }
    for (int s = 0; s < L::kSteps; ++s) {
      ptx::mbar_init(bar(L::kReady + s), relayed);
      ptx::mbar_init(bar(L::kDone + s), 1);
    }
    ptx::mbar_init(bar(L::kMmaDone), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    ptx::prefetch_tensormap(&p.tm_q);
    ptx::prefetch_tensormap(&p.tm_kh);
    ptx::prefetch_tensormap(&p.tm_v);
  }
  // both CTAs' barriers are initialised before either signals the other's
  ptx::cluster_sync();
  if (warp == kMmaWarp) {
    ptx::tmem_alloc2(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish2();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp >= 8) {
    ptx::setmaxnreg_dec<kControlRegs>();
    if (warp == kLoadWarp) {
      if (lane == 0) fwd2_producer<E>(p, sbase, rank, ctl);
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        if (rank == 0) fwd2_mma<E>(p, sbase, tmem, ctl);
        else fwd2_relay<E>(p, sbase, ctl);
      }
    }
  } else {
    ptx::setmaxnreg_inc<kSoftmaxRegs>();
    fwd2_softmax<E>(p, warp / 4, sbase, tmem, rank, ctl);
  }

  ptx::tc_fence_before();
  __syncthreads();
  // the leader's MMAs (which write both CTAs' TMEM) and the follower's remote arrivals
  // are over before either CTA frees TMEM or leaves
  ptx::cluster_sync();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc2(tmem, kTmemCols);
  }
  ptx::cluster_sync();
}

}  // namespace fa
