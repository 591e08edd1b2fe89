// Attention forward for sm_103a: f16/bf16 (head dim 64 or 128) and E4M3 (head dim 128).
//
// Computes O = softmax(scale * Q K^T [+ causal mask]) V and the per-row natural-log
// LSE, tile by tile with an online softmax, so the N x N score matrix never leaves
// the SM (the tiling and the streaming softmax with a running maximum and a
// correction factor at each tile boundary are the method of "FlashAttention 2 + 3 —
// speicherbewusste Attention-Kernels", sections "Kernpunkte" and "Begriffe auf
// dieser Seite"; the asynchronous copy of the next block during compute, the
// producer/consumer warp roles and the block-quantised FP8 mode are the levers of
// the FlashAttention-3 news piece, section "Drei technische Hebel", re-designed
// here for TMA + tcgen05/TMEM).
//
// One persistent CTA per SM walks work units (b*h, q-block of 256 rows = two
// 128-row Q tiles).  Warp roles (384 threads, three warpgroups):
//   warps 0-3   softmax warpgroup for Q tile 0 (thread i owns row i, TMEM lane i)
//   warps 4-7   softmax warpgroup for Q tile 1
//   warp  8     TMA producer: Q tiles, then K_j, V_j into a shared-memory ring
//   warp  9     MMA issuer: S_t = Q_t K_j^T and O_t += P_t V_j on tcgen05, TMEM alloc
//   warps 10-11 idle
// The softmax warpgroups hold a whole 128-score row in registers, so registers move
// to them (setmaxnreg): 2 x 128 threads x 216 + 128 x 72 = 384 x 168 at launch.  The
// producer and MMA roles are separate (non-inlined) functions so that nothing the
// softmax code keeps live has to fit the control warps' 72 registers.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1.  P_t overwrites the first columns of
// S_t (two 16-bit or four E4M3 values per column) and feeds the P.V MMA from TMEM.
//
// E4M3: Q, K are [N, d] codes and V arrives transposed ([d, N] codes), all with one
// scale per 64-row block.  The dequantisation factors fold into the exponent:
//   p~_ij = 2^(acc_ij * c * s_q(i) * s_k(j) - m_i + log2(s_v(j) / s_v,max))
// is P times V's block scale relative to the head's largest, rounded to E4M3 for
// the P.V MMA; the row sum divides the V factor back out, and the epilogue
// multiplies by s_v,max.
#pragma once

#include "fa_params.h"
#include "ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;          // query rows per Q tile
constexpr int kBlockN = 128;          // key rows per K/V tile
constexpr int kQTiles = 2;            // Q tiles per work unit
constexpr int kUnitRows = kBlockM * kQTiles;
constexpr int kThreads = 384;
constexpr uint32_t kSoftmaxRegs = 216;
constexpr uint32_t kControlRegs = 72;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
// The running max is only moved when it grows by more than 2^8 (log2 units): the
// un-normalised weights then stay below 256, and the output and the sum are
// rescaled far less often.  Exact in real arithmetic; the final division uses the
// same stale maximum for numerator and denominator.
constexpr float kRescaleThreshold = 8.0f;
constexpr int kHoldStoresMinTiles = 15;   // units longer than this hold SMSP-shared O stores
constexpr float kLn2 = 0.693147180559945309f;

// Bits of the device status word.
constexpr unsigned kStatusLoadTimeout = 1u;
constexpr unsigned kStatusMmaTimeout = 2u;
constexpr unsigned kStatusSoftmaxTimeout = 4u;
constexpr unsigned kStatusDrainTimeout = 8u;

enum class Elem : int { F16 = 0, BF16 = 1, E4M3 = 2 };

template <int D, Elem E>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static_assert(E != Elem::E4M3 || D == 128, "E4M3 path is built for head dim 128");
  static constexpr bool kFp8 = E == Elem::E4M3;
  static constexpr bool kBf16Out = E != Elem::F16;
  static constexpr int kElemBytes = kFp8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElemBytes;
  static constexpr int kAtoms = kRowBytes / 128;        // 128-byte swizzle atoms along d
  static constexpr int kAtomElems = 128 / kElemBytes;
  static constexpr int kAtomBytes = kBlockM * 128;      // one atom of a 128-row tile
  static constexpr int kTileBytes = kBlockM * kRowBytes; // Q, K, V tile (V^T tile for E4M3: d x 128 bytes)
  static constexpr int kMmaK = kFp8 ? 32 : 16;           // reduction depth of one MMA
  static constexpr uint32_t kAbType = (E == Elem::BF16) ? 1u : 0u;
  static constexpr int kPvSteps = kBlockN / kMmaK;
  static constexpr int kStages = kFp8 ? 12 : (D == 128 ? 5 : 8);
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQTiles * kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  // barrier indices.  K/V handoff is per MMA step, not per ring slot: the loads a
  // step consumes complete on one "ready" barrier and one commit per step frees
  // its slots ("done").  A ring of kSteps > kStages step barriers never aliases a
  // phase: every step carries at least one load, so a slot's previous occupant
  // belongs to a step at most kStages back.
  static constexpr int kSteps = 16;
  static_assert(kSteps > kStages, "step ring must outlast the load ring");
  static constexpr int kQFull = 0, kQEmpty = 2, kReady = 4, kDone = 4 + kSteps;
  static constexpr int kSFull = 4 + 2 * kSteps, kPFull = kSFull + 2, kOFull = kPFull + 2;
  static constexpr int kMmaDone = kOFull + 2;
  static constexpr int kNumBars = kMmaDone + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM base slot, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;             // room to align the base to 1 KB
  static constexpr uint32_t kTmemS = 0;                    // + t * 128
  static constexpr uint32_t kTmemO = 256;                  // + t * D
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// The k-th causal unit (b*h, block) of CTA c of a persistent grid of G CTAs, for n blocks
// per head whose cost grows with the block index (cost_grows: the forward's q-blocks and the
// dQ kernel's Q tiles) or shrinks with it (the dK/dV kernel's K/V tiles); false once the CTA
// has none left.  Blocks b and n-1-b of one head form a pair of equal total cost.
//  - Whole rounds of G pairs: a CTA takes whole pairs round-robin in head-major order (the
//    longer half first), which balances those rounds and keeps concurrent CTAs on few
//    heads, so their K/V or Q re-reads hit L2.
//  - The rest (the partial last round, and with n >= 16 blocks a head the last whole round
//    as well; the middle block of each head when n is odd): their units sorted by cost,
//    longest first, and dealt in snake order (G CTAs left to right, then right to left), so
//    the grid's last wave ends nearly level instead of leaving part of it idle.  The long
//    halves of the remaining pairs come first (by pair position within the head, then
//    head), then the middle blocks, then the short halves in reverse.  Units dealt this way
//    lose the head order; below 16 blocks a head a unit is too short for that to pay with a
//    whole round.
static __device__ __noinline__ bool causal_unit(int G, int c, int BH, int n, int k, bool cost_grows, int& bh,
                                            int& blk) {
  const int P = n / 2;                                // pairs per head
  const int pairs = BH * P;
  const int R = max(0, pairs / G - (n >= 16 ? 1 : 0));   // rounds dealt as whole pairs
  if (k < 2 * R) {
    const int s = c + (k >> 1) * G;
    bh = s / P;
    const int i = s % P;
    const int lo = i, hi = n - 1 - i;
    const int longer = cost_grows ? hi : lo, shorter = cost_grows ? lo : hi;
    blk = (k & 1) ? shorter : longer;
    return true;
  }
  const int t = k - 2 * R;
  const int idx = t * G + ((t & 1) ? G - 1 - c : c);
  const int S0 = R * G;                               // first remaining pair
  const int Ltot = pairs - S0;                        // remaining pairs
  const int M = (n & 1) ? BH : 0;                     // middle blocks
  // the x-th remaining pair ordered by position i within its head, then by head
  auto entry = [&](int x, int& h, int& i) {
    const int h0 = S0 / P, i0 = S0 % P;
    const int A = BH - 1 - h0;                        // whole heads after the first remaining one
    int r;
    if (x < i0 * A) {
      i = x / A;
      r = x % A;
    } else {
      i = (x + i0) / (A + 1);
      r = (x + i0) % (A + 1);
    }
    h = (i >= i0 ? h0 : h0 + 1) + r;
  };
  if (idx < Ltot) {
    int h, i;
    entry(idx, h, i);
    bh = h;
    blk = cost_grows ? n - 1 - i : i;                 // the longer half
    return true;
  }
  if (idx < Ltot + M) {
    bh = idx - Ltot;
    blk = P;
    return true;
  }
  if (idx < 2 * Ltot + M) {
    int h, i;
    entry(Ltot - 1 - (idx - Ltot - M), h, i);
    bh = h;
    blk = cost_grows ? i : n - 1 - i;                 // the shorter half
    return true;
  }
  return false;
}

// The k-th (b*h, q-block) unit of this CTA of the persistent grid; false once the CTA
// has none left.  Every role of the CTA walks the same sequence.  Non-causal: units in
// head-major order, dealt round-robin, so the CTAs running at the same time share a few
// heads and their K/V re-reads hit L2.  Causal: causal_unit (the cost of q-block qb grows
// with qb).
__device__ __forceinline__ bool unit_at(const FwdParams& p, int k, int& bh, int& qb) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  if (!p.causal) {
    const int u = c + k * G;
    if (u >= p.num_units) return false;
    bh = u / p.n_qblk;
    qb = u % p.n_qblk;
    return true;
  }
  return causal_unit(G, c, p.BH, p.n_qblk, k, true, bh, qb);
}

// Number of K/V tiles Q tile t of q-block qb attends to (0 if the tile is past N).
__device__ __forceinline__ int tile_nkv(const FwdParams& p, int qb, int t) {
  const int r0 = qb * kUnitRows + t * kBlockM;
  if (r0 >= p.N) return 0;
  const int nkv = (p.N + kBlockN - 1) / kBlockN;
  return p.causal ? min(nkv, r0 / kBlockN + 1) : nkv;
}

// Order of the K/V loads of a unit with n key tiles: K_0, K_1, V_0, K_2, V_1, ...,
// K_{n-1}, V_{n-2}, V_{n-1}.  K runs one tile ahead of V, matching the MMA order
// (S_t(j) needs K_j one step before O_t += P_t V_j), so the ring holds about two
// steps of lead for both operands.
__device__ __forceinline__ uint32_t k_pos(int j) { return j == 0 ? 0u : 2u * j - 1u; }
__device__ __forceinline__ uint32_t v_pos(int j, int n) { return j + 1 < n ? 2u * j + 2u : 2u * n - 1u; }

// ---------------------------------------------------------------------------- producer

// MMA step j of a unit consumes K_j (j < n) and V_{j-1} (j >= 1); the producer issues
// them in that order into consecutive ring slots, completing on the step's ready
// barrier, once the steps that consumed those slots' previous tiles are done.
template <int D, Elem E>
__device__ __noinline__ void fwd_producer(const FwdParams& p, uint32_t sbase,
                                             const ptx::WaitCtl& ctl) {
  using L = FwdCfg<D, E>;
  auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
  uint32_t load_idx = 0;                 // ring position of the next K/V tile
  uint32_t step = 0;                     // MMA steps prepared so far
  uint32_t q_fills[kQTiles] = {0, 0};
  uint32_t slot_step[L::kStages];        // 1 + the step consuming each slot's tile (0: empty)
#pragma unroll
  for (int s = 0; s < L::kStages; ++s) slot_step[s] = 0;
  uint32_t armed = 0;                    // bit g % kSteps: step g's loads were issued
  // the whole warp runs this loop converged (its waits included); one lane issues
  const bool lead = ptx::elect_one() != 0;

  int bh, qb;
  for (int k = 0; unit_at(p, k, bh, qb); ++k) {
    const int n0 = tile_nkv(p, qb, 0), n1 = tile_nkv(p, qb, 1);
    const int n = max(n0, n1);
    {
      // Q is read once, so its next load comes from HBM; start that unit's Q on its
      // way into L2 now, a whole unit ahead of the load
      int bhn, qbn;
      if (unit_at(p, k + 1, bhn, qbn)) {
#pragma unroll
        for (int t = 0; t < kQTiles; ++t)
          if (lead && tile_nkv(p, qbn, t) > 0)
#pragma unroll
            for (int a = 0; a < L::kAtoms; ++a)
              ptx::tma_prefetch_3d(&p.tm_q, a * L::kAtomElems, qbn * kUnitRows + t * kBlockM, bhn);
      }
    }
    for (int j = 0; j <= n; ++j, ++step) {
      const uint32_t cnt = (j < n ? 1u : 0u) + (j >= 1 ? 1u : 0u);
      const uint32_t bit = 1u << (step % L::kSteps);
      const uint32_t rb = bar(L::kReady + step % L::kSteps);
      armed &= ~bit;
      // test hook: the step holding load number dbg_skip_load gets none of its loads
      const bool skip = p.dbg_skip_load >= 0 && static_cast<uint32_t>(p.dbg_skip_load) >= load_idx &&
                        static_cast<uint32_t>(p.dbg_skip_load) < load_idx + cnt;
      // each tile goes out as soon as its own slot is free; the step's last tile
      // arrives on the ready barrier, earlier ones only add their bytes
      for (uint32_t i = 0; i < cnt; ++i) {
        const uint32_t slot = (load_idx + i) % L::kStages;
        const uint32_t prev = slot_step[slot];
        if (prev != 0 && !ptx::mbar_wait(bar(L::kDone + (prev - 1) % L::kSteps),
                                         ((prev - 1) / L::kSteps) & 1u, ctl, kStatusLoadTimeout)) {
          if (i > 0 && !skip) {
            // a copy of this step is in flight: arrive so its phase completes when it lands
            if (lead) ptx::mbar_arrive(rb);
            armed |= bit;
          }
          goto drain;
        }
        if (!skip && lead) {
          if (i + 1 < cnt) ptx::mbar_expect_tx(rb, L::kTileBytes);
          else ptx::mbar_arrive_expect_tx(rb, L::kTileBytes);
          const bool is_k = i == 0 && j < n;
          const int jj = is_k ? j : j - 1;
          const uint32_t dst = sbase + L::kKVOff + slot * L::kTileBytes;
          if (L::kFp8 && !is_k) {
            // V^T tile: 128 rows of d, 128 keys (bytes) each
            ptx::tma_load_3d(dst, &p.tm_v, rb, jj * kBlockN, 0, bh);
          } else {
#pragma unroll
            for (int a = 0; a < L::kAtoms; ++a)
              ptx::tma_load_3d(dst + a * L::kAtomBytes, is_k ? &p.tm_k : &p.tm_v, rb, a * L::kAtomElems,
                               jj * kBlockN, bh);
          }
        }
        slot_step[slot] = step + 1;
      }
      if (!skip) armed |= bit;
      load_idx += cnt;
      if (j == 0) {
        // The unit's Q tiles go out after its K_0: the MMA thread issues this unit's
        // S_t(0) at the end of the previous unit, tile 0's possibly a step before
        // tile 1's last S frees Q buffer 1, so K_0 must not queue behind that wait.
#pragma unroll
        for (int t = 0; t < kQTiles; ++t) {
          if ((t == 0 ? n0 : n1) == 0) continue;
          if (!ptx::mbar_wait(bar(L::kQEmpty + t), (q_fills[t] & 1u) ^ 1u, ctl, kStatusLoadTimeout))
            goto drain;
          if (lead) {
            ptx::mbar_arrive_expect_tx(bar(L::kQFull + t), L::kTileBytes);
#pragma unroll
            for (int a = 0; a < L::kAtoms; ++a)
              ptx::tma_load_3d(sbase + L::kQOff + t * L::kTileBytes + a * L::kAtomBytes, &p.tm_q,
                               bar(L::kQFull + t), a * L::kAtomElems, qb * kUnitRows + t * kBlockM, bh);
          }
          ++q_fills[t];
        }
      }
    }
  }
drain:
  // Copies still in flight must land before the CTA may exit: wait for the ready
  // phase of every step issued among the last kSteps (immediate on the normal path).
  for (uint32_t g = step > static_cast<uint32_t>(L::kSteps) ? step - L::kSteps : 0; g < step; ++g)
    if (((armed >> (g % L::kSteps)) & 1u) &&
        !ptx::mbar_wait_drain(bar(L::kReady + g % L::kSteps), (g / L::kSteps) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, kStatusDrainTimeout);
  for (int t = 0; t < kQTiles; ++t)
    if (q_fills[t] > 0 &&
        !ptx::mbar_wait_drain(bar(L::kQFull + t), (q_fills[t] - 1u) & 1u, ctl.timeout_ns))
      atomicOr(ctl.status, kStatusDrainTimeout);
}

// ---------------------------------------------------------------------------- MMA issuer

// PV and S MMAs of Q tile t for key step j (called by the single MMA thread).
// Descriptor low words of ring slot s are the slot-0 word plus s * (tile bytes >> 4):
// shared addresses stay below 2^18, so the sum never carries into the LBO field.
template <int D, Elem E>
__host__ __device__ constexpr uint32_t v_lbo() {
  // 16-bit V is [N, d] (MN-major B, 64-wide d atoms one atom apart); E4M3 V^T is K-major
  return FwdCfg<D, E>::kFp8 ? 16u : static_cast<uint32_t>(FwdCfg<D, E>::kAtomBytes);
}

// The MMAs of one PV or S block, unrolled at compile time so that every operand
// offset is an immediate (see the _o wrappers).
template <int D, Elem E, bool ACC, int KK = 0>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tS, uint32_t v_lo, uint32_t lead = 1) {
  using L = FwdCfg<D, E>;
  if constexpr (KK < L::kPvSteps) {
    constexpr uint32_t idesc_pv = ptx::idesc_make(kBlockM, D, L::kAbType, false, !L::kFp8);
    constexpr uint32_t desc_hi = ptx::sdesc_hi(1024);
    constexpr int kAcc = (ACC || KK > 0) ? 1 : 0;
    // P: 8 TMEM columns per step (16 packed 16-bit or 32 packed E4M3 keys).  B: 16-bit
    // V is [N, d], 16 key rows (2 KB) per step; E4M3 V^T rows hold 32 keys per step.
    constexpr uint32_t kOb = L::kFp8 ? (KK * 32) >> 4 : (KK * 16 * 128) >> 4;
    if constexpr (L::kFp8) ptx::mma_f8_ts_oe<kAcc, KK * 8, kOb>(lead, tO, tS, v_lo, desc_hi, idesc_pv);
    else ptx::mma_f16_ts_oe<kAcc, KK * 8, kOb>(lead, tO, tS, v_lo, desc_hi, idesc_pv);
    issue_pv<D, E, ACC, KK + 1>(tO, tS, v_lo, lead);
  }
}

template <int D, Elem E, int KK = 0>
__device__ __forceinline__ void issue_s(uint32_t tS, uint32_t q_lo, uint32_t k_lo, uint32_t lead = 1) {
  using L = FwdCfg<D, E>;
  if constexpr (KK < D / L::kMmaK) {
    constexpr uint32_t idesc_qk = ptx::idesc_make(kBlockM, kBlockN, L::kAbType, false, false);
    constexpr uint32_t desc_hi = ptx::sdesc_hi(1024);
    // K-major operands: 32 bytes of d per step inside a 128-byte swizzle atom
    constexpr uint32_t kOff = ((KK * 32 / 128) * L::kAtomBytes + (KK * 32) % 128) >> 4;
    if constexpr (L::kFp8) ptx::mma_f8_ss_oe<KK ? 1 : 0, kOff, kOff>(lead, tS, q_lo, k_lo, desc_hi, idesc_qk);
    else ptx::mma_f16_ss_oe<KK ? 1 : 0, kOff, kOff>(lead, tS, q_lo, k_lo, desc_hi, idesc_qk);
    issue_s<D, E, KK + 1>(tS, q_lo, k_lo, lead);
  }
}

// One lane of the MMA warp issues every MMA (the warp runs the loop converged, see
// ptx::mma_f16_ss_oe), in the order
//   O_0 += P_0 V_{j-1};  S_0 = Q_0 K_j^T;  O_1 += P_1 V_{j-1};  S_1 = Q_1 K_j^T
// so the tensor pipe runs one tile's pair while the other tile's softmax works.
// tcgen05.mma issue blocks on a very short queue: an MMA takes about as long to
// issue as the tensor pipe takes to run the one before it, so every instruction
// between MMA groups leaves the pipe idle.  The steps where both tiles do the same
// thing (all but the first two and the last ones of a unit) therefore run in a
// separate loop without per-tile conditions, with ring slots and barrier parities
// advanced incrementally and descriptors formed by one add.  MMAs run in issue
// order, which is what lets S_t(j+1) overwrite the TMEM holding P_t(j) after
// O_t += P_t(j) V_j.
template <int D, Elem E>
__device__ __noinline__ void fwd_mma(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                     const ptx::WaitCtl& ctl) {
  using L = FwdCfg<D, E>;
  const uint32_t bar0 = sbase + L::kBarOff;
  auto bar = [bar0](int i) { return bar0 + 8u * i; };
  constexpr uint32_t kSlotDesc = L::kTileBytes >> 4;
  const uint32_t q_lo0 = ptx::sdesc_lo(sbase + L::kQOff, 16);
  const uint32_t q_lo1 = ptx::sdesc_lo(sbase + L::kQOff + L::kTileBytes, 16);
  const uint32_t k_lo0 = ptx::sdesc_lo(sbase + L::kKVOff, 16);
  const uint32_t v_lo0 = ptx::sdesc_lo(sbase + L::kKVOff, v_lbo<D, E>());
  const uint32_t tS0 = tmem + L::kTmemS, tS1 = tS0 + kBlockN;
  const uint32_t tO0 = tmem + L::kTmemO, tO1 = tO0 + D;
  const uint32_t ready0 = bar(L::kReady), done0 = bar(L::kDone);
  uint32_t load_idx = 0;
  uint32_t step = 0;                     // MMA steps issued so far (the producer counts alike)
  uint32_t q_uses[kQTiles] = {0, 0};
  uint32_t p_uses[kQTiles] = {0, 0};
  const uint32_t lead = ptx::elect_one();   // the whole warp runs this loop, one lane issues

  int bh, qb;
  bool have = unit_at(p, 0, bh, qb);
  int j0 = 0;                            // 1 once a unit's step 0 ran inside the previous unit
  for (int k = 0; have; ++k) {
    const int nt[kQTiles] = {tile_nkv(p, qb, 0), tile_nkv(p, qb, 1)};
    const int n = max(nt[0], nt[1]);
    // steps 2 .. steady_end - 1: both tiles run PV(j-1) and S(j), none of them is a
    // tile's last PV or last S, and V_{j-1} sits right after K_j in the ring
    const int steady_end = min(nt[0], nt[1]) - 1;
    // The next unit's step 0 (S_t = Q_t K_0^T) is issued inside this unit, right after
    // tile t's last PV (in the last step for a tile with no PV), so each softmax group
    // finds its next S as soon as its epilogue ends.
    int bhn = 0, qbn = 0;
    const bool has_next = unit_at(p, k + 1, bhn, qbn);
    const int ntn[kQTiles] = {has_next ? tile_nkv(p, qbn, 0) : 0, has_next ? tile_nkv(p, qbn, 1) : 0};
    bool next_ready = false;
    for (int j = j0; j <= n; ++j, ++step) {
      if (j == 2 && steady_end > 2) {
        uint32_t ks = (load_idx + 2u * j - 1u) % L::kStages;     // ring slot of K_j
        uint32_t pp0 = p_uses[0] & 1u, pp1 = p_uses[1] & 1u;
        for (; j < steady_end; ++j, ++step) {
          const uint32_t vs = ks + 1 == L::kStages ? 0u : ks + 1;  // V_{j-1} follows K_j
          const uint32_t v_lo = v_lo0 + vs * kSlotDesc, k_lo = k_lo0 + ks * kSlotDesc;
          const uint32_t si = step % L::kSteps, sph = (step / L::kSteps) & 1u;
          if (!ptx::mbar_wait(ready0 + 8u * si, sph, ctl, kStatusMmaTimeout)) goto done;
          if (!ptx::mbar_wait(bar(L::kPFull), pp0, ctl, kStatusMmaTimeout)) goto done;
          ptx::tc_fence_after();
          issue_pv<D, E, true>(tO0, tS0, v_lo, lead);
          issue_s<D, E>(tS0, q_lo0, k_lo, lead);
          ptx::mma_commit_e(lead, bar(L::kSFull));
          if (!ptx::mbar_wait(bar(L::kPFull + 1), pp1, ctl, kStatusMmaTimeout)) goto done;
          ptx::tc_fence_after();
          issue_pv<D, E, true>(tO1, tS1, v_lo, lead);
          issue_s<D, E>(tS1, q_lo1, k_lo, lead);
          ptx::mma_commit_e(lead, bar(L::kSFull + 1));
          ptx::mma_commit_e(lead, done0 + 8u * si);
          pp0 ^= 1u;
          pp1 ^= 1u;
          ks = vs + 1 == L::kStages ? 0u : vs + 1;
        }
        p_uses[0] += steady_end - 2;
        p_uses[1] += steady_end - 2;
      }
      // every load of this step has landed
      if (!ptx::mbar_wait(ready0 + 8u * (step % L::kSteps), (step / L::kSteps) & 1u, ctl, kStatusMmaTimeout))
        goto done;
      const uint32_t vslot = j >= 1 ? (load_idx + v_pos(j - 1, n)) % L::kStages : 0u;
      const uint32_t kslot = j < n ? (load_idx + k_pos(j)) % L::kStages : 0u;
      const uint32_t next0 = step - j + n + 1;                        // the next unit's step 0
      const uint32_t kslot_next = (load_idx + 2u * n) % L::kStages;   // and its K_0
#pragma unroll
      for (int t = 0; t < kQTiles; ++t) {
        const uint32_t tS = t ? tS1 : tS0;
        if (j >= 1 && j - 1 < nt[t]) {
          // O_t += P_t V_{j-1}
          if (!ptx::mbar_wait(bar(L::kPFull + t), p_uses[t] & 1u, ctl, kStatusMmaTimeout)) goto done;
          ++p_uses[t];
          ptx::tc_fence_after();
          const uint32_t v_lo = v_lo0 + vslot * kSlotDesc;
          if (j - 1 > 0) issue_pv<D, E, true>(t ? tO1 : tO0, tS, v_lo, lead);
          else issue_pv<D, E, false>(t ? tO1 : tO0, tS, v_lo, lead);
          if (j - 1 == nt[t] - 1) ptx::mma_commit_e(lead, bar(L::kOFull + t));
        }
        if (j < nt[t]) {
          // S_t = Q_t K_j^T
          if (j == 0) {
            if (!ptx::mbar_wait(bar(L::kQFull + t), q_uses[t] & 1u, ctl, kStatusMmaTimeout)) goto done;
            ++q_uses[t];
          }
          issue_s<D, E>(tS, t == 0 ? q_lo0 : q_lo1, k_lo0 + kslot * kSlotDesc, lead);
          ptx::mma_commit_e(lead, bar(L::kSFull + t));
          if (j == nt[t] - 1) ptx::mma_commit_e(lead, bar(L::kQEmpty + t));
        }
        if (has_next && ntn[t] > 0 && j == (nt[t] > 0 ? nt[t] : n)) {
          // the next unit's S_t = Q_t K_0^T, right after this tile's last P.V (its O is
          // then ready for the epilogue before anything waits on the next unit's loads)
          if (!next_ready) {
            if (!ptx::mbar_wait(ready0 + 8u * (next0 % L::kSteps), (next0 / L::kSteps) & 1u, ctl,
                                kStatusMmaTimeout))
              goto done;
            next_ready = true;
          }
          if (!ptx::mbar_wait(bar(L::kQFull + t), q_uses[t] & 1u, ctl, kStatusMmaTimeout)) goto done;
          ++q_uses[t];
          issue_s<D, E>(tS, t == 0 ? q_lo0 : q_lo1, k_lo0 + kslot_next * kSlotDesc, lead);
          ptx::mma_commit_e(lead, bar(L::kSFull + t));
          if (ntn[t] == 1) ptx::mma_commit_e(lead, bar(L::kQEmpty + t));
        }
      }
      ptx::mma_commit_e(lead, done0 + 8u * (step % L::kSteps));
      if (j == n && has_next) ptx::mma_commit_e(lead, done0 + 8u * (next0 % L::kSteps));
    }
    load_idx += 2u * n;
    // the next unit's step 0 has been issued: it starts at step 1
    if (has_next) ++step;
    j0 = has_next ? 1 : 0;
    have = has_next;
    bh = bhn;
    qb = qbn;
  }
done:
  // Every MMA issued so far must finish before TMEM is released.
  ptx::mma_commit_e(lead, bar(L::kMmaDone));
  if (!ptx::mbar_wait_drain(bar(L::kMmaDone), 0, ctl.timeout_ns)) atomicOr(ctl.status, kStatusDrainTimeout);
}

// ---------------------------------------------------------------------------- softmax

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
  return x;
}

template <int D, Elem E>
__device__ __forceinline__ void fwd_softmax(const FwdParams& p, int t, uint32_t sbase, uint32_t tmem,
                                            const ptx::WaitCtl& ctl) {
  using L = FwdCfg<D, E>;
  auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
  const int r = threadIdx.x - t * kBlockM;                          // row within the tile
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x / 32) & 3) * 32u;
  const uint32_t tS = tmem + (lane_base << 16) + L::kTmemS + t * kBlockN;
  const uint32_t tO = tmem + (lane_base << 16) + L::kTmemO + t * D;
  const float sl2 = p.scale_log2;
  uint32_t s_uses = 0, o_uses = 0;
  const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
  const int lane = threadIdx.x & 31;

  int bh, qb;
  for (int k = 0; unit_at(p, k, bh, qb); ++k) {
    const int ntile = tile_nkv(p, qb, t);
    if (ntile == 0) continue;
    const int r0 = qb * kUnitRows + t * kBlockM;
    const int row = r0 + r;
    float m = -INFINITY, l = 0.f;

    // E4M3 dequantisation: row factor, and the head's largest V block scale
    float c_row = sl2, sv_max = 1.f;
    const float* ks = nullptr;
    const float* vs = nullptr;
    if constexpr (L::kFp8) {
      const size_t sb = static_cast<size_t>(bh) * p.n_sblk;
      ks = p.k_scale + sb;
      vs = p.v_scale + sb;
      c_row = sl2 * __ldg(p.q_scale + sb + min(row / 64, p.n_sblk - 1));
      float mx = 0.f;
      for (int i = lane; i < p.n_sblk; i += 32) mx = fmaxf(mx, __ldg(vs + i));
      sv_max = warp_max(mx);
    }
    // E4M3: the K and V scales of the tile about to be processed, loaded one tile
    // ahead so that their latency stays off the softmax's critical path
    const float inv_sv_max = 1.f / sv_max;
    float nk0 = 1.f, nk1 = 1.f, nv0 = 1.f, nv1 = 1.f;
    if constexpr (L::kFp8) {
      nk0 = __ldg(ks);
      nk1 = __ldg(ks + min(1, p.n_sblk - 1));
      nv0 = __ldg(vs);
      nv1 = __ldg(vs + min(1, p.n_sblk - 1));
    }

    for (int j = 0; j < ntile; ++j) {
      const bool got = ptx::mbar_wait(bar(L::kSFull + t), s_uses & 1u, ctl, kStatusSoftmaxTimeout);
      if (!__all_sync(0xFFFFFFFFu, got)) return;
      ++s_uses;
      ptx::tc_fence_after();

      uint32_t sr[4][32];
#define S_(c) __uint_as_float(sr[(c) / 32][(c) % 32])
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + 32 * c, sr[c]);

      // per-half factors (E4M3: one K and one V scale per 64 keys)
      float f0 = sl2, f1 = sl2, b0 = 0.f, b1 = 0.f;
      if constexpr (L::kFp8) {
        f0 = c_row * nk0;
        f1 = c_row * nk1;
        b0 = ptx::lg2(nv0 * inv_sv_max);              // log2 of V's relative block scale (<= 0)
        b1 = ptx::lg2(nv1 * inv_sv_max);
        const int kb0 = min(2 * j + 2, p.n_sblk - 1), kb1 = min(2 * j + 3, p.n_sblk - 1);
        nk0 = __ldg(ks + kb0);
        nk1 = __ldg(ks + kb1);
        nv0 = __ldg(vs + kb0);
        nv1 = __ldg(vs + kb1);
      }
      ptx::tmem_wait_ld();

      const int col0 = j * kBlockN;
      if (col0 + kBlockN > p.N || (p.causal && col0 + kBlockN - 1 > r0)) {
        // columns c >= visible of this tile are masked (past N, or past the diagonal)
        const int visible = (p.causal ? min(p.N, row + 1) : p.N) - col0;
#pragma unroll
        for (int c = 0; c < kBlockN; ++c)
          if (c >= visible) sr[c / 32][c % 32] = __float_as_uint(-INFINITY);
      }
      // row maxima of the two 64-column halves: 3-input max trees, 4 chains per half
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
      const float m_new = fmaxf(m, fmaxf(mh[0] * f0, mh[1] * f1));

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

      // P = 2^(s * f - m) (times V's relative block scale for E4M3), packed for the MMA;
      // s * f - m in packed pairs, row sums in 4 packed accumulators per half
      float2 hs[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float2 fh = make_float2(h ? f1 : f0, h ? f1 : f0);
        const float nbh = (h ? b1 : b0) - m_use;
        const float2 nb = make_float2(nbh, nbh);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < 16; ++q) {           // four columns per step
          const int c = 64 * h + 4 * q;
          const float2 x01 = ptx::fma2(make_float2(S_(c), S_(c + 1)), fh, nb);
          const float2 x23 = ptx::fma2(make_float2(S_(c + 2), S_(c + 3)), fh, nb);
          const float2 p01 = make_float2(ptx::ex2(x01.x), ptx::ex2(x01.y));
          const float2 p23 = make_float2(ptx::ex2(x23.x), ptx::ex2(x23.y));
          acc[q & 3] = ptx::add2(acc[q & 3], ptx::add2(p01, p23));
          // packed P overwrites scores already consumed (slot index <= c)
          if constexpr (L::kFp8) {
            sr[(c / 4) / 32][(c / 4) % 32] = ptx::pack4_e4m3(p01.x, p01.y, p23.x, p23.y);
          } else {
            sr[(c / 2) / 32][(c / 2) % 32] = ptx::pack2<L::kBf16Out>(p01.x, p01.y);
            sr[(c / 2 + 1) / 32][(c / 2 + 1) % 32] = ptx::pack2<L::kBf16Out>(p23.x, p23.y);
          }
        }
        const float2 t = ptx::add2(ptx::add2(acc[0], acc[1]), ptx::add2(acc[2], acc[3]));
        hs[h] = t;
      }
      const float sum0 = hs[0].x + hs[0].y, sum1 = hs[1].x + hs[1].y;
      if constexpr (L::kFp8) {
        // row sum of P itself: divide V's relative scale back out of each half
        l = l * alpha + (sum0 * ptx::ex2(-b0) + sum1 * ptx::ex2(-b1));
      } else {
        l = l * alpha + (sum0 + sum1);
      }

      if (rescale_o) {
        // The previous O_t += P V has completed: the S_t commit that woke us tracks it.
        // Two 32-column chunks per TMEM round trip.
#pragma unroll 1
        for (int c = 0; c < D / 32; c += 2) {
          uint32_t orr[2][32];
          ptx::tmem_ld32(tO + 32 * c, orr[0]);
          ptx::tmem_ld32(tO + 32 * c + 32, orr[1]);
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
          ptx::tmem_st32(tO + 32 * c, orr[0]);
          ptx::tmem_st32(tO + 32 * c + 32, orr[1]);
        }
      }
#undef S_
      ptx::tmem_st32(tS + 0, sr[0]);
      if constexpr (!L::kFp8) ptx::tmem_st32(tS + 32, sr[1]);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(L::kPFull + t));
      m = m_use;
    }

    // epilogue: O = O_acc / l (x s_v,max for E4M3), LSE = ln 2 * (m + log2 l)
    const bool got = ptx::mbar_wait(bar(L::kOFull + t), o_uses & 1u, ctl, kStatusSoftmaxTimeout);
    if (!__all_sync(0xFFFFFFFFu, got)) return;
    ++o_uses;
    ptx::tc_fence_after();
    const float inv_l = l > 0.f ? sv_max / l : 0.f;
    const bool live = row < p.N;
    uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                           (static_cast<size_t>(bh) * p.N + (live ? row : 0)) * D);
    // all of the row's O columns in one TMEM round trip, scaled and packed
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
    // In long units, the warps that share an SMSP with the MMA-issuing warp hold their O
    // stores until the next unit's S_t(0) is in (the wait step 0 of that unit does anyway):
    // their row-scattered stores queue ahead of that warp's tcgen05 instructions, and by
    // then the MMA thread has issued this unit boundary's MMAs.  In short units the held
    // stores would delay the next unit more than they save.
    if (ntile > kHoldStoresMinTiles && ((threadIdx.x / 32) & 3) == (kMmaWarp & 3)) {
      int bhn, qbn;
      if (unit_at(p, k + 1, bhn, qbn) && tile_nkv(p, qbn, t) > 0) {
        const bool held = ptx::mbar_wait(bar(L::kSFull + t), s_uses & 1u, ctl, kStatusSoftmaxTimeout);
        if (!__all_sync(0xFFFFFFFFu, held)) return;
      }
    }
    if (live) {
      if (o_v8) {
        // 32-byte stores fill whole sectors (rows are 128 or 256 bytes; base 32-aligned)
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

template <int D, Elem E>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = FwdCfg<D, E>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  if (threadIdx.x == 0) {
    auto bar = [&](int i) { return sbase + L::kBarOff + 8u * i; };
    for (int t = 0; t < kQTiles; ++t) {
      ptx::mbar_init(bar(L::kQFull + t), 1);
      ptx::mbar_init(bar(L::kQEmpty + t), 1);
      ptx::mbar_init(bar(L::kSFull + t), 1);
      ptx::mbar_init(bar(L::kPFull + t), 4);   // one arrival per softmax warp
      ptx::mbar_init(bar(L::kOFull + t), 1);
    }
    for (int s = 0; s < L::kSteps; ++s) {
      ptx::mbar_init(bar(L::kReady + s), 1);
      ptx::mbar_init(bar(L::kDone + s), 1);
    }
    ptx::mbar_init(bar(L::kMmaDone), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    ptx::prefetch_tensormap(&p.tm_q);
    ptx::prefetch_tensormap(&p.tm_k);
    ptx::prefetch_tensormap(&p.tm_v);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp >= 8) {
    ptx::setmaxnreg_dec<kControlRegs>();
    if (warp == kLoadWarp) {
      fwd_producer<D, E>(p, sbase, ctl);
    } else if (warp == kMmaWarp) {
      fwd_mma<D, E>(p, sbase, tmem, ctl);
    }
  } else {
    ptx::setmaxnreg_inc<kSoftmaxRegs>();
    fwd_softmax<D, E>(p, warp / 4, sbase, tmem, ctl);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
