// Kernel parameter blocks, shared by the host launch code and the kernels.
// Passed by value as __grid_constant__, so the TMA descriptors they hold live in
// kernel parameter space (64-byte aligned, as TMA requires).
#pragma once

#include <cuda.h>
#include <cstdint>

namespace fa {

struct FwdParams {
  CUtensorMap tm_q;   // 3-D {d, N, B*H}, box {128 bytes of d, 128 rows, 1}, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;   // as Q for 16-bit inputs; E4M3: V^T, 3-D {N, d, B*H}, box {128, 128, 1}
  CUtensorMap tm_kh;  // CTA-pair kernel only: K with a 64-row box (half a key tile per CTA)
  void* o;            // [B, H, N, d]: the input type for 16-bit inputs, bf16 for E4M3
  float* lse;         // [B, H, N] or nullptr
  unsigned int* status;
  unsigned long long timeout_ns;
  float scale_log2;   // scale * log2(e)
  int N;
  int BH;
  int n_qblk;         // ceil(N / 256); the CTA-pair kernel: ceil(N / 512)
  int num_units;      // BH * n_qblk
  int causal;
  int dbg_skip_load;  // K/V load index the producer leaves out (fault-path test), -1 = none
  // E4M3 path only: per-(b*h, 64-row block) dequantisation scales, [B*H, n_sblk]
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  int n_sblk;         // ceil(N / 64)
};

// FP8 prologue: block absmax E4M3 quantisation with an optional Hadamard rotation, of
// one tensor or of up to three tensors of the same shape in one launch (Q, K and V).
struct QuantParams {
  const void* x[3];       // bf16 [B*H, N, d] per tensor
  uint8_t* x8[3];         // e4m3 [B*H, N, d], or [B*H, d, N] when that tensor's transpose_out
  float* scale[3];        // [B*H, n_sblk] per tensor
  int hadamard[3];
  int transpose_out[3];
  int ntens;              // tensors in this launch, 1..3
  int N;
  int d;
  int BH;
  int n_sblk;
  unsigned long long flips_lo;   // randomised rotation: bit c negates coordinate c (c < 64) ...
  unsigned long long flips_hi;   // ... and c - 64 (64 <= c < 128) before the transform
  int per_head;                  // one absmax per (b, h) instead of per 64-row block (one tensor)
  int amax_mode;                 // 0: own block absmax; 1: write the block absmax only;
                                 // 2: quantise with the absmax already in `scale`
  int sm_count;                  // SMs of the device; the persistent grid is a multiple of it
  unsigned int* status;
  unsigned long long timeout_ns;
};

// Split-KV attention of N_q query rows against N_k cached keys.
struct DecodeParams {
  CUtensorMap tm_k;   // 3-D {d, Nk, B*H}, box {64, 64, 1}, 128-byte swizzle
  CUtensorMap tm_v;
  const void* q;      // [B*H, Nq, d]
  const void* k;      // [B*H, Nk, d]
  const void* v;
  void* o;            // [B*H, Nq, d]
  float* lse;         // [B*H, Nq] or nullptr
  float* part_o;      // scratch [B*H, splits, Nq, d] (splits > 1)
  float* part_lse;    // scratch [B*H, splits, Nq]
  unsigned int* status;
  unsigned long long timeout_ns;
  float scale_log2;
  int BH;
  int Nq;
  int Nk;
  int splits;
  int chunk;          // keys per split, a multiple of 64
  int causal;
};

// Attention backward: dQ, dK, dV from Q, K, V, O, LSE and dO.
struct BwdParams {
  CUtensorMap tm_q;   // 3-D {d, N, B*H}, box {128 bytes of d, 128 rows, 1}, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  // d = 128: the epilogues' TMA stores of dQ, dK and dV, box {128 bytes of d, 32 rows, 1}
  // (one compute warp's slice), 128-byte swizzle
  CUtensorMap tm_dq;
  CUtensorMap tm_dk;
  CUtensorMap tm_dv;
  const void* o;      // [B*H, N, d] (prep kernel)
  const void* dout;   // [B*H, N, d] (prep kernel)
  const float* lse;   // [B*H, N] natural-log LSE of the forward pass
  float* nlse2;       // workspace [B*H, n_pad]: -lse * log2(e), -inf on padded rows
  float* ndelta;      // workspace [B*H, n_pad]: -sum_c dO_ic O_ic, 0 on padded rows
  void* dq;           // [B*H, N, d], same type as the inputs
  void* dk;
  void* dv;
  unsigned int* status;
  unsigned long long timeout_ns;
  float scale;
  float scale_log2;   // scale * log2(e)
  int N;
  int n_pad;          // N rounded up to 128
  int BH;
  int n_blk;          // ceil(N / 128): Q tiles = K/V tiles per head
  int num_units;      // BH * n_blk (each kernel)
  int causal;
};

}  // namespace fa
