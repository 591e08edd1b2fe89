// Kernel parameter blocks, shared by the host launch code and the kernels.
// Passed by value as __grid_constant__, so the TMA descriptors they hold live in
// kernel parameter space (64-byte aligned, as TMA requires).
#pragma once

#include <cuda.h>
#include <cstdint>

namespace fa {

struct FwdParams {
  CUtensorMap tm_q;   // 3-D {d, N, B*H}, box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  void* o;            // [B, H, N, d], same 16-bit type as Q
  float* lse;         // [B, H, N] or nullptr
  unsigned int* status;
  unsigned long long timeout_ns;
  float scale_log2;   // scale * log2(e)
  int N;
  int BH;
  int n_qblk;         // ceil(N / 256)
  int num_units;      // BH * n_qblk
  int causal;
  int dbg_skip_load;  // K/V load index the producer leaves out (fault-path test), -1 = none
};

}  // namespace fa
