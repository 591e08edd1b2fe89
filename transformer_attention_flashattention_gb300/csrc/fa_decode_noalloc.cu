// fa_decode_noalloc: the decode entry point for callers that cannot allocate
// device memory (a plugin that the host program gives only its input and output
// buffers, a serving loop that must not allocate after start-up).  Its split
// scratch is a fixed device array inside this library rather than a
// caller-provided workspace; everything else is fa_decode, called unchanged.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_launch.h"

namespace {

// One array per device, reserved when this library's device code is loaded there.
// The 256-byte alignment meets fa_decode's workspace rule.
__device__ __align__(256) unsigned char g_decode_scratch[FA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxScratchDevices] = {};

// Device address of the current device's array; looked up once per device.
int scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr) return FA_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *addr = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_decode_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                 int H, int Nq, int Nk, int d, float scale, int causal, int dtype,
                                 int num_splits, void* stream) {
  // fa_decode's own argument checks, in its order, so that a bad call returns the code
  // fa_decode would return rather than FA_ERR_WORKSPACE (and does no device set-up)
  if (!q || !k || !v || !o) return FA_ERR_NULL;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return FA_ERR_UNSUPPORTED;
  int st = fa::check_decode(B, H, Nq, Nk, d);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_UNSUPPORTED;
  auto misaligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) || (lse && misaligned(lse, 4)))
    return FA_ERR_ALIGN;
  unsigned long long need = 0;
  st = fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits, &need);
  if (st != FA_OK) return st;
  if (need > FA_DECODE_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  // the look-up runs on the first call on a device whatever `need` is, so that
  // later calls never do set-up work
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  // every partial slot the merge reads is written first by the split kernel of
  // the same call, so the array is never cleared
  return fa_decode(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, num_splits, scratch,
                   FA_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
