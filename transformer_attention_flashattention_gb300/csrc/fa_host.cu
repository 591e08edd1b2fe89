// fa_fwd_host: the attention forward on HOST buffers, with the host<->device copies
// overlapped with the computation.
//
// The heads are cut into chunks.  Chunk c's Q, K, V go to the device on one copy
// stream, its fa_fwd runs on the caller's stream once they have landed, and its O
// and LSE come back on a second copy stream once it is done.  The link carries chunk
// c+1 in while chunk c computes and chunk c-1 goes out, so a call costs about one
// pass of the inputs over the link instead of inputs + compute + outputs in a row.
// The device copies live in a caller-provided workspace; the copy streams and
// events are created once per device and reused.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fa.h"

namespace {

constexpr int kMaxHostDevices = 64;
constexpr int kMaxChunks = 32;
constexpr int kAutoChunks = 8;

struct CopyEngine {
  bool ready = false;
  cudaStream_t h2d = nullptr;
  cudaStream_t d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t out_done = nullptr;
  cudaEvent_t in[kMaxChunks] = {};
  cudaEvent_t computed[kMaxChunks] = {};
};

std::mutex g_host_mu;
CopyEngine g_engine[kMaxHostDevices];

// The current device's copy streams and events, created on first use (caller holds g_host_mu).
int engine(CopyEngine** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxHostDevices) return FA_ERR_CUDA;
  CopyEngine& e = g_engine[dev];
  if (!e.ready) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&e.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&e.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&e.start, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&e.out_done, ef) != cudaSuccess)
      return FA_ERR_CUDA;
    for (int i = 0; i < kMaxChunks; ++i)
      if (cudaEventCreateWithFlags(&e.in[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&e.computed[i], ef) != cudaSuccess)
        return FA_ERR_CUDA;
    e.ready = true;
  }
  *out = &e;
  return FA_OK;
}

unsigned long long round256(unsigned long long x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" int fa_fwd_host_workspace_size(int B, int H, int N, int d, unsigned long long* bytes) {
  if (!bytes) return FA_ERR_NULL;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const unsigned long long elems = static_cast<unsigned long long>(B) * H * N * d;
  const unsigned long long rows = static_cast<unsigned long long>(B) * H * N;
  *bytes = 4 * round256(2 * elems) + round256(4 * rows);   // Q, K, V, O (16-bit) and LSE
  return FA_OK;
}

extern "C" int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                           int N, int d, float scale, int causal, int dtype, int chunks, void* workspace,
                           unsigned long long workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !workspace) return FA_ERR_NULL;
  unsigned long long need = 0;
  int st = fa_fwd_host_workspace_size(B, H, N, d, &need);
  if (st != FA_OK) return st;
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return FA_ERR_ALIGN;
  if (chunks < 0 || (dtype != FA_F16 && dtype != FA_BF16) || (causal != 0 && causal != 1) ||
      !(scale > 0.f) || !(scale < 3.4e38f))
    return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  int nc = chunks == 0 ? kAutoChunks : chunks;
  if (nc > kMaxChunks) nc = kMaxChunks;
  if (nc > BH) nc = static_cast<int>(BH);
  const long long per_chunk = (BH + nc - 1) / nc;

  const unsigned long long head_bytes = 2ull * N * d;
  const unsigned long long tensor_bytes = round256(BH * head_bytes);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* dq = base;
  uint8_t* dk = base + tensor_bytes;
  uint8_t* dv = base + 2 * tensor_bytes;
  uint8_t* dO = base + 3 * tensor_bytes;
  float* dl = reinterpret_cast<float*>(base + 4 * tensor_bytes);
  const uint8_t* hq = static_cast<const uint8_t*>(q);
  const uint8_t* hk = static_cast<const uint8_t*>(k);
  const uint8_t* hv = static_cast<const uint8_t*>(v);
  uint8_t* ho = static_cast<uint8_t*>(o);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // one call's enqueue at a time per process: the events are shared
  std::lock_guard<std::mutex> lock(g_host_mu);
  CopyEngine* e = nullptr;
  st = engine(&e);
  if (st != FA_OK) return st;
  // the workspace may still be in use by earlier work on the caller's stream
  if (cudaEventRecord(e->start, s) != cudaSuccess || cudaStreamWaitEvent(e->h2d, e->start, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  for (int c = 0; c < nc; ++c) {
    const long long h0 = c * per_chunk;
    const long long hn = BH - h0 < per_chunk ? BH - h0 : per_chunk;
    if (hn <= 0) break;
    const unsigned long long off = static_cast<unsigned long long>(h0) * head_bytes;
    const unsigned long long len = static_cast<unsigned long long>(hn) * head_bytes;
    if (cudaMemcpyAsync(dq + off, hq + off, len, cudaMemcpyHostToDevice, e->h2d) != cudaSuccess ||
        cudaMemcpyAsync(dk + off, hk + off, len, cudaMemcpyHostToDevice, e->h2d) != cudaSuccess ||
        cudaMemcpyAsync(dv + off, hv + off, len, cudaMemcpyHostToDevice, e->h2d) != cudaSuccess ||
        cudaEventRecord(e->in[c], e->h2d) != cudaSuccess || cudaStreamWaitEvent(s, e->in[c], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    st = fa_fwd(dq + off, dk + off, dv + off, dO + off, lse ? dl + h0 * N : nullptr, 1, static_cast<int>(hn), N,
                d, scale, causal, dtype, s);
    if (st != FA_OK) return st;
    if (cudaEventRecord(e->computed[c], s) != cudaSuccess ||
        cudaStreamWaitEvent(e->d2h, e->computed[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(ho + off, dO + off, len, cudaMemcpyDeviceToHost, e->d2h) != cudaSuccess)
      return FA_ERR_CUDA;
    if (lse && cudaMemcpyAsync(lse + h0 * N, dl + h0 * N, static_cast<size_t>(hn) * N * sizeof(float),
                               cudaMemcpyDeviceToHost, e->d2h) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  // the caller's stream resumes once the last result is on the host
  if (cudaEventRecord(e->out_done, e->d2h) != cudaSuccess || cudaStreamWaitEvent(s, e->out_done, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}
