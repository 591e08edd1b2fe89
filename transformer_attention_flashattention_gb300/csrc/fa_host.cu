// fa_fwd_host and fa_fwd_fp8_host: the attention forward on HOST buffers, with the
// host<->device copies overlapped with the computation.
//
// The heads are cut into chunks.  Chunk c's Q, K, V go to the device on one copy
// stream, its fa_fwd runs on one of two compute streams (in turn) once they have
// landed, and its O and LSE come back on a second copy stream once it is done.  The
// link carries chunk c+1 in while chunk c computes and chunk c-1 goes out, so a call
// costs about one pass of the inputs over the link instead of inputs + compute +
// outputs in a row.  The two compute streams let chunk c+1's persistent grid take the
// SMs that chunk c's last CTAs leave idle (a chunk of a few heads is only a few units
// per SM, so each launch alone would end on a ragged last wave).
// The device copies live in a caller-provided workspace; the copy streams and
// events are created once per device and reused.  The FP8 variant runs the E4M3
// prologue (one launch for Q, K and V) and the E4M3 forward on each chunk.
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
  cudaStream_t comp[2] = {nullptr, nullptr};
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
        cudaStreamCreateWithFlags(&e.comp[0], cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&e.comp[1], cudaStreamNonBlocking) != cudaSuccess ||
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

// Head counts of the chunks; returns how many.  `chunks` > 0: that many equal chunks (the
// last one shorter).  0: chunks that grow 1, 2, 4, ... heads up to a cap of BH / 8 and
// shrink the same way at the end, so that only a small first chunk's inputs and a small
// last chunk's outputs cross the link while nothing computes; equal chunks of BH / 8
// where BH is too small (or too large) for that.
int chunk_sizes(long long BH, int chunks, long long (&size)[kMaxChunks]) {
  if (chunks == 0) {
    const long long cap = (BH + kAutoChunks - 1) / kAutoChunks;
    long long ramp[kMaxChunks];
    int nr = 0;
    long long ramp_sum = 0;
    for (long long h = 1; h < cap && nr < 8; h *= 2) {
      ramp[nr++] = h;
      ramp_sum += h;
    }
    const long long middle = BH - 2 * ramp_sum;
    const long long nm = middle > 0 ? (middle + cap - 1) / cap : 0;
    if (nr > 0 && middle > 0 && 2 * nr + nm <= kMaxChunks) {
      int n = 0;
      for (int i = 0; i < nr; ++i) size[n++] = ramp[i];
      for (long long left = middle; left > 0; left -= cap) size[n++] = left < cap ? left : cap;
      for (int i = nr - 1; i >= 0; --i) size[n++] = ramp[i];
      return n;
    }
  }
  int nc = chunks == 0 ? kAutoChunks : chunks;
  if (nc > kMaxChunks) nc = kMaxChunks;
  if (nc > BH) nc = static_cast<int>(BH);
  const long long per_chunk = (BH + nc - 1) / nc;
  int n = 0;
  for (long long h0 = 0; h0 < BH; h0 += per_chunk) size[n++] = BH - h0 < per_chunk ? BH - h0 : per_chunk;
  return n;
}

// The chunked schedule shared by both entry points.  `compute(h0, hn, cs)` enqueues the
// work on heads h0 .. h0+hn-1 on stream cs, after their inputs landed; the
// three inputs are `in_bytes` per head from the host to `dev_in[i]`, and `out_bytes` per
// head of O (plus N floats of LSE when `lse`) come back from `dev_o` / `dev_lse`.
template <class Compute>
int run_chunked(const void* const host_in[3], uint8_t* const dev_in[3], unsigned long long in_bytes,
                void* host_o, const uint8_t* dev_o, unsigned long long out_bytes, float* host_lse,
                const float* dev_lse, long long BH, int N, int chunks, cudaStream_t s, Compute compute) {
  long long size[kMaxChunks];
  const int nc = chunk_sizes(BH, chunks, size);
  // one call's enqueue at a time per process: the events are shared
  std::lock_guard<std::mutex> lock(g_host_mu);
  CopyEngine* e = nullptr;
  int st = engine(&e);
  if (st != FA_OK) return st;
  // the workspace may still be in use by earlier work on the caller's stream
  if (cudaEventRecord(e->start, s) != cudaSuccess || cudaStreamWaitEvent(e->h2d, e->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(e->comp[0], e->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(e->comp[1], e->start, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  long long h0 = 0;
  for (int c = 0; c < nc; h0 += size[c], ++c) {
    const long long hn = size[c];
    for (int i = 0; i < 3; ++i)
      if (cudaMemcpyAsync(dev_in[i] + h0 * in_bytes, static_cast<const uint8_t*>(host_in[i]) + h0 * in_bytes,
                          hn * in_bytes, cudaMemcpyHostToDevice, e->h2d) != cudaSuccess)
        return FA_ERR_CUDA;
    cudaStream_t cs = e->comp[c & 1];
    if (cudaEventRecord(e->in[c], e->h2d) != cudaSuccess || cudaStreamWaitEvent(cs, e->in[c], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    st = compute(h0, hn, cs);
    if (st != FA_OK) return st;
    if (cudaEventRecord(e->computed[c], cs) != cudaSuccess ||
        cudaStreamWaitEvent(e->d2h, e->computed[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(host_o) + h0 * out_bytes, dev_o + h0 * out_bytes, hn * out_bytes,
                        cudaMemcpyDeviceToHost, e->d2h) != cudaSuccess)
      return FA_ERR_CUDA;
    if (host_lse && cudaMemcpyAsync(host_lse + h0 * N, dev_lse + h0 * N, static_cast<size_t>(hn) * N * sizeof(float),
                                    cudaMemcpyDeviceToHost, e->d2h) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  // the caller's stream resumes once the last result is on the host (the copy stream
  // ran every chunk's copy after that chunk's computation)
  if (cudaEventRecord(e->out_done, e->d2h) != cudaSuccess || cudaStreamWaitEvent(s, e->out_done, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

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
  const unsigned long long head_bytes = 2ull * N * d;
  const unsigned long long tensor_bytes = round256(BH * head_bytes);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* const dev_in[3] = {base, base + tensor_bytes, base + 2 * tensor_bytes};
  uint8_t* dO = base + 3 * tensor_bytes;
  float* dl = reinterpret_cast<float*>(base + 4 * tensor_bytes);
  const void* const host_in[3] = {q, k, v};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return run_chunked(host_in, dev_in, head_bytes, o, dO, head_bytes, lse, dl, BH, N, chunks, s,
                     [&](long long h0, long long hn, cudaStream_t cs) {
                       const unsigned long long off = static_cast<unsigned long long>(h0) * head_bytes;
                       return fa_fwd(dev_in[0] + off, dev_in[1] + off, dev_in[2] + off, dO + off,
                                     lse ? dl + h0 * N : nullptr, 1, static_cast<int>(hn), N, d, scale, causal,
                                     dtype, cs);
                     });
}

extern "C" int fa_fwd_fp8_host_workspace_size(int B, int H, int N, int d, unsigned long long* bytes) {
  if (!bytes) return FA_ERR_NULL;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (N % 16 != 0) return FA_ERR_SHAPE;
  const unsigned long long elems = static_cast<unsigned long long>(B) * H * N * d;
  const unsigned long long rows = static_cast<unsigned long long>(B) * H * N;
  const unsigned long long nsb = static_cast<unsigned long long>(B) * H * ((N + 63) / 64);
  // bf16 Q, K, V and O; E4M3 Q, K, V^T; three scale arrays; LSE
  *bytes = 4 * round256(2 * elems) + 3 * round256(elems) + 3 * round256(4 * nsb) + round256(4 * rows);
  return FA_OK;
}

extern "C" int fa_fwd_fp8_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                               int N, int d, float scale, int causal, int hadamard, int chunks, void* workspace,
                               unsigned long long workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !workspace) return FA_ERR_NULL;
  unsigned long long need = 0;
  int st = fa_fwd_fp8_host_workspace_size(B, H, N, d, &need);
  if (st != FA_OK) return st;
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return FA_ERR_ALIGN;
  if (chunks < 0 || (causal != 0 && causal != 1) || (hadamard != 0 && hadamard != 1) || !(scale > 0.f) ||
      !(scale < 3.4e38f))
    return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  const int nsb = (N + 63) / 64;
  const unsigned long long head_elems = static_cast<unsigned long long>(N) * d;
  const unsigned long long t16 = round256(BH * 2 * head_elems), t8 = round256(BH * head_elems);
  const unsigned long long ts = round256(4ull * BH * nsb);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* const dev_in[3] = {base, base + t16, base + 2 * t16};
  uint8_t* dO = base + 3 * t16;
  uint8_t* x8[3];
  float* sc[3];
  for (int i = 0; i < 3; ++i) {
    x8[i] = base + 4 * t16 + i * t8;
    sc[i] = reinterpret_cast<float*>(base + 4 * t16 + 3 * t8 + i * ts);
  }
  float* dl = reinterpret_cast<float*>(base + 4 * t16 + 3 * t8 + 3 * ts);
  const void* const host_in[3] = {q, k, v};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return run_chunked(host_in, dev_in, 2 * head_elems, o, dO, 2 * head_elems, lse, dl, BH, N, chunks, s,
                     [&](long long h0, long long hn, cudaStream_t cs) {
                       const unsigned long long o16 = h0 * 2 * head_elems, o8 = h0 * head_elems;
                       const long long os = h0 * nsb;
                       const int n = static_cast<int>(hn);
                       // Q, K rotated; V transposed, not rotated: one launch
                       const int r = fa_quantize_fp8_qkv(dev_in[0] + o16, dev_in[1] + o16, dev_in[2] + o16,
                                                         x8[0] + o8, x8[1] + o8, x8[2] + o8, sc[0] + os,
                                                         sc[1] + os, sc[2] + os, 1, n, N, d, hadamard, cs);
                       if (r != FA_OK) return r;
                       return fa_fwd_fp8(x8[0] + o8, x8[1] + o8, x8[2] + o8, dO + o16, lse ? dl + h0 * N : nullptr,
                                         1, n, N, d, scale, causal, sc[0] + os, sc[1] + os, sc[2] + os, hadamard, cs);
                     });
}
