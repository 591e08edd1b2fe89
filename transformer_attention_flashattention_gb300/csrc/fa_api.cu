// C ABI of libfa.so: argument validation, TMA descriptor encoding, launch, status.
// The operations and their contracts are documented in include/fa.h.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_launch.h"
#include "fa_params.h"

namespace fa {

// Per-device word that kernels set when a bounded wait gives up.
__device__ unsigned int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kUnitRows = 256;   // query rows per forward work unit (two 128-row tiles)

struct DeviceInfo {
  bool probed = false;
  bool is_sm103 = false;
  int sm_count = 0;
  unsigned int* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
int g_dbg_skip_load = -1;
int g_dbg_timeout_ms = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Current device's cached properties (probed once); nullptr if a CUDA call failed.
const DeviceInfo* current_device(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = FA_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      *status = FA_ERR_CUDA;
      return nullptr;
    }
    di.is_sm103 = (major == 10 && minor == 3);
    di.sm_count = sms;
    if (di.is_sm103) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) {
        *status = FA_ERR_CUDA;
        return nullptr;
      }
      di.status = static_cast<unsigned int*>(ptr);
    }
    if (g_encode == nullptr) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        *status = FA_ERR_CUDA;
        return nullptr;
      }
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    di.probed = true;
  }
  if (!di.is_sm103) {
    *status = FA_ERR_ARCH;
    return nullptr;
  }
  *status = FA_OK;
  return &di;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 3-D tiled map over a contiguous [outer, rows, inner] tensor, box {box_inner, box_rows, 1},
// 128-byte swizzle, out-of-bounds elements read as zero.
bool encode_3d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base,
               uint64_t inner, uint64_t rows, uint64_t outer, uint32_t box_inner, uint32_t box_rows) {
  const cuuint64_t dims[3] = {inner, rows, outer};
  const cuuint64_t strides[2] = {inner * elem_bytes, inner * rows * elem_bytes};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned long long timeout_ns_for_call() {
  if (g_dbg_timeout_ms > 0) return static_cast<unsigned long long>(g_dbg_timeout_ms) * 1000000ull;
  const char* env = std::getenv("FA_TIMEOUT_MS");
  long ms = env ? std::strtol(env, nullptr, 10) : 0;
  if (ms <= 0) ms = 2000;
  return static_cast<unsigned long long>(ms) * 1000000ull;
}

int check_shape(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long double total = static_cast<long double>(B) * H * N * d;
  if (total >= static_cast<long double>(1ull << 40)) return FA_ERR_SHAPE;
  if (static_cast<long long>(B) * H >= (1ll << 31)) return FA_ERR_SHAPE;
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

namespace {

// fa_fwd and fa_fwd_2cta: the same checks and parameters; `pair` selects the CTA-pair
// kernel (head dim 128 only, 512-row units, two CTAs a cluster).
int fwd_call(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             float scale, int causal, int dtype, void* stream, bool pair) {
  if (!q || !k || !v || !o) return FA_ERR_NULL;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return FA_ERR_UNSUPPORTED;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (pair && d != 128) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (lse && !aligned(lse, 4)))
    return FA_ERR_ALIGN;

  const DeviceInfo* di = current_device(&st);
  if (!di) return st;

  FwdParams p;
  const CUtensorMapDataType dt = dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t BH = static_cast<uint64_t>(B) * H;
  if (!encode_3d(&p.tm_q, dt, 2, q, d, N, BH, 64, 128) || !encode_3d(&p.tm_k, dt, 2, k, d, N, BH, 64, 128) ||
      !encode_3d(&p.tm_v, dt, 2, v, d, N, BH, 64, 128) || !encode_3d(&p.tm_kh, dt, 2, k, d, N, BH, 64, 64))
    return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.status = di->status;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.N = N;
  p.BH = static_cast<int>(BH);
  // head dim 64 (16-bit) runs one 128-row Q tile per CTA, two CTAs per SM
  const bool one_tile = !pair && d == 64;
  const int unit_rows = pair ? 2 * kUnitRows : (one_tile ? kUnitRows / 2 : kUnitRows);
  p.n_qblk = (N + unit_rows - 1) / unit_rows;
  const long long units = static_cast<long long>(p.n_qblk) * p.BH;
  if (units >= (1ll << 31)) return FA_ERR_SHAPE;
  p.num_units = static_cast<int>(units);
  p.causal = causal;
  p.q_scale = p.k_scale = p.v_scale = nullptr;
  p.n_sblk = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    p.timeout_ns = timeout_ns_for_call();
    p.dbg_skip_load = g_dbg_skip_load;
    g_dbg_skip_load = -1;
    g_dbg_timeout_ms = 0;
  }
  cudaError_t e;
  if (pair) {
    const long long pairs = di->sm_count / 2;
    const int grid = 2 * static_cast<int>(units < pairs ? units : pairs);
    e = launch_fwd2(dtype == FA_BF16, p, grid, static_cast<cudaStream_t>(stream));
  } else if (one_tile) {
    const long long slots = 2ll * di->sm_count;
    const int grid = static_cast<int>(units < slots ? units : slots);
    e = launch_fwd1(dtype == FA_BF16, p, grid, static_cast<cudaStream_t>(stream));
  } else {
    const int grid = static_cast<int>(units < di->sm_count ? units : di->sm_count);
    e = launch_fwd(d, dtype == FA_BF16, p, grid, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                      int N, int d, float scale, int causal, int dtype, void* stream) {
  return fwd_call(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream, false);
}

extern "C" int fa_fwd_2cta(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                           int N, int d, float scale, int causal, int dtype, void* stream) {
  return fwd_call(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream, true);
}

namespace fa {
namespace {

int quantize_fp8(const void* x, void* x8, float* scale, int B, int H, int N, int d, int hadamard,
                 unsigned long long flips_lo, unsigned long long flips_hi, int per_head, int transpose_out,
                 void* stream) {
  if (!x || !x8 || !scale) return FA_ERR_NULL;
  if ((hadamard != 0 && hadamard != 1) || (transpose_out != 0 && transpose_out != 1) ||
      (per_head != 0 && per_head != 1))
    return FA_ERR_UNSUPPORTED;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  // sign flips only make sense with the rotation, and only on the d coordinates
  if ((flips_lo | flips_hi) != 0 && (!hadamard || (d == 64 && flips_hi != 0))) return FA_ERR_UNSUPPORTED;
  if (transpose_out && N % 16 != 0) return FA_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(scale, 4)) return FA_ERR_ALIGN;
  const DeviceInfo* di = current_device(&st);
  if (!di) return st;
  QuantParams p = {};
  p.x[0] = x;
  p.x8[0] = static_cast<uint8_t*>(x8);
  p.scale[0] = scale;
  p.hadamard[0] = hadamard;
  p.transpose_out[0] = transpose_out;
  p.ntens = 1;
  p.N = N;
  p.d = d;
  p.BH = B * H;
  p.n_sblk = (N + 63) / 64;
  p.flips_lo = flips_lo;
  p.flips_hi = flips_hi;
  p.per_head = per_head;
  p.amax_mode = 0;
  p.sm_count = di->sm_count;
  p.status = di->status;
  p.timeout_ns = timeout_ns_for_call();
  const cudaError_t e = launch_quant_fp8(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace
}  // namespace fa

extern "C" int fa_quantize_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8t,
                                   float* q_scale, float* k_scale, float* v_scale, int B, int H, int N, int d,
                                   int hadamard, void* stream) {
  if (!q || !k || !v || !q8 || !k8 || !v8t || !q_scale || !k_scale || !v_scale) return FA_ERR_NULL;
  if (hadamard != 0 && hadamard != 1) return FA_ERR_UNSUPPORTED;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (N % 16 != 0) return FA_ERR_SHAPE;                    // V is written transposed
  const void* xs[3] = {q, k, v};
  void* x8s[3] = {q8, k8, v8t};
  float* scs[3] = {q_scale, k_scale, v_scale};
  for (int i = 0; i < 3; ++i)
    if (!aligned(xs[i], 16) || !aligned(x8s[i], 16) || !aligned(scs[i], 4)) return FA_ERR_ALIGN;
  const DeviceInfo* di = current_device(&st);
  if (!di) return st;
  QuantParams p = {};
  for (int i = 0; i < 3; ++i) {
    p.x[i] = xs[i];
    p.x8[i] = static_cast<uint8_t*>(x8s[i]);
    p.scale[i] = scs[i];
    p.hadamard[i] = i < 2 ? hadamard : 0;                  // Q and K rotated, V never
    p.transpose_out[i] = i == 2 ? 1 : 0;                   // V transposed for the P.V MMA
  }
  p.ntens = 3;
  p.N = N;
  p.d = d;
  p.BH = B * H;
  p.n_sblk = (N + 63) / 64;
  p.amax_mode = 0;
  p.sm_count = di->sm_count;
  p.status = di->status;
  p.timeout_ns = timeout_ns_for_call();
  const cudaError_t e = launch_quant_fp8(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

extern "C" int fa_quantize_fp8(const void* x, void* x8, float* scale, int B, int H, int N, int d,
                               int hadamard, int transpose_out, void* stream) {
  return fa::quantize_fp8(x, x8, scale, B, H, N, d, hadamard, 0, 0, 0, transpose_out, stream);
}

extern "C" int fa_quantize_fp8_ex(const void* x, void* x8, float* scale, int B, int H, int N, int d,
                                  int hadamard, unsigned long long sign_flips_lo,
                                  unsigned long long sign_flips_hi, int per_head, int transpose_out,
                                  void* stream) {
  return fa::quantize_fp8(x, x8, scale, B, H, N, d, hadamard, sign_flips_lo, sign_flips_hi, per_head,
                          transpose_out, stream);
}

extern "C" int fa_fwd_fp8(const void* q8, const void* k8, const void* v8t, void* o, float* lse, int B,
                          int H, int N, int d, float scale, int causal, const float* q_scale,
                          const float* k_scale, const float* v_scale, int hadamard, void* stream) {
  if (!q8 || !k8 || !v8t || !o || !q_scale || !k_scale || !v_scale) return FA_ERR_NULL;
  if ((causal != 0 && causal != 1) || (hadamard != 0 && hadamard != 1)) return FA_ERR_UNSUPPORTED;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (N % 16 != 0) return FA_ERR_SHAPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_UNSUPPORTED;
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(v8t, 16) || !aligned(o, 16) ||
      (lse && !aligned(lse, 4)) || !aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return FA_ERR_ALIGN;
  const DeviceInfo* di = current_device(&st);
  if (!di) return st;

  FwdParams p;
  const uint64_t BH = static_cast<uint64_t>(B) * H;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (!encode_3d(&p.tm_q, u8, 1, q8, d, N, BH, 128, 128) || !encode_3d(&p.tm_k, u8, 1, k8, d, N, BH, 128, 128) ||
      !encode_3d(&p.tm_v, u8, 1, v8t, N, d, BH, 128, 128))
    return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.status = di->status;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.N = N;
  p.BH = static_cast<int>(BH);
  p.n_qblk = (N + kUnitRows - 1) / kUnitRows;
  const long long units = static_cast<long long>(p.n_qblk) * p.BH;
  if (units >= (1ll << 31)) return FA_ERR_SHAPE;
  p.num_units = static_cast<int>(units);
  p.causal = causal;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.n_sblk = (N + 63) / 64;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    p.timeout_ns = timeout_ns_for_call();
    p.dbg_skip_load = -1;
  }
  const int grid = static_cast<int>(units < di->sm_count ? units : di->sm_count);
  const cudaError_t e = launch_fwd_fp8(p, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

namespace fa {
namespace {

constexpr int kDecodeMaxQ = 16;

unsigned long long decode_workspace(int BH, int Nq, int d, int splits) {
  if (splits <= 1) return 0;
  const unsigned long long o = static_cast<unsigned long long>(BH) * splits * Nq * d * 4;
  const unsigned long long l = static_cast<unsigned long long>(BH) * splits * Nq * 4;
  return (o + 255) / 256 * 256 + l;
}

// Key chunks per head.  Two split CTAs share an SM at d = 64 and, with at most 4 query
// rows, at d = 128 (registers and a 96 KB ring each); one fills an SM at d = 128 with more
// rows.  So B*H*splits CTAs run in waves of `slots`.  With splits = 0 the
// count minimises  waves * (64-key tiles per chunk + 4 tiles of per-CTA overhead),
// taking the fewest splits within 2 % of the best, with chunks of at least 256 keys
// and at most 4 MiB of split scratch (so that every automatic choice also fits the
// static area of fa_decode_noalloc).
constexpr unsigned long long kAutoSplitScratch = 4ull << 20;

void decode_split(int BH, int Nq, int Nk, int d, int requested, int sm_count, int* splits, int* chunk) {
  auto shape = [&](int s, int* c_out) {
    int c = (Nk + s - 1) / s;
    c = (c + 63) / 64 * 64;
    *c_out = c;
    return (Nk + c - 1) / c;
  };
  if (requested > 0) {
    *splits = shape(requested, chunk);
    return;
  }
  const long long slots = static_cast<long long>(sm_count) * (d == 64 || Nq <= 4 ? 2 : 1);
  int s_max = Nk / 256;
  if (s_max > 128) s_max = 128;
  if (s_max < 1) s_max = 1;
  long long cost[129];
  long long best = -1;
  for (int s = 1; s <= s_max; ++s) {
    int c;
    const int sp = shape(s, &c);
    cost[s] = -1;
    if (sp > 1 && decode_workspace(BH, Nq, d, sp) > kAutoSplitScratch) continue;
    cost[s] = ((static_cast<long long>(BH) * sp + slots - 1) / slots) * (c / 64 + 4);
    if (best < 0 || cost[s] < best) best = cost[s];
  }
  for (int s = 1; s <= s_max; ++s) {
    if (cost[s] >= 0 && cost[s] * 50 <= best * 51) {
      *splits = shape(s, chunk);
      return;
    }
  }
  *splits = shape(1, chunk);
}

}  // namespace

int check_decode(int B, int H, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (Nq > kDecodeMaxQ || Nq > Nk) return FA_ERR_SHAPE;
  if (static_cast<long double>(B) * H * Nk * d >= static_cast<long double>(1ull << 40)) return FA_ERR_SHAPE;
  if (static_cast<long long>(B) * H * 4096 >= (1ll << 31)) return FA_ERR_SHAPE;
  return FA_OK;
}

}  // namespace fa

extern "C" int fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits,
                                        unsigned long long* bytes) {
  if (!bytes) return FA_ERR_NULL;
  int st = check_decode(B, H, Nq, Nk, d);
  if (st != FA_OK) return st;
  const DeviceInfo* di = current_device(&st);
  if (!di) return st;
  int splits, chunk;
  decode_split(B * H, Nq, Nk, d, num_splits, di->sm_count, &splits, &chunk);
  *bytes = decode_workspace(B * H, Nq, d, splits);
  return FA_OK;
}

extern "C" int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                         int Nq, int Nk, int d, float scale, int causal, int dtype, int num_splits,
                         void* workspace, unsigned long long workspace_bytes, void* stream) {
  if (!q || !k || !v || !o) return FA_ERR_NULL;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return FA_ERR_UNSUPPORTED;
  int st = check_decode(B, H, Nq, Nk, d);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)) ||
      (workspace && !aligned(workspace, 256)))
    return FA_ERR_ALIGN;
  const DeviceInfo* di = current_device(&st);
  if (!di) return st;
  DecodeParams p;
  const CUtensorMapDataType dt = dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!encode_3d(&p.tm_k, dt, 2, k, d, Nk, static_cast<uint64_t>(B) * H, 64, 64) ||
      !encode_3d(&p.tm_v, dt, 2, v, d, Nk, static_cast<uint64_t>(B) * H, 64, 64))
    return FA_ERR_CUDA;
  decode_split(B * H, Nq, Nk, d, num_splits, di->sm_count, &p.splits, &p.chunk);
  const unsigned long long need = decode_workspace(B * H, Nq, d, p.splits);
  if (need > 0 && (!workspace || workspace_bytes < need)) return FA_ERR_WORKSPACE;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.part_o = need ? static_cast<float*>(workspace) : nullptr;
  p.part_lse = need ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                               (static_cast<unsigned long long>(B) * H * p.splits * Nq * d * 4 + 255) / 256 * 256)
                    : nullptr;
  p.status = di->status;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.BH = B * H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.causal = causal;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    p.timeout_ns = timeout_ns_for_call();
  }
  const cudaError_t e = launch_decode(d, dtype == FA_BF16, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

extern "C" int fa_bwd_workspace_size(int B, int H, int N, int d, unsigned long long* bytes) {
  if (!bytes) return FA_ERR_NULL;
  const int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  const unsigned long long n_pad = (static_cast<unsigned long long>(N) + 127) / 128 * 128;
  *bytes = 2ull * static_cast<unsigned long long>(B) * H * n_pad * 4ull;
  return FA_OK;
}

extern "C" int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                      int causal, int dtype, void* workspace, unsigned long long workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return FA_ERR_NULL;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return FA_ERR_UNSUPPORTED;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(workspace, 256))
    return FA_ERR_ALIGN;
  unsigned long long need = 0;
  fa_bwd_workspace_size(B, H, N, d, &need);
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  const DeviceInfo* di = current_device(&st);
  if (!di) return st;

  BwdParams p;
  const CUtensorMapDataType dt = dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t BH = static_cast<uint64_t>(B) * H;
  if (!encode_3d(&p.tm_q, dt, 2, q, d, N, BH, 64, 128) || !encode_3d(&p.tm_k, dt, 2, k, d, N, BH, 64, 128) ||
      !encode_3d(&p.tm_v, dt, 2, v, d, N, BH, 64, 128) || !encode_3d(&p.tm_do, dt, 2, dout, d, N, BH, 64, 128))
    return FA_ERR_CUDA;
  if (d == 128 && (!encode_3d(&p.tm_dq, dt, 2, dq, d, N, BH, 64, 32) || !encode_3d(&p.tm_dk, dt, 2, dk, d, N, BH, 64, 32) ||
                   !encode_3d(&p.tm_dv, dt, 2, dv, d, N, BH, 64, 32)))
    return FA_ERR_CUDA;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.N = N;
  p.n_pad = (N + 127) / 128 * 128;
  p.n_blk = p.n_pad / 128;
  p.BH = static_cast<int>(BH);
  p.nlse2 = static_cast<float*>(workspace);
  p.ndelta = p.nlse2 + BH * static_cast<uint64_t>(p.n_pad);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = di->status;
  p.scale = scale;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.causal = causal;
  const long long units = static_cast<long long>(p.n_blk) * p.BH;
  if (units >= (1ll << 31)) return FA_ERR_SHAPE;
  p.num_units = static_cast<int>(units);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    p.timeout_ns = timeout_ns_for_call();
  }
  const int grid = static_cast<int>(units < di->sm_count ? units : di->sm_count);
  const cudaError_t e = launch_bwd(d, dtype == FA_BF16, p, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

namespace {
constexpr int kNaiveMaxN = 32768;   // the row softmax keeps a row in 256 threads' registers
constexpr unsigned long long kNaiveBlasWs = 32ull << 20;   // the cuBLAS GEMMs' scratch

// fp32 score row stride of the materialising path: N rounded up to whole float4 vectors.
long long naive_ld(int N) { return (static_cast<long long>(N) + 3) / 4 * 4; }
// bytes of the fp32 score matrices, rounded up to 256 (the GEMM scratch follows them)
unsigned long long naive_scores(int B, int H, int N) {
  return (static_cast<unsigned long long>(B) * H * N * static_cast<unsigned long long>(naive_ld(N)) * 4ull + 255) /
         256 * 256;
}
}  // namespace

extern "C" int fa_fwd_naive_workspace_size(int B, int H, int N, int d, unsigned long long* bytes) {
  if (!bytes) return FA_ERR_NULL;
  const int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (N > kNaiveMaxN) return FA_ERR_UNSUPPORTED;
  const long double rows = static_cast<long double>(B) * H * N;
  if (rows >= static_cast<long double>(1ll << 31)) return FA_ERR_SHAPE;
  *bytes = naive_scores(B, H, N) + kNaiveBlasWs;
  return FA_OK;
}

extern "C" int fa_fwd_naive(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                            int d, float scale, int causal, int dtype, void* workspace,
                            unsigned long long workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !workspace) return FA_ERR_NULL;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return FA_ERR_UNSUPPORTED;
  unsigned long long need = 0;
  int st = fa_fwd_naive_workspace_size(B, H, N, d, &need);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)) ||
      !aligned(workspace, 256))
    return FA_ERR_ALIGN;
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;
  const DeviceInfo* di = current_device(&st);
  if (!di) return st;
  uint8_t* const base = static_cast<uint8_t*>(workspace);
  return run_naive(q, k, v, o, lse, reinterpret_cast<float*>(base), naive_ld(N), base + naive_scores(B, H, N),
                   kNaiveBlasWs, B * H, N, d, scale, causal, dtype == FA_BF16, static_cast<cudaStream_t>(stream));
}

extern "C" int fa_last_device_status(void* stream, unsigned int* bits) {
  int st = FA_OK;
  const DeviceInfo* di = current_device(&st);
  if (!di) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  const unsigned int zero = 0;
  if (word != 0 && cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
    return FA_ERR_CUDA;
  if (bits) *bits = word;
  return word == 0 ? FA_OK : FA_ERR_DEVICE_TIMEOUT;
}

extern "C" int fa_debug_inject_stall(int load_index, int timeout_ms) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_dbg_skip_load = load_index < 0 ? -1 : load_index;
  g_dbg_timeout_ms = load_index < 0 ? 0 : (timeout_ms > 0 ? timeout_ms : 100);
  return FA_OK;
}

extern "C" const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "success";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_ALIGN: return "a pointer is not aligned (16 bytes for tensors, 4 for LSE and scales)";
    case FA_ERR_SHAPE: return "B, H or N out of range, or the sizes overflow";
    case FA_ERR_UNSUPPORTED: return "unsupported head dim, dtype or flag value";
    case FA_ERR_LAUNCH: return "kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a pipeline wait (device status word set)";
    case FA_ERR_ARCH: return "the current CUDA device is not an sm_103 GPU";
    case FA_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case FA_ERR_WORKSPACE: return "the workspace is missing or smaller than fa_decode_workspace_size reports";
    default: return "unknown status";
  }
}

extern "C" int fa_version(void) { return 100; }

#ifndef FA_BUILD_ID
#define FA_BUILD_ID "unknown"
#endif
// The tag lets the build script read the id from the file without loading it.
static const char kBuildIdTagged[] = "fa-build-id:" FA_BUILD_ID;

extern "C" const char* fa_build_id(void) { return kBuildIdTagged + 12; }
