// FP8 entry points (filled in by the E4M3 quantisation and forward kernels).
#include "../../include/fa.h"

extern "C" int fa_quantize_fp8(const void*, void*, float*, int, int, int, int, int, int, void*) {
  return FA_ERR_UNSUPPORTED;
}

extern "C" int fa_fwd_fp8(const void*, const void*, const void*, void*, float*, int, int, int, int,
                          float, int, const float*, const float*, const float*, int, void*) {
  return FA_ERR_UNSUPPORTED;
}
