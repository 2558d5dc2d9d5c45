// Element conversions of the KV store, shared by the KV write kernel and the
// decode partial kernel's append path, so that both store the same bytes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace tfpa {

// Eight float32 values -> eight e4m3 codes: value / scale rounded to float32
// (IEEE division), then e4m3 RNE, saturating.
__device__ __forceinline__ uint2 quant8(const float (&x)[8], float s) {
  uint32_t out[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = make_float2(__fdiv_rn(x[2 * i], s), __fdiv_rn(x[2 * i + 1], s));
    const __nv_fp8x2_storage_t b = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
    if (i & 1)
      out[i >> 1] |= (uint32_t)b << 16;
    else
      out[i >> 1] = (uint32_t)b;
  }
  return make_uint2(out[0], out[1]);
}

// Eight bf16 (one 16-byte load) -> eight float32.
__device__ __forceinline__ void unpack8(const uint4& in, float (&x)[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

}  // namespace tfpa
