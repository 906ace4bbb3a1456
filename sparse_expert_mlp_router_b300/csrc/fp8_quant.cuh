// Per-row E4M3 quantisation of bf16 rows, one warp per row: scale = max|row| / 448 and
// code = E4M3(value / scale), both divisions rounded once in float32, round to nearest even,
// saturated to +-448 (an all-zero row: scale 0, codes 0). Used for the FP8 expert weights and,
// in the W8A8 layer, for the activation rows that enter each expert contraction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.cuh"

namespace moe {

// 16 bytes of a row: through the read-only cache path when the row was written before the
// launch, or from L2 (__ldcg) when other SMs of the same launch may have just written it (the
// read-only path is not kept coherent with such writes).
template <bool FROM_L2>
__device__ __forceinline__ uint4 load_row16(const __nv_bfloat16* p) {
  if (FROM_L2) return __ldcg(reinterpret_cast<const uint4*>(p));
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Row `src` of `cols` bf16 values (cols a multiple of 16, rows 16-byte aligned) -> `dst`
// codes and *scale_out (written by lane 0). All 32 lanes of the warp call it together.
// FROM_L2: the row may have been written by other SMs during the same launch.
template <bool FROM_L2 = false>
__device__ __forceinline__ void quantize_row_e4m3_warp(const __nv_bfloat16* src, int cols, uint8_t* __restrict__ dst,
                                                       float* scale_out, int lane) {
  float mx = 0.0f;
  for (int c = lane * 8; c < cols; c += 256) {
    const uint4 u = load_row16<FROM_L2>(src + c);
    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mx = fmaxf(mx, fabsf(__uint_as_float(wd[i] << 16)));
      mx = fmaxf(mx, fabsf(__uint_as_float(wd[i] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float s = __fdiv_rn(mx, 448.0f);
  if (lane == 0) *scale_out = s;
  for (int c = lane * 16; c < cols; c += 512) {
    const uint4 a = load_row16<FROM_L2>(src + c);
    const uint4 b = load_row16<FROM_L2>(src + c + 8);
    const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t word = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t pair = wd[2 * i + h];
        float2 v = make_float2(__uint_as_float(pair << 16), __uint_as_float(pair & 0xFFFF0000u));
        if (s > 0.0f) {
          v.x = __fdiv_rn(v.x, s);
          v.y = __fdiv_rn(v.y, s);
        } else {
          v = make_float2(0.0f, 0.0f);
        }
        const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
        word |= (uint32_t)q << (16 * h);
      }
      out[i] = word;
    }
    *reinterpret_cast<uint4*>(dst + c) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

}  // namespace moe
