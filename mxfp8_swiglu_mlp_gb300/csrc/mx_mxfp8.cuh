// mx_mxfp8.cuh -- device helpers of the MXFP8 encoding shared by the kernels.
//
// Quantisation rule (OCP MX, as the Fish Audio post's mxfp8 format uses it,
// p2 "Estrategia de cuantizacion FP8"): for each 32-block, the UE8M0 byte is
// max(biased_exponent(amax) - 8, 0), i.e. e = floor(log2 amax) - 8 clamped at
// -127; elements are v * 2^-e converted to E4M3 with round-to-nearest-even
// and saturation (cvt ... satfinite).
#pragma once
#include <cuda_fp8.h>
#include <cstdint>

namespace fsops {
namespace dev {

__device__ __forceinline__ uint32_t ue8m0_from_amax(float amax) {
  const int be = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  return static_cast<uint32_t>(be > 8 ? be - 8 : 0);
}
// 2^-e for scale byte s = e + 127 (s <= 246 for finite fp32 inputs).
__device__ __forceinline__ float inv_scale_from_ue8m0(uint32_t s) {
  return __uint_as_float((254u - s) << 23);
}
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
// Two values to two E4M3 codes in one conversion instruction (round to
// nearest even, saturating): lo in bits 0..7, hi in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2_code(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Four values to four codes, a in bits 0..7 up to d in bits 24..31.
__device__ __forceinline__ uint32_t e4m3x4_code(float a, float b, float c, float d) {
  return e4m3x2_code(a, b) | (e4m3x2_code(c, d) << 16);
}
// Byte offset of the scale of row r, 32-block kb in the tcgen05 tiled layout
// (512-byte tiles of 128 rows x 4 blocks; n_kg = K / 128 tiles per row tile).
__device__ __forceinline__ uint32_t tiled_sf_offset(int r, int kb, int n_kg) {
  return static_cast<uint32_t>(((r >> 7) * n_kg + (kb >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 +
                               (kb & 3));
}
// SiLU(g) * u in fp32.  The fast divide (reciprocal approximation, 2 ulp)
// keeps this off the epilogue's critical path; its error is far below the
// E4M3 step the result is rounded to next.  For g below about -88, 1 + e^-g
// overflows to +inf and the quotient is 0, the limit of SiLU.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

}  // namespace dev
}  // namespace fsops
