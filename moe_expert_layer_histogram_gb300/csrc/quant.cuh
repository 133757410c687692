// quant.cuh -- device-side block quantisation and the scale-tile layout.
//
// NVFP4 (16-element blocks, e4m3 scale, activation global scale 1) and
// MXFP8 (32-element blocks, e8m0 scale) quantisation of fp32 values, as the
// layer applies it to its GEMM inputs: dynamic per-block scales computed in
// the kernel, with the activation global scale fixed at 1 (PR #40082 report,
// sec. 关键源码片段); block sizes 16 / 32 from the MegaMoE kernel-drop
// workflow page, sec. 三 (nvfp4_quantize_per_block_16 /
// mxfp8_quantize_per_block_32).
//   NVFP4: sf = e4m3_rn_satfinite(amax / 6); q_i = e2m1_rn_satfinite(x_i / sf)
//          with both divisions correctly rounded; sf == 0 gives zero codes.
//   MXFP8: X = floor(log2 amax) - 8 clamped to [-127, 127], scale byte X+127,
//          q_i = e4m3_rn_satfinite(x_i * 2^-X); amax == 0 gives scale 127 and
//          zero codes (OCP MX v1.0 conversion rule).
#pragma once

#include <cstdint>
#include <cuda_fp8.h>
#include <cuda_fp16.h>

namespace moe {

// ---------------------------------------------------------------- layout
// Block scales for the tensor cores are stored in tiles of 128 rows x 4
// consecutive scale bytes (512 bytes).  Inside a tile, row r of the tile sits
// at byte (r % 32) * 16 + (r / 32) * 4 + j for its j-th scale, so one 16-byte
// line holds rows r, r+32, r+64, r+96.  Tiles of one 128-row block are
// consecutive along the reduction dimension; `tiles_k` tiles per block.
__host__ __device__ __forceinline__ int64_t sf_tile_offset(int64_t row, int kg, int tiles_k) {
  return ((row >> 7) * tiles_k + (kg >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 +
         (kg & 3);
}

// ---------------------------------------------------------------- codecs
__device__ __forceinline__ float e4m3_to_float(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(__half(h));
}

__device__ __forceinline__ uint8_t float_to_e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// Eight fp32 values -> eight e2m1 codes, round to nearest even, saturating;
// q[2j] becomes the low nibble and q[2j+1] the high nibble of byte j (the
// conversion puts its first source operand in the high nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* q) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return out;
}

// ---------------------------------------------------------------- blocks
// x / s correctly rounded, for a positive e4m3 scale value s, r = RN(1 / s)
// and |x / s| small enough not to overflow, without a divide: q = x * r,
// then one Newton step on the residual, q + (x - q s) r, both steps fused.
// The residual is exact, and the step gives the correctly rounded quotient
// for every x with |x| >= 2^-99 (checked for all fp32 significands against
// the eight e4m3 significands; exponents only scale the steps above that).
// Below it the quotient is under 2^-90, nowhere near an e2m1 step, and only
// its sign matters, which is taken from x (the step alone turns -0 into +0).
__device__ __forceinline__ float div_e4m3_scale(float x, float s, float r) {
  const float q = __fmul_rn(x, r);
  const float rho = __fmaf_rn(-q, s, x);
  return copysignf(__fmaf_rn(rho, r, q), x);
}

// x[16] -> codes[2] (8 bytes, element 2j in the low nibble) and one e4m3
// scale byte.  Every element is divided by the quantised scale as above; a
// block whose maximum is infinite (inf * r would leave a NaN residual) takes
// correctly rounded divides instead.
__device__ __forceinline__ void quant_nvfp4_16(const float* x, uint32_t (&codes)[2],
                                               uint8_t& sf) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint8_t c = amax == 0.0f ? uint8_t{0} : float_to_e4m3(__fdiv_rn(amax, 6.0f));
  const float sv = e4m3_to_float(c);
  sf = c;
  if (sv == 0.0f) {
    codes[0] = codes[1] = 0u;
    return;
  }
  float q[16];
  if (amax != __int_as_float(0x7F800000)) {
    const float r = __frcp_rn(sv);
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = div_e4m3_scale(x[i], sv, r);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(x[i], sv);
  }
  codes[0] = cvt_e2m1x8(q);
  codes[1] = cvt_e2m1x8(q + 8);
}

// 2^e as an fp32 for e in [-127, 127] (exact; 2^-127 is subnormal).
__device__ __forceinline__ float exact_pow2(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                   : __uint_as_float(0x00400000u);
}

// x[32] -> codes[8] (32 bytes, byte i = element i) and one e8m0 scale byte.
__device__ __forceinline__ void quant_mxfp8_32(const float* x, uint32_t (&codes)[8],
                                               uint8_t& sf) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  if (amax == 0.0f) {
    sf = 127;
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = 0u;
    return;
  }
  const uint32_t bits = __float_as_uint(amax);
  const int ex = static_cast<int>((bits >> 23) & 0xFFu);
  const int fl = ex ? ex - 127 : (31 - __clz(static_cast<int>(bits & 0x7FFFFFu))) - 149;
  const int X = max(-127, min(127, fl - 8));
  sf = static_cast<uint8_t>(X + 127);
  const float scale = exact_pow2(-X);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t v = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b)
      v |= static_cast<uint32_t>(float_to_e4m3(x[4 * w + b] * scale)) << (8 * b);
    codes[w] = v;
  }
}

}  // namespace moe
