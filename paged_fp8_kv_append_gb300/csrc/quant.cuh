// quant.cuh -- bf16 -> e4m3 quantisation with a per-block scale.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": the cache is held as FP8 e4m3.  The pages give no
// scale or rounding rule; this library's reading: scale = amax / 448 in IEEE
// fp32 (1 when that is 0), code = e4m3 round-to-nearest-even with
// saturation of the fp32 quotient x / scale.  Shared by the append kernels
// and by the exhaustive division check in the GPU tests.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace kvfp8 {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) {
  return __uint_as_float((b & 0xFFFFu) << 16);
}

// Scale of a fresh block: amax / 448 in fp32; 1 when that is 0.
__device__ __forceinline__ float scale_from_amax(float amax) {
  const float s = __fdiv_rn(amax, 448.0f);
  return s > 0.0f ? s : 1.0f;
}

// the two bf16 values of a 32-bit word as fp32 (element 0 = low half)
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float amax2(uint32_t w) {
  return fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w)));
}

__device__ __forceinline__ float amax8(uint4 v) {
  return fmaxf(fmaxf(amax2(v.x), amax2(v.y)), fmaxf(amax2(v.z), amax2(v.w)));
}

__device__ __forceinline__ uint32_t e4m3x2(float q0, float q1) {
  return static_cast<uint32_t>(
             __nv_cvt_float2_to_fp8x2(make_float2(q0, q1), __NV_SATFINITE, __NV_E4M3)) &
         0xFFFFu;
}

// e4m3 codes of x / scale for two values (x0 -> low byte): IEEE fp32
// division, then the hardware round-to-nearest-even saturating conversion.
__device__ __forceinline__ uint32_t quant2(float x0, float x1, float scale) {
  return e4m3x2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale));
}

// 8 bf16 values -> 8 e4m3 codes (byte k = element k)
__device__ __forceinline__ uint2 quant8(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    c[k] = quant2(bf16_bits_to_f32(w[k]), bf16_bits_to_f32(w[k] >> 16), s);
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// x / s in fp32 round-to-nearest, for s > 0 and rs = __frcp_rn(s): the
// product with the correctly rounded reciprocal, corrected once with the
// remainder x - q0 * s (P. Markstein, "IA-64 and Elementary Functions", 2000:
// Newton-Raphson division on fused multiply-adds).  Used for blocks whose
// scale is at least 2^-90 (the caller decides once per block; smaller scales
// take the IEEE divide): there the remainder is exact whenever the quotient
// can reach an e4m3 code other than zero (an input below 2^-100 gives a
// quotient below 2^-10, which encodes as a signed zero whatever its low
// bits).  Branch-free: a quotient of magnitude >= 1024 (or an infinite / NaN
// input) stays uncorrected, since the e4m3 conversion saturates it the same
// way, and the result takes x's sign so that -0 stays -0.  Checked against
// __fdiv_rn on every bf16 x and every scale amax/448 of a bf16 amax (the
// inputs this library divides), comparing the e4m3 codes.
__device__ __forceinline__ bool scale_fast_ok(float s) { return s >= 0x1p-90f; }

__device__ __forceinline__ float div_fast(float x, float s, float rs) {
  const float q0 = x * rs;
  const float q1 = __fmaf_rn(__fmaf_rn(-q0, s, x), rs, q0);
  return copysignf(fabsf(q0) < 1024.0f ? q1 : q0, x);
}

// x / s where |x| <= amax and s = scale_from_amax(amax) >= 2^-90: the rows of
// a block whose scale they set.  There |x * rs| <= 448 (1 + 2^-22) < 1024, so
// div_fast's guard always takes the corrected quotient and can be left out.
__device__ __forceinline__ float div_fresh(float x, float s, float rs) {
  const float q0 = x * rs;
  return copysignf(__fmaf_rn(__fmaf_rn(-q0, s, x), rs, q0), x);
}

// e4m3 codes of the two bf16 values of w, under div_fresh's conditions
__device__ __forceinline__ uint32_t quant_word_fresh(uint32_t w, float s, float rs) {
  return e4m3x2(div_fresh(bf16_lo(w), s, rs), div_fresh(bf16_hi(w), s, rs));
}

// Largest magnitude among bf16 values, on their bit patterns: with the sign
// bits cleared, finite and infinite magnitudes order like unsigned integers
// (NaN patterns order above infinity: a result above 0x7F80 means a NaN was
// present, which the caller handles with the float maximum, which skips it).
__device__ __forceinline__ uint32_t absbits_max2(uint32_t m, uint32_t w) {
  return __vmaxu2(m, w & 0x7FFF7FFFu);
}
__device__ __forceinline__ uint32_t absbits_max8(uint32_t m, uint4 v) {
  return absbits_max2(absbits_max2(m, v.x), absbits_max2(v.y & 0x7FFF7FFFu,
                      __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
}
// the two halves of a packed maximum, reduced over the warp
__device__ __forceinline__ uint32_t absbits_warp_max(uint32_t m) {
  return __reduce_max_sync(0xffffffffu, max(m & 0xFFFFu, m >> 16));
}

// the division as the append kernels perform it, element by element
__device__ __forceinline__ float div_by_scale(float x, float s, float rs) {
  return scale_fast_ok(s) ? div_fast(x, s, rs) : __fdiv_rn(x, s);
}

// e4m3 codes of the two bf16 values of w, for a scale with scale_fast_ok
__device__ __forceinline__ uint32_t quant_word(uint32_t w, float s, float rs) {
  return e4m3x2(div_fast(bf16_lo(w), s, rs), div_fast(bf16_hi(w), s, rs));
}

// 8 bf16 values -> 8 e4m3 codes with the faster division
__device__ __forceinline__ uint2 quant8_rs(uint4 v, float s, float rs) {
  if (!scale_fast_ok(s)) return quant8(v, s);
  return make_uint2(quant_word(v.x, s, rs) | (quant_word(v.y, s, rs) << 16),
                    quant_word(v.z, s, rs) | (quant_word(v.w, s, rs) << 16));
}

}  // namespace kvfp8
