// W4A4 activation quantiser, fp32 arithmetic.  The W4A4 arm of an FP4 linear layer quantises
// its activations to the weights' block format: NVFP4 with the checkpoint's per-tensor
// activation global alpha ("input_scale"), MXFP4 with E8M0 group scales and no global --
// "re-verify 27B NVFP4 on the nvidia ModelOpt checkpoint" (PR #178), section "W4A16 is the
// default for ModelOpt"; "native MXFP4 keep-quant + Qwen e2e" (PR #38), commit "W0".
// Every rounding decision is taken in fp32 (IEEE, round to nearest even):
//   NVFP4: s = E4M3_sat(fl32(amax / fl32(6 alpha))), d = fl32(s alpha),
//          code = E2M1_sat(fl32(x / d)) (all codes 0 when s = 0)
//   MXFP4: e = min{e : 6 2^e >= amax} in [-127, 127], code = E2M1_sat(fl32(x 2^-e))
// E2M1_sat is the nearest point of the E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even
// code, saturating at 6 (the hardware conversion cvt.rn.satfinite.e2m1x2.f32); a magnitude
// that rounds to zero is code 0 (+0).  The kernels are built without fast-math (IEEE
// division, denormals kept), which these decisions rely on.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"  // act_maxmag8: a granule's largest magnitude (>= 0x7F80: inf or NaN)

namespace vt {

// 2^k in fp32, exact, for k <= 127: a normal power from the exponent field, a subnormal one
// (k in [-149, -127]) as a single mantissa bit, 0 below 2^-149.
__device__ __forceinline__ float aq_pow2(int k) {
  if (k >= -126) return __uint_as_float((uint32_t)(k + 127) << 23);
  return k >= -149 ? __uint_as_float(1u << (k + 149)) : 0.0f;
}

// Nearest non-negative finite E4M3 byte (bias 7, 3 mantissa bits, subnormal step 2^-9),
// ties to the even byte, saturating at 448 (0x7E).
__device__ __forceinline__ uint32_t aq_e4m3(float x) {
  if (!(x < 448.0f)) return 0x7E;
  if (x < 0.015625f) {  // below 2^-6: subnormal grid
    const float r = rintf(x * 512.0f);
    return r >= 8.0f ? 0x08u : (uint32_t)r;
  }
  // normal: round the 23 fp32 mantissa bits to 3, ties to even (a carry moves into the
  // exponent field), then rebias the exponent from 127 to 7; below 448 the result is <= 0x7E
  const uint32_t u = __float_as_uint(x);
  return ((u + 0x7FFFFu + ((u >> 20) & 1u)) >> 20) - (120u << 3);
}

__device__ __forceinline__ float aq_e4m3_val(uint32_t b) {
  const uint32_t e = (b >> 3) & 15, m = b & 7;
  return e == 0 ? (float)m * 0.001953125f : __uint_as_float(((b & 0x7Fu) << 20) + (120u << 23));
}

// Smallest e with 6 2^e >= a (a >= 0 finite), clamped to [-127, 127].  For a normal
// a = 1.f 2^(E - 127) it is E - 129 when 1.f <= 1.5 (mantissa field <= 2^22), else E - 128;
// zero and subnormal a (E = 0) give -127 after the clamp, as does E = 1.
__device__ __forceinline__ int aq_mx_exp(float a) {
  const uint32_t u = __float_as_uint(a);
  const int e = (int)(u >> 23) - 129 + ((u & 0x7FFFFFu) > 0x400000u ? 1 : 0);
  return e < -127 ? -127 : e;
}

// The NVFP4 group decision from the group's largest magnitude.
struct AqNvGroup {
  uint32_t sbyte;  // E4M3 scale byte
  float step;      // its value
  float d;         // fl32(step * alpha): the code divisor
};

__device__ __forceinline__ AqNvGroup aq_nv_group(float amax, float alpha, float alpha6) {
  AqNvGroup g;
  g.sbyte = aq_e4m3(__fdiv_rn(amax, alpha6));
  g.step = aq_e4m3_val(g.sbyte);
  g.d = __fmul_rn(g.step, alpha);
  return g;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Eight floats -> eight E2M1 codes, x[2q] in the low nibble of byte q, by the hardware
// conversion (nearest, ties to even, saturating at 6); a magnitude that rounds to zero, which
// the conversion returns with its sign, becomes +0.
__device__ __forceinline__ uint32_t aq_e2m1x8(const float x[8]) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  const uint32_t mag = r & 0x77777777u;  // a nibble's bit 3 survives when its magnitude is > 0
  return mag | (r & ((mag + 0x77777777u) & 0x88888888u));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// One 16-byte granule (8 activations, w[4]) of an NVFP4 group -> its 8 dequantised values
// c * s as f16 (exact: at most 6 significant bits, 2^-10 <= |c s| <= 2688, and s itself is
// an f16), or NaN when the group holds an inf or NaN (bad); codes (optional) receives the 8
// nibbles, low nibble first.
__device__ __forceinline__ uint4 aq_nv_granule(const uint32_t w[4], const AqNvGroup& g, bool bad,
                                               uint32_t* codes) {
  float x[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    x[2 * q] = __fdiv_rn(bf16_lo(w[q]), g.d);
    x[2 * q + 1] = __fdiv_rn(bf16_hi(w[q]), g.d);
  }
  const uint32_t cw = g.step == 0.0f ? 0u : aq_e2m1x8(x);
  if (codes) *codes = bad ? 0u : cw;
  uint32_t h[4], o[4];
  e2m1x8_to_f16x8(cw, h[0], h[1], h[2], h[3]);
  const __half2 s2 = __float2half2_rn(g.step);
#pragma unroll
  for (int q = 0; q < 4; ++q) o[q] = bad ? 0x7E007E00u : h2_bits(__hmul2_rn(bits_h2(h[q]), s2));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One granule of an MXFP4 group with exponent e -> c * 2^(e - p) as f16, rounded once (p: the
// power of two the consumer multiplies back; e - p <= 12 keeps it below 2^15).  While
// 2^(e - p) is itself an f16 (e - p >= -24) the f16 product rounds the exact value; below
// that the product is taken in fp32, where it is exact down to 2^-149.
__device__ __forceinline__ uint4 aq_mx_granule(const uint32_t w[4], int e, int p, bool bad,
                                               uint32_t* codes) {
  const float inv = aq_pow2(-e);
  float x[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    x[2 * q] = __fmul_rn(bf16_lo(w[q]), inv);
    x[2 * q + 1] = __fmul_rn(bf16_hi(w[q]), inv);
  }
  const uint32_t cw = aq_e2m1x8(x);
  if (codes) *codes = bad ? 0u : cw;
  uint32_t h[4], o[4];
  e2m1x8_to_f16x8(cw, h[0], h[1], h[2], h[3]);
  if (e - p >= -24) {
    const __half2 up = __float2half2_rn(aq_pow2(e - p));
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = h2_bits(__hmul2_rn(bits_h2(h[q]), up));
  } else {
    const float up = aq_pow2(e - p);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __half22float2(bits_h2(h[q]));
      o[q] = pack_half2(f.x * up, f.y * up);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) o[q] = bad ? 0x7E007E00u : o[q];
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One granule of an MXFP4 group with exponent e -> c * 2^e as bf16: exact (at most two
// significant bits, |c 2^e| >= 2^-128 for e >= -127; bf16 has fp32's exponent range, so a
// value beyond it is inf in both).  For the tiles of a wide MXFP4 weight (bf16 x bf16).
__device__ __forceinline__ uint4 aq_mx_granule_bf16(const uint32_t w[4], int e, bool bad) {
  const float inv = aq_pow2(-e), up = aq_pow2(e);
  float x[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    x[2 * q] = __fmul_rn(bf16_lo(w[q]), inv);
    x[2 * q + 1] = __fmul_rn(bf16_hi(w[q]), inv);
  }
  uint32_t h[4], o[4];
  e2m1x8_to_f16x8(aq_e2m1x8(x), h[0], h[1], h[2], h[3]);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __half22float2(bits_h2(h[q]));
    const __nv_bfloat162 v = __floats2bfloat162_rn(f.x * up, f.y * up);
    o[q] = bad ? 0x7FC07FC0u : *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace vt
