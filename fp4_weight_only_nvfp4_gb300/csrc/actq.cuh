// W4A4 activation quantiser, fp32 arithmetic.  The W4A4 arm of an FP4 linear layer quantises
// its activations to the weights' block format: NVFP4 with the checkpoint's per-tensor
// activation global alpha ("input_scale"), MXFP4 with E8M0 group scales and no global --
// "re-verify 27B NVFP4 on the nvidia ModelOpt checkpoint" (PR #178), section "W4A16 is the
// default for ModelOpt"; "native MXFP4 keep-quant + Qwen e2e" (PR #38), commit "W0".
// Every rounding decision is taken in fp32 (IEEE, round to nearest even):
//   NVFP4: s = E4M3_sat(fl32(amax / fl32(6 alpha))), d = fl32(s alpha),
//          code = E2M1_sat(fl32(x / d)) (all codes 0 when s = 0)
//   MXFP4: e = min{e : 6 2^e >= amax} in [-127, 127], code = E2M1_sat(fl32(x 2^-e))
// A magnitude that rounds to zero is code 0 (+0).  The kernels are built without fast-math
// (IEEE division, denormals kept), which these decisions rely on.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"  // act_maxmag8: a granule's largest magnitude (>= 0x7F80: inf or NaN)

namespace vt {

// Nearest point of the E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even code,
// saturating at 6; the comparisons are against the exact midpoints.
__device__ __forceinline__ uint32_t aq_e2m1(float q) {
  const float a = fabsf(q);
  uint32_t m;
  if (a <= 0.25f) m = 0;
  else if (a < 0.75f) m = 1;
  else if (a <= 1.25f) m = 2;
  else if (a < 1.75f) m = 3;
  else if (a <= 2.5f) m = 4;
  else if (a < 3.5f) m = 5;
  else if (a <= 5.0f) m = 6;
  else m = 7;
  return m == 0 ? 0u : ((q < 0.0f ? 8u : 0u) | m);
}

__device__ __forceinline__ float aq_e2m1_val(uint32_t c) {
  const uint32_t m = c & 7;
  // m = 0..3: 0, .5, 1, 1.5;  m = 4..7: 2, 3, 4, 6
  const float v = m < 4 ? 0.5f * (float)m : (float)(2u << ((m - 4) >> 1)) * (m & 1 ? 1.5f : 1.0f);
  return (c & 8) ? -v : v;
}

// Nearest non-negative finite E4M3 byte (bias 7, 3 mantissa bits, subnormal step 2^-9),
// ties to the even byte, saturating at 448 (0x7E).
__device__ __forceinline__ uint32_t aq_e4m3(float x) {
  if (!(x < 448.0f)) return 0x7E;
  if (x < 0.015625f) {  // below 2^-6: subnormal grid
    const float r = rintf(x * 512.0f);
    return r >= 8.0f ? 0x08u : (uint32_t)r;
  }
  int ex;
  const float f = frexpf(x, &ex);  // x = f 2^ex, f in [0.5, 1)
  int e = ex - 1;
  float mant = rintf((2.0f * f - 1.0f) * 8.0f);
  if (mant >= 8.0f) {
    mant = 0.0f;
    e += 1;
  }
  return (uint32_t)(((e + 7) << 3) | (int)mant);
}

__device__ __forceinline__ float aq_e4m3_val(uint32_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  return e == 0 ? ldexpf((float)m, -9) : ldexpf(1.0f + 0.125f * (float)m, e - 7);
}

// Smallest e with 6 2^e >= a (a >= 0 finite), clamped to [-127, 127]; with a = f 2^x,
// f in [0.5, 1): x - 3 when f <= 0.75, else x - 2.
__device__ __forceinline__ int aq_mx_exp(float a) {
  if (a == 0.0f) return -127;
  int x;
  const float f = frexpf(a, &x);
  const int e = (f <= 0.75f) ? x - 3 : x - 2;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
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

__device__ __forceinline__ uint32_t aq_nv_code(float x, const AqNvGroup& g) {
  return g.step == 0.0f ? 0u : aq_e2m1(__fdiv_rn(x, g.d));
}

// MXFP4 code with inv = 2^-e (exact in fp32 for e in [-127, 127]).
__device__ __forceinline__ uint32_t aq_mx_code(float x, float inv) {
  return aq_e2m1(__fmul_rn(x, inv));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// One 16-byte granule (8 activations, w[4]) of an NVFP4 group -> its 8 dequantised values
// c * s as f16 (exact: at most 6 significant bits, 2^-10 <= |c s| <= 2688), or NaN when the
// group holds an inf or NaN (bad); codes (optional) receives the 8 nibbles, low nibble first.
__device__ __forceinline__ uint4 aq_nv_granule(const uint32_t w[4], const AqNvGroup& g, bool bad,
                                               uint32_t* codes) {
  uint32_t o[4], cw = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t c0 = aq_nv_code(bf16_lo(w[q]), g), c1 = aq_nv_code(bf16_hi(w[q]), g);
    cw |= (c0 | (c1 << 4)) << (8 * q);
    o[q] = bad ? 0x7E007E00u : pack_half2(aq_e2m1_val(c0) * g.step, aq_e2m1_val(c1) * g.step);
  }
  if (codes) *codes = bad ? 0u : cw;
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One granule of an MXFP4 group with exponent e -> c * 2^(e - p) as f16 (p: the power of two
// the consumer multiplies back; exact while e - p >= -23, and below 2^15 while e - p <= 12).
__device__ __forceinline__ uint4 aq_mx_granule(const uint32_t w[4], int e, int p, bool bad,
                                               uint32_t* codes) {
  const float inv = ldexpf(1.0f, -e), up = ldexpf(1.0f, e - p);
  uint32_t o[4], cw = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t c0 = aq_mx_code(bf16_lo(w[q]), inv), c1 = aq_mx_code(bf16_hi(w[q]), inv);
    cw |= (c0 | (c1 << 4)) << (8 * q);
    o[q] = bad ? 0x7E007E00u : pack_half2(aq_e2m1_val(c0) * up, aq_e2m1_val(c1) * up);
  }
  if (codes) *codes = bad ? 0u : cw;
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One granule of an MXFP4 group with exponent e -> c * 2^e as bf16: exact (at most two
// significant bits, |c 2^e| >= 2^-128 for e >= -127; bf16 has fp32's exponent range, so a
// value beyond it is inf in both).  For the tiles of a wide MXFP4 weight (bf16 x bf16).
__device__ __forceinline__ uint4 aq_mx_granule_bf16(const uint32_t w[4], int e, bool bad) {
  const float inv = ldexpf(1.0f, -e), up = ldexpf(1.0f, e);
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t c0 = aq_mx_code(bf16_lo(w[q]), inv), c1 = aq_mx_code(bf16_hi(w[q]), inv);
    const __nv_bfloat162 h = __floats2bfloat162_rn(aq_e2m1_val(c0) * up, aq_e2m1_val(c1) * up);
    o[q] = bad ? 0x7FC07FC0u : *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace vt
