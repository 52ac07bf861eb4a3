// Quantiser for synthetic or user bf16 weights -> NVFP4 / MXFP4 codes and scales.
// Recipe (the synthetic-weight generation the workloads use): NVFP4 global
// G = fl32(amax / (6*448)), group scale s = E4M3_RNE_sat(amax_g / (6 G)),
// code = E2M1_RNE_sat(w / (s G)); MXFP4 group exponent e = min{e : 2^e >= amax_g/6},
// code = E2M1_RNE_sat(w / 2^e).  Quotients in fp64 (IEEE division), ties to even.
// Format definitions: "keep the ModelOpt NVFP4 lm_head packed" (vllm.cpp PR #263), "Why
// this row matters" (U8 codes + FP8 scale per 16 + FP32 second scale) and "native MXFP4
// keep-quant + Qwen e2e" (PR #38), commit "W2" (E8M0 scale per 32, no global).
#include <cuda_bf16.h>

#include "actq.cuh"
#include "common.cuh"
#include "kernels.h"

namespace vt {

// Round-to-nearest-even onto the E2M1 grid {0,.5,1,1.5,2,3,4,6}, saturating at 6; the
// comparisons encode the exact midpoints, with ties resolved towards the even code.
__device__ __forceinline__ uint32_t e2m1_rne(double q) {
  const double a = fabs(q);
  uint32_t m;
  if (a <= 0.25) m = 0;
  else if (a < 0.75) m = 1;
  else if (a <= 1.25) m = 2;
  else if (a < 1.75) m = 3;
  else if (a <= 2.5) m = 4;
  else if (a < 3.5) m = 5;
  else if (a <= 5.0) m = 6;
  else m = 7;
  if (m == 0) return 0;  // a magnitude rounding to zero is +0
  return (q < 0.0 ? 8u : 0u) | m;
}

// Round-to-nearest-even onto non-negative finite E4M3 (bias 7, 3 mantissa bits,
// subnormal step 2^-9), saturating at 448.
__device__ __forceinline__ uint32_t e4m3_rne(double x) {
  if (!(x < 448.0)) return 0x7E;
  if (x < 0.015625) {  // below 2^-6: subnormal grid of step 2^-9
    const double r = rint(x * 512.0);
    return r >= 8.0 ? 0x08u : (uint32_t)r;
  }
  int ex;
  const double f = frexp(x, &ex);  // x = f * 2^ex, f in [0.5, 1)
  int e = ex - 1;                   // x = (2f) * 2^e, 2f in [1, 2)
  double mant = rint((2.0 * f - 1.0) * 8.0);
  if (mant >= 8.0) {
    mant = 0.0;
    e += 1;
  }
  return (uint32_t)(((e + 7) << 3) | (int)mant);
}

__device__ __forceinline__ double e4m3_val(uint32_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  return e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
}

// Smallest e with 6 * 2^e >= a (a > 0): with a = f 2^x, f in [0.5, 1), that is x-3 when
// f <= 0.75 and x-2 otherwise.
__device__ __forceinline__ int mx_exp(double a) {
  if (a == 0.0) return -127;
  int x;
  const double f = frexp(a, &x);
  int e = (f <= 0.75) ? x - 3 : x - 2;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

__global__ void k_q_init(uint32_t* scratch) {
  scratch[0] = 0u;
  scratch[1] = 0u;
}

__global__ void k_q_amax(const uint16_t* __restrict__ W, int64_t total, uint32_t* scratch) {
  uint32_t m = 0;
  const int64_t nv = total / 8;
  const uint4* w4 = reinterpret_cast<const uint4*>(W);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nv;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = w4[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = max(m, w[j] & 0x7FFFu);
      m = max(m, (w[j] >> 16) & 0x7FFFu);
    }
  }
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(&scratch[0], m);
}

__global__ void k_q_global(uint32_t* scratch, float* global_out) {
  const uint32_t bits = scratch[0] << 16;
  const double amax = (double)__uint_as_float(bits);
  const float G = amax > 0.0 ? (float)(amax / (6.0 * 448.0)) : 1.0f;
  scratch[1] = __float_as_uint(G);
  *global_out = G;
}

__device__ __forceinline__ double bf16_bits_val(uint32_t h) {
  return (double)__uint_as_float((h & 0xFFFFu) << 16);
}

// One thread per group.  NVFP4: 16 values -> 8 code bytes + 1 scale byte.
__global__ void k_q_nv(const uint16_t* __restrict__ W, int64_t N, int64_t K,
                       const uint32_t* scratch, uint8_t* __restrict__ codes,
                       uint8_t* __restrict__ scales) {
  const int64_t gpr = K / 16, total = N * gpr;
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t n = i / gpr, grp = i % gpr;
  const uint4* src = reinterpret_cast<const uint4*>(W + n * K + grp * 16);
  const uint4 v0 = src[0], v1 = src[1];
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  double vals[16];
  double amax = 0.0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    vals[2 * j] = bf16_bits_val(w[j]);
    vals[2 * j + 1] = bf16_bits_val(w[j] >> 16);
    amax = fmax(amax, fmax(fabs(vals[2 * j]), fabs(vals[2 * j + 1])));
  }
  const double G = (double)__uint_as_float(scratch[1]);
  const uint32_t sb = e4m3_rne(amax / (6.0 * G));
  const double denom = e4m3_val(sb) * G;
  uint32_t packed[2] = {0, 0};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t c = denom == 0.0 ? 0u : e2m1_rne(vals[j] / denom);
    packed[j >> 3] |= c << (4 * (j & 7));
  }
  *reinterpret_cast<uint2*>(codes + n * (K / 2) + grp * 8) = make_uint2(packed[0], packed[1]);
  scales[i] = (uint8_t)sb;
}

// MXFP4: 32 values -> 16 code bytes + 1 E8M0 byte.
__global__ void k_q_mx(const uint16_t* __restrict__ W, int64_t N, int64_t K,
                       uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int64_t gpr = K / 32, total = N * gpr;
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t n = i / gpr, grp = i % gpr;
  const uint4* src = reinterpret_cast<const uint4*>(W + n * K + grp * 32);
  double vals[32];
  double amax = 0.0;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 x = src[v];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      vals[8 * v + 2 * j] = bf16_bits_val(w[j]);
      vals[8 * v + 2 * j + 1] = bf16_bits_val(w[j] >> 16);
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmax(amax, fabs(vals[j]));
  const int e = mx_exp(amax);
  uint32_t packed[4] = {0, 0, 0, 0};
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t c = e2m1_rne(ldexp(vals[j], -e));
    packed[j >> 3] |= c << (4 * (j & 7));
  }
  *reinterpret_cast<uint4*>(codes + n * (K / 2) + grp * 16) =
      make_uint4(packed[0], packed[1], packed[2], packed[3]);
  scales[i] = (uint8_t)(e + 127);
}

// W4A4 activation quantiser (fp32 decisions, actq.cuh): one thread per group.  A group
// holding an inf or NaN gets the format's NaN scale byte (E4M3 0x7F, E8M0 0xFF) and zero codes.
template <int FMT>
__global__ void k_qa(const uint16_t* __restrict__ A, int64_t M, int64_t lda, int64_t K,
                     float alpha, float alpha6, uint8_t* __restrict__ codes,
                     uint8_t* __restrict__ scales) {
  constexpr int G = FMT == FMT_NV ? 16 : 32, NG = G / 8;
  const int64_t gpr = K / G, total = M * gpr;
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t m = i / gpr, grp = i % gpr;
  const uint4* src = reinterpret_cast<const uint4*>(A + m * lda + grp * G);
  uint32_t w[NG][4];
  int mx = 0;
#pragma unroll
  for (int v = 0; v < NG; ++v) {
    const uint4 x = src[v];
    w[v][0] = x.x;
    w[v][1] = x.y;
    w[v][2] = x.z;
    w[v][3] = x.w;
    mx = max(mx, act_maxmag8(w[v]));
  }
  const bool bad = mx >= 0x7F80;
  const float amax = __uint_as_float((uint32_t)(bad ? 0 : mx) << 16);
  uint32_t cw[NG];
  uint32_t sbyte;
  if constexpr (FMT == FMT_NV) {
    const AqNvGroup g = aq_nv_group(amax, alpha, alpha6);
#pragma unroll
    for (int v = 0; v < NG; ++v) aq_nv_granule(w[v], g, bad, &cw[v]);
    sbyte = bad ? 0x7Fu : g.sbyte;
  } else {
    const int e = aq_mx_exp(amax);
#pragma unroll
    for (int v = 0; v < NG; ++v) aq_mx_granule(w[v], e, e, bad, &cw[v]);
    sbyte = bad ? 0xFFu : (uint32_t)(e + 127);
  }
  uint8_t* dst = codes + m * (K / 2) + grp * (G / 2);
  if constexpr (FMT == FMT_NV) *reinterpret_cast<uint2*>(dst) = make_uint2(cw[0], cw[1]);
  else *reinterpret_cast<uint4*>(dst) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  scales[i] = (uint8_t)sbyte;
}

cudaError_t launch_quantize_act(const void* A, int64_t M, int64_t lda, int64_t K, int fmt,
                                float alpha, uint8_t* codes, uint8_t* scales, cudaStream_t s) {
  const uint16_t* a = reinterpret_cast<const uint16_t*>(A);
  const int64_t groups = M * (K / (fmt == FMT_NV ? 16 : 32));
  const unsigned blocks = (unsigned)((groups + 255) / 256);
  if (fmt == FMT_NV) k_qa<FMT_NV><<<blocks, 256, 0, s>>>(a, M, lda, K, alpha, 6.0f * alpha, codes, scales);
  else k_qa<FMT_MX><<<blocks, 256, 0, s>>>(a, M, lda, K, alpha, 6.0f * alpha, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void* W, int64_t N, int64_t K, int fmt, uint8_t* codes,
                            uint8_t* scales, float* global_out, void* scratch, cudaStream_t s) {
  const uint16_t* w = reinterpret_cast<const uint16_t*>(W);
  uint32_t* sc = reinterpret_cast<uint32_t*>(scratch);
  if (fmt == FMT_NV) {
    k_q_init<<<1, 1, 0, s>>>(sc);
    const int64_t total = N * K;
    const int64_t nb = (total / 8 + 255) / 256;
    const int blocks = (int)(nb < 8192 ? nb : 8192);
    k_q_amax<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(w, total, sc);
    k_q_global<<<1, 1, 0, s>>>(sc, global_out);
    const int64_t groups = N * (K / 16);
    k_q_nv<<<(unsigned)((groups + 255) / 256), 256, 0, s>>>(w, N, K, sc, codes, scales);
  } else {
    const int64_t groups = N * (K / 32);
    k_q_mx<<<(unsigned)((groups + 255) / 256), 256, 0, s>>>(w, N, K, codes, scales);
  }
  return cudaGetLastError();
}

}  // namespace vt
