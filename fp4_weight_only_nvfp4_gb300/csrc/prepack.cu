// Prepack (source layout -> tile layout), its inverse, and the dequantisation used by the
// bit-exact tests.  Source for the packed-resident design: "keep the ModelOpt NVFP4
// lm_head packed" (vllm.cpp PR #263), "Why this row matters" -- the weight is kept packed
// and its kernel-ready form is built once at load.
#include "common.cuh"
#include "kernels.h"

namespace vt {

// Source description of one or two stacked weights (fused gate_up uses two).
struct SrcPair {
  const uint8_t* codes[2];
  const uint8_t* scales[2];
  int64_t split;  // rows [0, split) come from source 0, the rest from source 1
  uint32_t layout;  // packed row order (kLayoutRows / kLayoutPaired)
};

__device__ __forceinline__ void src_row(const SrcPair& s, int64_t row, int& which,
                                        int64_t& r) {
  which = row < s.split ? 0 : 1;
  r = which ? row - s.split : row;
}

__global__ void k_header(PackedHeader* h, int fmt, int64_t N, int64_t K, int64_t split,
                         float f0, float f1, uint32_t layout) {
  if (threadIdx.x == 0) {
    h->magic = kMagic;
    h->layout = layout;
    h->fmt = static_cast<uint32_t>(fmt);
    h->N = N;
    h->K = K;
    h->seg_split = split;
    h->factor[0] = f0;
    h->factor[1] = f1;
    h->emax[0] = -1;
    h->emax[1] = -1;
    h->emin[0] = 256;
    h->emin[1] = 256;
    h->wide = 0;
  }
}

// MXFP4: largest and smallest finite E8M0 byte of each segment (over every group, whatever
// its codes, so that the packed form keeps every byte recoverable).
__global__ void k_mx_emax(SrcPair s, int64_t N, int64_t K, PackedHeader* h) {
  const int64_t gpr = K / 32;
  const int64_t total = N * gpr;
  int hi[2] = {-1, -1}, lo[2] = {256, 256};
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t row = i / gpr, grp = i % gpr;
    int which;
    int64_t r;
    src_row(s, row, which, r);
    int e = s.scales[which][r * gpr + grp];
    if (e != 0xFF) {
      hi[which] = max(hi[which], e);
      lo[which] = min(lo[which], e);
    }
  }
  for (int w = 0; w < 2; ++w) {
    int v = hi[w], u = lo[w];
    for (int o = 16; o > 0; o >>= 1) {
      v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
      u = min(u, __shfl_xor_sync(0xffffffffu, u, o));
    }
    if ((threadIdx.x & 31) == 0 && v >= 0) {
      atomicMax(&h->emax[w], v);
      atomicMin(&h->emin[w], u);
    }
  }
}

// MXFP4: choose the scale encoding once the exponent range is known.  When every segment's
// finite scale bytes lie within the 30 exponents [emax - 29, emax], the tiles hold them as
// f16 powers of two relative to emax (mx_encode) and the epilogue factor is 2^(emax - 140);
// otherwise (a wider range) the tiles keep the raw bytes, the kernels multiply each group by
// its exact scale 2^(e - 127) in fp32, and the factor is 1.
__global__ void k_mx_factor(PackedHeader* h) {
  if (threadIdx.x == 0) {
    bool wide = false;
    for (int w = 0; w < 2; ++w) {
      int e = h->emax[w];
      if (e < 0) e = 127;  // no finite scale: any offset works
      h->emax[w] = e;
      if (h->emin[w] <= 255 && h->emin[w] < e - 29) wide = true;
    }
    h->wide = wide ? 1u : 0u;
    for (int w = 0; w < 2; ++w) h->factor[w] = wide ? 1.0f : ldexpf(1.0f, h->emax[w] - 140);
  }
}

// E8M0 byte -> high byte of the f16 2^x, x = e - emax + 13, so that the largest scale of
// the segment maps to 2^13 (codes up to 6 stay below the f16 limit) and scales down to
// 2^-16 stay exact; 0xFF (NaN) maps to an f16 NaN.  Used only when every finite byte of the
// weight lies in that window (k_mx_factor), so no scale is lost.
__device__ __forceinline__ uint8_t mx_encode(int e, int emax) {
  if (e == 0xFF) return 0x7E;
  int x = e - emax + 13;
  if (x >= -14) return static_cast<uint8_t>((x + 15) << 2);
  if (x == -15) return 0x02;
  if (x == -16) return 0x01;
  return 0;
}

// One block per tile; 256 threads.  Thread i < 256 writes the 16 code bytes of
// (row block j = i/32, lane = i%32); the first 32 (NVFP4) / 16 (MXFP4) threads also
// write the scale bytes.
__global__ void __launch_bounds__(256) k_pack(SrcPair s, int fmt, int64_t N, int64_t K,
                                              int64_t KT, uint8_t* tiles,
                                              const PackedHeader* h) {
  const int64_t tile = blockIdx.x;
  const int64_t rt = tile / KT, kt = tile % KT;
  const int tb = tile_bytes(fmt);
  uint8_t* out = tiles + tile * tb;
  const int i = threadIdx.x;
  const int j = i >> 5, lane = i & 31, g = lane >> 2, t = lane & 3;
  const int64_t kb = K / 2;  // code bytes per row
  uint32_t words[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t row =
          packed_to_row(s.layout, rt * kTileRows + j * 16 + g + ((b & 1) ? 8 : 0), N, s.split);
      int64_t col = kt * 32 + 8 * t + 2 * q + (b >> 1);
      uint32_t v = 0;
      if (row >= 0 && col < kb) {
        int which;
        int64_t r;
        src_row(s, row, which, r);
        v = s.codes[which][r * kb + col];
      }
      w |= v << (8 * b);
    }
    words[q] = w;
  }
  *reinterpret_cast<uint4*>(out + j * 512 + lane * 16) =
      make_uint4(words[0], words[1], words[2], words[3]);

  // scale bytes: thread (j, lane) writes the pair (rows g, g+8) of row block j for NVFP4;
  // for MXFP4 the threads with t < 2 write the pair of (j, g, h = t)
  const bool nv = (fmt == FMT_NV);
  if (nv || t < 2) {
    const int64_t gpr = K / (nv ? 16 : 32);
    const int64_t grp = nv ? kt * 4 + t : kt * 2 + t;
    uint32_t pair = 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int64_t row = packed_to_row(s.layout, rt * kTileRows + j * 16 + g + half * 8, N, s.split);
      uint32_t v = 0;
      if (row >= 0 && grp < gpr) {
        int which;
        int64_t r;
        src_row(s, row, which, r);
        const uint8_t b = s.scales[which][r * gpr + grp];
        v = (nv || h->wide) ? b : mx_encode(b, h->emax[which]);
      }
      pair |= v << (8 * half);
    }
    const int off = nv ? scale_offset(FMT_NV, j, g, t) : scale_offset(FMT_MX, j, g, 2 * t);
    *reinterpret_cast<uint16_t*>(out + off) = static_cast<uint16_t>(pair);
  }
}

// Inverse of k_pack for the codes and scale bytes.  MXFP4 scale bytes of a narrow weight are
// recovered from the re-encoding and the segment's emax; a wide weight keeps them raw.
__device__ __forceinline__ int mx_decode(uint8_t enc, int emax) {
  if (enc == 0x7E) return 0xFF;
  int x;
  if (enc >= 0x04) x = (enc >> 2) - 15;
  else if (enc == 0x02) x = -15;
  else if (enc == 0x01) x = -16;
  else return -1;  // flushed: not recoverable
  return x + emax - 13;
}

__global__ void __launch_bounds__(256) k_unpack(const uint8_t* tiles, int fmt, int64_t N,
                                                int64_t K, int64_t KT, int64_t split,
                                                uint32_t layout, const PackedHeader* h,
                                                uint8_t* codes, uint8_t* scales) {
  const int64_t tile = blockIdx.x;
  const int64_t rt = tile / KT, kt = tile % KT;
  const uint8_t* in = tiles + tile * tile_bytes(fmt);
  const int i = threadIdx.x;
  const int j = i >> 5, lane = i & 31, g = lane >> 2, t = lane & 3;
  const int64_t kb = K / 2;
  uint4 v = *reinterpret_cast<const uint4*>(in + j * 512 + lane * 16);
  uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t row =
          packed_to_row(layout, rt * kTileRows + j * 16 + g + ((b & 1) ? 8 : 0), N, split);
      int64_t col = kt * 32 + 8 * t + 2 * q + (b >> 1);
      if (row >= 0 && col < kb) codes[row * kb + col] = (words[q] >> (8 * b)) & 0xFF;
    }
  const bool nv = (fmt == FMT_NV);
  if (nv || t < 2) {
    const int64_t gpr = K / (nv ? 16 : 32);
    const int64_t grp = nv ? kt * 4 + t : kt * 2 + t;
    const int off = nv ? scale_offset(FMT_NV, j, g, t) : scale_offset(FMT_MX, j, g, 2 * t);
    const uint32_t pair = *reinterpret_cast<const uint16_t*>(in + off);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int64_t row = packed_to_row(layout, rt * kTileRows + j * 16 + g + half * 8, N, split);
      if (row >= 0 && grp < gpr) {
        const uint8_t b = (pair >> (8 * half)) & 0xFF;
        if (nv || h->wide) {
          scales[row * gpr + grp] = b;
        } else {
          int e = mx_decode(b, h->emax[row < split ? 0 : 1]);
          scales[row * gpr + grp] = static_cast<uint8_t>(e < 0 ? 0 : e);
        }
      }
    }
  }
}

// Dequantise through the same conversions the GEMM uses: E2M1 pair -> f16x2, scale ->
// f16x2, one f16 multiply (exact), then fp32 multiply by the segment factor.  A wide MXFP4
// weight (raw E8M0 bytes in its tiles) gives c * 2^(e - 127) by one fp32 multiply of the
// code's value by the exact scale, as its GEMM does.
__global__ void __launch_bounds__(256) k_dequant(const uint8_t* tiles, int fmt, int64_t N,
                                                 int64_t K, int64_t KT, int64_t split,
                                                 uint32_t layout, const PackedHeader* h,
                                                 float* out) {
  const int64_t tile = blockIdx.x;
  const int64_t rt = tile / KT, kt = tile % KT;
  const uint8_t* in = tiles + tile * tile_bytes(fmt);
  const int i = threadIdx.x;
  const int j = i >> 5, lane = i & 31, g = lane >> 2, t = lane & 3;
  uint4 v = *reinterpret_cast<const uint4*>(in + j * 512 + lane * 16);
  uint32_t words[4] = {v.x, v.y, v.z, v.w};
  const uint32_t two = *reinterpret_cast<const uint16_t*>(in + scale_offset(fmt, j, g, t));
  const bool wide = fmt == FMT_MX && h->wide;
  const uint32_t sc2 = (fmt == FMT_NV) ? e4m3x2_to_f16x2(two) : mxenc2_to_f16x2(two);
  const uint32_t s_g = bcast_lo(sc2), s_g8 = bcast_hi(sc2);
  const float w_g = e8m0_to_f32(two & 0xFFu), w_g8 = e8m0_to_f32(two >> 8);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t r[4];
    e2m1x8_to_f16x8(words[q], r[0], r[1], r[2], r[3]);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t row =
          packed_to_row(layout, rt * kTileRows + j * 16 + g + ((b & 1) ? 8 : 0), N, split);
      int64_t k0 = kt * kTileK + 16 * t + 4 * q + ((b >> 1) ? 2 : 0);
      if (row >= 0 && k0 < K) {
        float lo, hi;
        if (wide) {
          const __half2 hc = *reinterpret_cast<const __half2*>(&r[b]);
          const float sw = (b & 1) ? w_g8 : w_g;
          lo = __low2float(hc) * sw;
          hi = __high2float(hc) * sw;
        } else {
          uint32_t p = hmul2_u32(r[b], (b & 1) ? s_g8 : s_g);
          __half2 hp = *reinterpret_cast<__half2*>(&p);
          float f = h->factor[row < split ? 0 : 1];
          lo = __low2float(hp) * f;
          hi = __high2float(hp) * f;
        }
        out[row * K + k0] = lo;
        out[row * K + k0 + 1] = hi;
      }
    }
  }
}

// ------------------------------------------------------------------ host launchers
cudaError_t launch_prepack(const uint8_t* const codes[2], const uint8_t* const scales[2],
                           int64_t split, float f0, float f1, int fmt, int64_t N, int64_t K,
                           int64_t RT, int64_t KT, uint32_t layout, void* dst, cudaStream_t s) {
  PackedHeader* h = reinterpret_cast<PackedHeader*>(dst);
  uint8_t* tiles = reinterpret_cast<uint8_t*>(dst) + kHeaderBytes;
  SrcPair sp{{codes[0], codes[1]}, {scales[0], scales[1]}, split, layout};
  k_header<<<1, 32, 0, s>>>(h, fmt, N, K, split, f0, f1, layout);
  if (fmt == FMT_MX) {
    int64_t total = N * (K / 32);
    int64_t nb = (total + 255) / 256;
    int blocks = static_cast<int>(nb < 4096 ? nb : 4096);
    k_mx_emax<<<blocks, 256, 0, s>>>(sp, N, K, h);
    k_mx_factor<<<1, 32, 0, s>>>(h);
  }
  k_pack<<<static_cast<unsigned>(RT * KT), 256, 0, s>>>(sp, fmt, N, K, KT, tiles, h);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const void* packed, int fmt, int64_t N, int64_t K, int64_t RT,
                          int64_t KT, int64_t split, uint32_t layout, uint8_t* codes,
                          uint8_t* scales, cudaStream_t s) {
  const PackedHeader* h = reinterpret_cast<const PackedHeader*>(packed);
  const uint8_t* tiles = reinterpret_cast<const uint8_t*>(packed) + kHeaderBytes;
  k_unpack<<<static_cast<unsigned>(RT * KT), 256, 0, s>>>(tiles, fmt, N, K, KT, split, layout,
                                                          h, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const void* packed, int fmt, int64_t N, int64_t K, int64_t RT,
                           int64_t KT, int64_t split, uint32_t layout, float* out,
                           cudaStream_t s) {
  const PackedHeader* h = reinterpret_cast<const PackedHeader*>(packed);
  const uint8_t* tiles = reinterpret_cast<const uint8_t*>(packed) + kHeaderBytes;
  k_dequant<<<static_cast<unsigned>(RT * KT), 256, 0, s>>>(tiles, fmt, N, K, KT, split, layout,
                                                           h, out);
  return cudaGetLastError();
}

}  // namespace vt
