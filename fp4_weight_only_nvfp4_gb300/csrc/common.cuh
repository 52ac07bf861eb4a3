// Shared device-side definitions of libvtfp4: the prepacked tile layout and small PTX
// wrappers (TMA bulk copies, mbarriers, FP4/FP8 conversions, mma.sync).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vt {

// ------------------------------------------------------------------ packed layout
// A weight W[N][K] is stored as a 256-byte header followed by tiles of 128 rows x 64 k,
// tile (rt, kt) at byte 256 + (rt * KT + kt) * tile_bytes, rows padded to 128 and k to 64
// with zero bytes.  Inside a tile:
//   codes  [8 row blocks j][32 lanes][16 B]  (4096 B).  Lane l = 4g + t, byte 4q + b:
//          b=0: row 16j+g,   source byte kt*32 + 8t + 2q       (k = 64kt+16t+4q+{0,1})
//          b=1: row 16j+g+8, same byte
//          b=2: row 16j+g,   source byte kt*32 + 8t + 2q + 1   (k = 64kt+16t+4q+{2,3})
//          b=3: row 16j+g+8, same byte
//          i.e. word q of lane l is the f16 A-operand fragment of an m16n8k16 MMA for k
//          step q, with the MMA's logical k columns {2t,2t+1,2t+8,2t+9} mapped onto the
//          four consecutive physical k = 64kt+16t+4q+{0..3}.  Lane t therefore covers
//          physical k in [16t, 16t+16) of the tile over the four steps.
//   scales NVFP4 [4 row-block pairs jp][32 lanes][2 j][2 B] (512 B): E4M3 bytes of rows
//          16j+g and 16j+g+8 (j = 2jp + j&1) for group 4kt+t (the 16 k lane t covers).
//   scales MXFP4 [4 jp][8 g][2 h][2 j][2 B] (256 B): rows 16j+g, 16j+g+8, group 2kt+h;
//          the bytes are re-encoded as the high byte of an f16 power of two (see prepack),
//          or kept as raw E8M0 bytes when the weight's scales span more exponents than
//          that encoding holds (header field `wide`).
//   so the four scale bytes lane (g, t) needs for a row-block pair form one 32-bit word.
constexpr int kHeaderBytes = 256;
constexpr int kTileRows = 128;
constexpr int kTileK = 64;
constexpr int kCodeBytes = 4096;
constexpr int kScaleBytesNV = 512;
constexpr int kScaleBytesMX = 256;
constexpr int kTileBytesNV = kCodeBytes + kScaleBytesNV;  // 4608
constexpr int kTileBytesMX = kCodeBytes + kScaleBytesMX;  // 4352

enum { FMT_NV = 0, FMT_MX = 1 };

__host__ __device__ constexpr int tile_bytes(int fmt) {
  return fmt == FMT_NV ? kTileBytesNV : kTileBytesMX;
}

// Byte offset, inside a tile, of the two scale bytes (rows g, g+8) lane (g, t) of row
// block j needs.
__host__ __device__ constexpr int scale_offset(int fmt, int j, int g, int t) {
  return fmt == FMT_NV ? kCodeBytes + (j >> 1) * 128 + (4 * g + t) * 4 + (j & 1) * 2
                       : kCodeBytes + (j >> 1) * 64 + (g * 2 + (t >> 1)) * 4 + (j & 1) * 2;
}

// Header written by the prepack kernels and read by the GEMM epilogue.
struct PackedHeader {
  uint32_t magic;      // 'VTF4'
  uint32_t fmt;
  int64_t N, K;
  int64_t seg_split;   // rows [0, seg_split) use factor[0], the rest factor[1]
  float factor[2];     // epilogue multiplier per segment (NVFP4 global, MXFP4 2^(emax-140))
  int32_t emax[2];     // MXFP4: largest finite E8M0 byte per segment
  uint32_t layout;     // kLayoutRows or kLayoutPaired
  int32_t emin[2];     // MXFP4: smallest finite E8M0 byte per segment
  uint32_t wide;       // MXFP4: 1 when a segment's finite scale bytes span more than the
                       // 30 exponents the f16 re-encoding holds; the tiles then keep the raw
                       // E8M0 bytes and the kernels apply each group scale exactly (factor 1)
  uint32_t pad[48];
};
static_assert(sizeof(PackedHeader) == kHeaderBytes, "header size");
constexpr uint32_t kMagic = 0x34465456u;  // "VTF4"

// Row order of the packed tiles.  kLayoutRows: packed row p is weight row p (a fused
// gate_up weight stacks gate rows [0, I) over up rows [I, 2I)).  kLayoutPaired (fused
// gate_up only): each 128-row tile holds 64 gate rows and the same 64 up rows, so the
// SiLU-and-multiply of a pair happens inside one tile: packed row p of tile r = p / 128 is
// gate row 64r + (p % 128) when p % 128 < 64, else up row 64r + (p % 128) - 64.
enum : uint32_t { kLayoutRows = 0, kLayoutPaired = 1 };

// The weight row (in gate-over-up order, 0 <= n < 2I or < N) that packed row p holds, or
// -1 for a padding row.  `I` is the gate/up split (the fused weight's half size).
__host__ __device__ __forceinline__ int64_t packed_to_row(uint32_t layout, int64_t p, int64_t N,
                                                          int64_t I) {
  if (layout == kLayoutPaired) {
    const int64_t r = (p >> 7) * 64 + (p & 63);
    if (r >= I) return -1;
    return (p & 64) ? I + r : r;
  }
  return p < N ? p : -1;
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D TMA bulk copy global -> shared, completion signalled on `bar` (tx bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after `limit_ns` of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Two E2M1 codes (one byte, low nibble -> low half) to f16x2, exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 lo;\n .reg .b16 h;\n cvt.u16.u32 h, %1;\n cvt.u8.u16 lo, h;\n"
      " cvt.rn.f16x2.e2m1x2 %0, lo;\n}"
      : "=r"(r)
      : "r"(byte));
  return r;
}

// Four codes bytes of a word -> four f16x2.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t& r0, uint32_t& r1,
                                                uint32_t& r2, uint32_t& r3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) to f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  uint16_t h = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}

// Two re-encoded MXFP4 scale bytes -> f16x2 (each byte is the high byte of its f16).
__device__ __forceinline__ uint32_t mxenc2_to_f16x2(uint32_t two_bytes) {
  return __byte_perm(two_bytes, 0u, 0x1404);
}

// E8M0 byte -> its value 2^(e - 127) as an fp32 (exact: 2^-127 is an fp32 subnormal);
// 0xFF -> NaN.  The OCP Microscaling definition of the MXFP4 scale.
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  return e == 0xFFu ? __uint_as_float(0x7FC00000u)
                    : (e == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Broadcast the low / high f16 of a pair to both halves.
__device__ __forceinline__ uint32_t bcast_lo(uint32_t x) { return __byte_perm(x, 0u, 0x1010); }
__device__ __forceinline__ uint32_t bcast_hi(uint32_t x) { return __byte_perm(x, 0u, 0x3232); }

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int4 ld_shared_v4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// ---------------------------------------------------- activation conversion (bf16 -> f16)
// A tile of bf16 activations becomes f16 values A * 2^-p with one power of two p per tile:
// p = (exponent of the largest magnitude) - 14, clamped to [-120, 113], so that every value
// lands below 2^15 and values down to about 2^-31 of the largest one keep all their bits (the
// f16 subnormals end at 2^-24); p = 0 for an all-zero tile or one holding a NaN (infinities
// and NaNs pass through as such).

// Largest bf16 magnitude pattern (sign cleared) among the 8 values of a 16-byte granule.
__device__ __forceinline__ int act_maxmag8(const uint32_t w[4]) {
  int mx = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    mx = max(mx, (int)(w[q] & 0x7FFFu));
    mx = max(mx, (int)((w[q] >> 16) & 0x7FFFu));
  }
  return mx;
}

// The tile's power of two from its largest magnitude pattern.
__device__ __forceinline__ int act_pow2(int mx) {
  if (mx <= 0 || mx > 0x7F80) return 0;
  const int p = ((mx >> 7) - 127) - 14;  // exponent of the largest magnitude (subnormals: -127)
  return p < -120 ? -120 : (p > 113 ? 113 : p);
}

// 2^k in fp32 for k in [-126, 127] (a normal power of two), from its exponent field.
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// One granule times 2^-p, rounded to f16, as four f16x2 words (p in [-120, 113]).
__device__ __forceinline__ uint4 act_granule_f16(const uint32_t w[4], int p) {
  const float down = pow2f(-p);
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2 h = __floats2half2_rn(__uint_as_float(w[q] << 16) * down,
                                        __uint_as_float(w[q] & 0xFFFF0000u) * down);
    o[q] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ int4 ld_global_nc_v4(const void* p) {
  int4 v;
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace vt
