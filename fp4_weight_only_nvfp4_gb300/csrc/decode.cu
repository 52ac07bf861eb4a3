// Decode GEMM (M <= 16): C[M][N] = A[M][K] . W[N][K]^T with W streamed from the packed
// tile layout.  Sources: "keep the ModelOpt NVFP4 lm_head packed" (vllm.cpp PR #263),
// "Why this row matters" (W4A16 decode is pure weight traffic); "re-verify 27B NVFP4"
// (PR #178), "Attribution" (the FP4 MLP GEMM at ~68% of the bandwidth roof is the lever);
// "MXFP4 decode-graph + gate_up FUSION" (PR #54), "Step 3" (CTA count per SM decides the
// residual; a regrouped fp32 reduce moves bf16 ULPs, so reductions here have a fixed
// order); "re-verify 27B NVFP4" (PR #178): a split-K workspace whose spin-locks were not
// zeroed hung the GPU, so this kernel has no spin-locks (the last CTA to arrive reduces).
//
// Design (GB300): one persistent CTA per SM, W warps.  Work items are (128-row tile,
// 64-k tile) pairs in row-tile-major order; CTA c owns items [c*I/G, (c+1)*I/G).  Each
// warp streams its items (every W-th item of the CTA's range) through its own ring of D
// shared-memory stages filled by 1-D TMA bulk copies (weights + the matching slice of the
// converted activations), dequantises in registers (E2M1 -> f16 by cvt, times the group
// scale in f16, both exact) and accumulates with m16n8k16 MMAs in fp32.  At the end of
// each row-tile segment the warps' partial sums are added in warp order through shared
// memory; a row tile shared by several CTAs is finished by the last CTA to arrive, which
// adds the CTAs' partials in CTA order.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace vt {

constexpr int kSlotPad = 132;  // floats per token row of a warp's reduction slot
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

int decode_mt(int M) { return M <= 8 ? 8 : 16; }

size_t decode_smem_bytes(int fmt, int mt, int warps, int stages) {
  size_t stage = tile_bytes(fmt) + (size_t)mt * 128;
  return (size_t)warps * stages * stage + (size_t)warps * mt * kSlotPad * 4 +
         (size_t)warps * stages * 8 + 64;
}

// ------------------------------------------------------------- activation pre-pass
// One block per token row m: A'[kt][m][64] (f16) = A[m][k] * 2^-p[m], rowscale[m] = 2^p[m],
// with p chosen from the row's largest magnitude so that every value lands below 2^15
// (no f16 overflow) and values down to 2^-31 of the maximum stay exact.  The 16-byte
// granules of each 128-byte row are stored XOR-swizzled by (m & 7) so that the MMA
// fragment reads from shared memory are free of bank conflicts.
__global__ void __launch_bounds__(256) k_prep_a(const __nv_bfloat16* __restrict__ A,
                                                int64_t lda, int64_t K, int64_t KT, int mt,
                                                __half* __restrict__ Ap,
                                                float* __restrict__ rowscale) {
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t sm_row[];
  __shared__ int red[8];
  const int m = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(A + m * lda);
  uint4* row = reinterpret_cast<uint4*>(sm_row);
  int mx = 0;
  for (int64_t v = threadIdx.x; v < K / 8; v += blockDim.x) {
    uint4 x = src[v];
    row[v] = x;
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mx = max(mx, (int)(w[i] & 0x7FFFu));
      mx = max(mx, (int)((w[i] >> 16) & 0x7FFFu));
    }
  }
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) mx = max(mx, red[i]);
  int p = 0;
  if (mx > 0 && mx <= 0x7F80) {
    int e = (mx >> 7) - 127;  // exponent of the largest magnitude (subnormals: -127)
    p = e - 14;
    p = p < -120 ? -120 : (p > 113 ? 113 : p);
  }
  const float down = ldexpf(1.0f, -p);
  const __nv_bfloat16* rb = reinterpret_cast<const __nv_bfloat16*>(sm_row);
  for (int64_t c = threadIdx.x; c < KT * 8; c += blockDim.x) {
    const int64_t kt = c >> 3;
    const int gi = (int)(c & 7);
    const int64_t k0 = kt * 64 + gi * 8;
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo = (k0 + 2 * i < K) ? __bfloat162float(rb[k0 + 2 * i]) * down : 0.0f;
      float hi = (k0 + 2 * i + 1 < K) ? __bfloat162float(rb[k0 + 2 * i + 1]) * down : 0.0f;
      __half2 h = __floats2half2_rn(lo, hi);
      o[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    uint4* dst = reinterpret_cast<uint4*>(Ap + ((kt * mt + m) * 64 + ((gi ^ (m & 7)) * 8)));
    *dst = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) rowscale[m] = ldexpf(1.0f, p);
}

// ------------------------------------------------------------------- main kernel
struct DecodeParams {
  const uint8_t* tiles;
  const PackedHeader* hdr;
  int64_t N, KT, items, seg_split, ldc;
  int M, stages;
  const __half* Ap;
  const float* rowscale;
  __nv_bfloat16* C;
  float* partials;
  int* counters;
  int* status;
};

__device__ __forceinline__ int64_t owner_of(int64_t i, int64_t I, int64_t G) {
  return ((i + 1) * G - 1) / I;  // the CTA c with c*I/G <= i < (c+1)*I/G
}

template <int FMT, int MT>
__global__ void __launch_bounds__(256, 1) k_decode(const DecodeParams p) {
  constexpr int TB = tile_bytes(FMT);
  constexpr int AB = MT * 128;  // activation bytes of one k tile (all MT rows)
  constexpr int NJ = MT / 8;    // n8 MMA column blocks
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_flag;

  const int W = blockDim.x >> 5;
  const int D = p.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t G = gridDim.x, c = blockIdx.x, I = p.items, KT = p.KT;
  const int64_t i0 = c * I / G, i1 = (c + 1) * I / G;
  const int STAGE = TB + AB;

  uint8_t* ring = smem + (size_t)warp * D * STAGE;
  float* slots = reinterpret_cast<float*>(smem + (size_t)W * D * STAGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)W * D * STAGE +
                                               (size_t)W * MT * kSlotPad * 4) +
                   warp * D;
  const uint32_t ring_u = smem_u32(ring);
  const uint32_t bar_u = smem_u32(bars);
  const int abytes = p.M * 128;  // only the valid token rows are copied
  const uint32_t tx = TB + abytes;

  const int64_t span = i1 - i0;
  const int64_t n_my = span > warp ? (span - warp + W - 1) / W : 0;

  if (lane == 0)
    for (int d = 0; d < D; ++d) mbar_init(bar_u + 8 * d, 1);
  fence_mbar_init();
  __syncthreads();

  const uint64_t pol = l2_evict_first_policy();   // weights: streamed once
  const uint64_t pol_a = l2_evict_last_policy();  // activations: re-read by every CTA
  // Weights do not depend on the activation pre-pass: start streaming them first.
  if (lane == 0) {
    for (int64_t n = 0; n < n_my && n < D; ++n) {
      const int64_t item = i0 + warp + W * n;
      const uint32_t bar = bar_u + 8 * (uint32_t)n;
      mbar_expect_tx(bar, tx);  // one arrival for the stage: weights + activations
      bulk_g2s(ring_u + (uint32_t)n * STAGE, p.tiles + item * TB, TB, bar, pol);
    }
  }
  pdl_wait();  // the converted activations are ready past this point
  if (lane == 0) {
    fence_proxy_async_all();
    for (int64_t n = 0; n < n_my && n < D; ++n) {
      const int64_t item = i0 + warp + W * n;
      const int64_t kt = item % KT;
      const uint32_t bar = bar_u + 8 * (uint32_t)n;
      bulk_g2s(ring_u + (uint32_t)n * STAGE + TB, p.Ap + kt * MT * 64, abytes, bar, pol_a);
    }
  }

  const float f0 = p.hdr->factor[0], f1 = p.hdr->factor[1];
  bool ok = true;
  int64_t n = 0;  // this warp's item counter
  int64_t issued = n_my < D ? n_my : D;
  const int64_t rt_first = i0 / KT, rt_last = (i1 - 1) / KT;

  for (int64_t rt = rt_first; rt <= rt_last; ++rt) {
    const int64_t seg_hi = min(i1, (rt + 1) * KT);
    float acc[8][NJ][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int u = 0; u < NJ; ++u)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[j][u][r] = 0.0f;

    while (n < n_my) {
      const int64_t item = i0 + warp + W * n;
      if (item >= seg_hi) break;
      const int slot = (int)(n % D);
      const uint32_t parity = (uint32_t)((n / D) & 1);
      if (ok) ok = mbar_wait_bounded(bar_u + 8 * slot, parity, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        const uint32_t sbase = ring_u + (uint32_t)slot * STAGE;
        // activation fragments (B operand): token rows g and g+8, physical k 16t..16t+15
        uint32_t bfr[NJ][4][2];
#pragma unroll
        for (int u = 0; u < NJ; ++u) {
          const int m = g + 8 * u;
          if (m < p.M) {
            const uint32_t rowa = sbase + TB + m * 128;
            const int4 v0 = ld_shared_v4(rowa + (((2 * t) ^ (m & 7)) << 4));
            const int4 v1 = ld_shared_v4(rowa + (((2 * t + 1) ^ (m & 7)) << 4));
            bfr[u][0][0] = v0.x; bfr[u][0][1] = v0.y;
            bfr[u][1][0] = v0.z; bfr[u][1][1] = v0.w;
            bfr[u][2][0] = v1.x; bfr[u][2][1] = v1.y;
            bfr[u][3][0] = v1.z; bfr[u][3][1] = v1.w;
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) bfr[u][q][0] = bfr[u][q][1] = 0u;
          }
        }
        const int soff = (FMT == FMT_NV) ? lane * 16 : ((g * 2 + (t >> 1)) * 16);
        const int4 sv = ld_shared_v4(sbase + kCodeBytes + soff);
        const uint32_t sw[4] = {(uint32_t)sv.x, (uint32_t)sv.y, (uint32_t)sv.z, (uint32_t)sv.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int4 wv = ld_shared_v4(sbase + j * 512 + lane * 16);
          const uint32_t two = (sw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
          const uint32_t sc = (FMT == FMT_NV) ? e4m3x2_to_f16x2(two) : mxenc2_to_f16x2(two);
          const __half2 sc2 = *reinterpret_cast<const __half2*>(&sc);
          const __half2 sg = __low2half2(sc2), sg8 = __high2half2(sc2);
          const uint32_t words[4] = {(uint32_t)wv.x, (uint32_t)wv.y, (uint32_t)wv.z,
                                     (uint32_t)wv.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t r0, r1, r2, r3;
            e2m1x8_to_f16x8(words[q], r0, r1, r2, r3);
            __half2 h0 = __hmul2(*reinterpret_cast<__half2*>(&r0), sg);
            __half2 h1 = __hmul2(*reinterpret_cast<__half2*>(&r1), sg8);
            __half2 h2 = __hmul2(*reinterpret_cast<__half2*>(&r2), sg);
            __half2 h3 = __hmul2(*reinterpret_cast<__half2*>(&r3), sg8);
            const uint32_t a0 = *reinterpret_cast<uint32_t*>(&h0);
            const uint32_t a1 = *reinterpret_cast<uint32_t*>(&h1);
            const uint32_t a2 = *reinterpret_cast<uint32_t*>(&h2);
            const uint32_t a3 = *reinterpret_cast<uint32_t*>(&h3);
#pragma unroll
            for (int u = 0; u < NJ; ++u)
              mma_f16_16816(acc[j][u], a0, a1, a2, a3, bfr[u][q][0], bfr[u][q][1]);
          }
        }
      }
      __syncwarp();
      // refill this slot with the item D ahead
      if (lane == 0 && ok && issued < n_my) {
        fence_proxy_async_smem();
        const int64_t nitem = i0 + warp + W * issued;
        const uint32_t bar = bar_u + 8 * slot;
        const uint32_t dst = ring_u + (uint32_t)slot * STAGE;
        mbar_expect_tx(bar, tx);
        bulk_g2s(dst, p.tiles + nitem * TB, TB, bar, pol);
        bulk_g2s(dst + TB, p.Ap + (nitem % KT) * MT * 64, abytes, bar, pol_a);
      }
      issued = (ok && issued < n_my) ? issued + 1 : issued;
      ++n;
    }

    // ---- segment flush: warp partials -> slots -> fixed-order sum
    float* my = slots + (size_t)warp * MT * kSlotPad;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int u = 0; u < NJ; ++u) {
        const int m0 = 2 * t + 8 * u;
        const int r0 = j * 16 + g;
        my[m0 * kSlotPad + r0] = acc[j][u][0];
        my[(m0 + 1) * kSlotPad + r0] = acc[j][u][1];
        my[m0 * kSlotPad + r0 + 8] = acc[j][u][2];
        my[(m0 + 1) * kSlotPad + r0 + 8] = acc[j][u][3];
      }
    __syncthreads();

    const int64_t seg_lo = max(i0, rt * KT);
    const int64_t c_lo = owner_of(rt * KT, I, G), c_hi = owner_of(rt * KT + KT - 1, I, G);
    const bool complete = (c_lo == c_hi);
    (void)seg_lo;
    const int sel = (rt == rt_first) ? 0 : 1;
    const int nout = p.M * 128;
    for (int idx = threadIdx.x; idx < nout; idx += blockDim.x) {
      const int m = idx >> 7, row = idx & 127;
      float s = 0.0f;
      for (int w = 0; w < W; ++w) s += slots[((size_t)w * MT + m) * kSlotPad + row];
      const int64_t rowg = rt * kTileRows + row;
      if (complete) {
        if (rowg < p.N) {
          const float f = rowg < p.seg_split ? f0 : f1;
          p.C[(int64_t)m * p.ldc + rowg] = __float2bfloat16_rn(s * f * p.rowscale[m]);
        }
      } else {
        p.partials[(((size_t)c * 2 + sel) * MT + m) * 128 + row] = s;
      }
    }
    if (!complete) {
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) {
        const int prev = atomicAdd(&p.counters[rt], 1);
        const int last = (prev == (int)(c_hi - c_lo));
        if (last) {
          __threadfence();
          p.counters[rt] = 0;  // self-reset for the next call
        }
        s_flag = last;
      }
      __syncthreads();
      if (s_flag) {
        for (int idx = threadIdx.x; idx < nout; idx += blockDim.x) {
          const int m = idx >> 7, row = idx & 127;
          float s = 0.0f;
          for (int64_t cc = c_lo; cc <= c_hi; ++cc) {
            const int selc = (rt == (cc * I / G) / KT) ? 0 : 1;
            s += __ldcg(&p.partials[(((size_t)cc * 2 + selc) * MT + m) * 128 + row]);
          }
          const int64_t rowg = rt * kTileRows + row;
          if (rowg < p.N) {
            const float f = rowg < p.seg_split ? f0 : f1;
            p.C[(int64_t)m * p.ldc + rowg] = __float2bfloat16_rn(s * f * p.rowscale[m]);
          }
        }
      }
    }
    __syncthreads();  // slots are rewritten by the next segment
  }

  if (!ok) {
    if (lane == 0) atomicExch(p.status, 5);
    // wait (bounded) for this warp's copies still in flight before leaving
    for (int64_t x = n; x < issued; ++x)
      mbar_wait_bounded(bar_u + 8 * (int)(x % D), (uint32_t)((x / D) & 1), 100000000ull);
  }
}

// Raises a kernel's dynamic shared memory limit once per device (never during a capture:
// the first call on a device, made before any capture, does it).
template <typename Kern>
static cudaError_t allow_smem(Kern* k, int bytes, int* done_per_device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done_per_device[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done_per_device[dev] = bytes;
  return e;
}

template <int FMT, int MT>
static cudaError_t launch_t(const DecodeLaunch& L, cudaStream_t s) {
  static int done[64] = {0};
  const size_t smem = decode_smem_bytes(FMT, MT, L.warps, L.stages);
  cudaError_t e = allow_smem(k_decode<FMT, MT>, 227 * 1024, done);
  if (e != cudaSuccess) return e;
  DecodeParams p;
  p.tiles = reinterpret_cast<const uint8_t*>(L.packed) + kHeaderBytes;
  p.hdr = reinterpret_cast<const PackedHeader*>(L.packed);
  p.N = L.N;
  p.KT = L.KT;
  p.items = L.RT * L.KT;
  p.seg_split = L.seg_split;
  p.ldc = L.ldc;
  p.M = L.M;
  p.stages = L.stages;
  p.Ap = reinterpret_cast<const __half*>(L.Ap);
  p.rowscale = L.rowscale;
  p.C = reinterpret_cast<__nv_bfloat16*>(L.C);
  p.partials = L.partials;
  p.counters = L.counters;
  p.status = L.status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)L.grid);
  cfg.blockDim = dim3((unsigned)(L.warps * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode<FMT, MT>, p);
}

cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t s, int* launches) {
  const int mt = decode_mt(L.M);
  static int done[64] = {0};
  const size_t prep_smem = (size_t)((L.K + 7) / 8) * 16;
  cudaError_t e = cudaSuccess;
  if (prep_smem > 48 * 1024) {
    if (prep_smem > 227 * 1024) return cudaErrorInvalidValue;
    e = allow_smem(k_prep_a, 227 * 1024, done);
    if (e != cudaSuccess) return e;
  }
  k_prep_a<<<L.M, 256, prep_smem, s>>>(reinterpret_cast<const __nv_bfloat16*>(L.A), L.lda,
                                       L.K, L.KT, mt, reinterpret_cast<__half*>(L.Ap),
                                       L.rowscale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (L.fmt == FMT_NV) e = (mt == 8) ? launch_t<FMT_NV, 8>(L, s) : launch_t<FMT_NV, 16>(L, s);
  else e = (mt == 8) ? launch_t<FMT_MX, 8>(L, s) : launch_t<FMT_MX, 16>(L, s);
  if (launches) *launches = 2;
  return e;
}

}  // namespace vt
