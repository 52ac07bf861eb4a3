// Prefill GEMM (M > 16): C[M][N] = A[M][K] . W[N][K]^T on the 5th-generation tensor cores.
// Sources: the "FP4 weight-only" path of the pages applies to every M, and a prefill-sized
// batch makes the layer a dense contraction ("keep the ModelOpt NVFP4 lm_head packed",
// vllm.cpp PR #263: the packed FP4 weight is the only copy kept in memory, so the weights
// are dequantised on the fly inside the GEMM rather than materialised).
//
// Design (GB300, one persistent CTA per SM, 14 warps):
//   warp 0      TMA producer: per 64-k step, the activation tile (128 tokens x 64 k, f16,
//               128-byte swizzled by the tensor map) and the two packed 128-row weight tiles.
//   warp 1      allocates TMEM (two 128 x 256 fp32 accumulators) and, on one thread, issues
//               tcgen05.mma kind::f16 (M=128 tokens, N=256 weight rows, K=16) per k step.
//   warps 2-9   dequantise the packed tiles in registers (E2M1 -> f16 by cvt, times the
//               group scale in f16: exact) into a 256 x 64 f16 K-major 128-byte-swizzled
//               shared-memory tile, the MMA's B operand.
//   warps 10-13 epilogue: tcgen05.ld of the finished accumulator, times the token's
//               activation scale and the weight's global factor, RNE to bf16, store.
// Activations: a pre-pass writes A' = A * 2^-p (f16) with one power-of-two p per token row,
// so every row lands below 2^15; the epilogue multiplies by 2^p.  Products of f16 operands
// are exact and accumulate in fp32 in TMEM.
//
// Every wait is bounded (2 s of wall time); a timeout sets the workspace status word and
// makes every role leave its loop; in-flight copies and MMAs are drained (again bounded)
// before TMEM is released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "actq.cuh"
#include "common.cuh"
#include "kernels.h"

namespace vt {

namespace {

constexpr uint64_t kPfWaitNs = 2000000000ull;  // drains of copies and MMAs in flight
constexpr int kBM = 128;          // tokens per tile (MMA M)
constexpr int kBN = 256;          // weight rows per tile (MMA N): two packed row tiles
// A tile is 256 weight rows x 2 token tiles of 128: one dequantised B tile serves two MMAs
// per k step (the B-tile work and shared-memory traffic per flop are halved); the two
// accumulators then fill the 512 TMEM columns, so the epilogue of a tile does not overlap
// the next tile's MMAs.
constexpr int kPair = 2;
constexpr int kAStages = 4;       // activation stages, each the pair of 128 x 64 tiles
constexpr int kPStages = 3;
constexpr int kBStages = 2;
constexpr int kDeqWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kPfThreads = (2 + kDeqWarps + kEpiWarps) * 32;  // 448
constexpr int kABytes = kBM * kTileK * 2;                     // 16 KB
constexpr int kAStageBytes = kPair * kABytes;                 // 32 KB
constexpr int kBBytes = kBN * kTileK * 2;                     // 32 KB
constexpr uint32_t kTmemCols = 512;                           // 2 x 256 fp32 columns

// Shared-memory map (from a 1024-byte aligned base).
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kAStages * kAStageBytes;
constexpr int kOffP = kOffB + kBStages * kBBytes;
__host__ __device__ constexpr int off_bar(int fmt) { return kOffP + kPStages * 2 * tile_bytes(fmt); }
constexpr int kNumBars = 2 * kAStages + 2 * kPStages + 2 * kBStages + 4 + 1;
__host__ __device__ constexpr int prefill_smem(int fmt) { return off_bar(fmt) + kNumBars * 8 + 16 + 1024; }

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[tmem] (+)= A[smem desc] . B[smem desc]^T, kind::f16, one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// 32 lanes x 32 columns of fp32 from TMEM (lane = this warp's quarter + thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// The same load, only issued: the registers are valid after tmem_ld_wait on them.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
// Waits for every TMEM load this thread issued; v (the last one's registers) is read
// and written by the wait, so no use of v moves above it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
        "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
        "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]),
        "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]),
        "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
      :
      : "memory");
}
// 32 bytes to global memory in one store (address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(ptr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                  "r"(w[6]), "r"(w[7])
               : "memory");
}
// 2-D tiled TMA load (tensor map in kernel parameter space), completion on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Shared-memory matrix descriptor of a K-major operand tile whose rows are 128 bytes, stored
// in the canonical 128-byte swizzle (8-row groups 1024 bytes apart; base 1024-aligned).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor: kind::f16, A = B = f16, D = f32, both K-major, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);
// The same with A = B = bf16 (the operand-format fields: 0 = f16, 1 = bf16): the tiles of a
// wide MXFP4 weight, whose exact values c * 2^(e - 127) need bf16's exponent range.
constexpr uint32_t kIdescBF16 = kIdesc | (1u << 7) | (1u << 10);

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bounded wait that also gives up when another role has already given up.
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                        uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
}

struct PrefillParams {
  const uint8_t* tiles;
  const PackedHeader* hdr;
  int64_t N, RT, KT, M, ldc, seg_split;
  int64_t mtiles, mptiles, tiles_total;  // token tiles, token-tile pairs, (pair, 256 rows) tiles
  const float* rowscale;
  __nv_bfloat16* C;
  int* status;
  int vec_store;     // C 16-byte aligned and ldc % 8 == 0
  int vec32_store;   // C 32-byte aligned and ldc % 16 == 0
  int pair_store;    // C 4-byte aligned and ldc even: two outputs per 32-bit store
  uint64_t wait_ns;  // limit of every bounded wait
  int withhold;      // test hook: issue no copies (the waits then run out)
  uint32_t layout;   // packed row order (kLayoutRows / kLayoutPaired)
  int silu;          // paired gate_up: C[M][I] = silu(gate) * up
};

// SiLU(x) = x / (1 + e^-x) in fp32 (e^-x overflowing to infinity gives -0 for large -x).
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

template <int FMT>
__global__ void __launch_bounds__(kPfThreads, 1)
    k_prefill(const __grid_constant__ CUtensorMap tmA, const PrefillParams p) {
  constexpr int TB = tile_bytes(FMT);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base_u = (raw_u + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u - raw_u);
  const uint32_t sA = base_u + kOffA, sB = base_u + kOffB, sP = base_u + kOffP;
  const uint32_t bars = base_u + off_bar(FMT);
  const uint32_t a_full = bars, a_empty = a_full + 8 * kAStages;
  const uint32_t p_full = a_empty + 8 * kAStages, p_empty = p_full + 8 * kPStages;
  const uint32_t b_full = p_empty + 8 * kPStages, b_empty = b_full + 8 * kBStages;
  const uint32_t acc_full = b_empty + 8 * kBStages, acc_empty = acc_full + 16;
  const uint32_t drain = acc_empty + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + off_bar(FMT) + kNumBars * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(a_full + 8 * s, 1);
      mbar_init(a_empty + 8 * s, 1);
    }
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(p_full + 8 * s, 1);
      mbar_init(p_empty + 8 * s, kDeqWarps);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(b_full + 8 * s, kDeqWarps);
      mbar_init(b_empty + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(acc_full + 8 * s, 1);
      mbar_init(acc_empty + 8 * s, kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort = 0;
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t KT = p.KT, RT = p.RT, mtiles = p.mtiles, mptiles = p.mptiles, T = p.tiles_total;
  const int64_t G = gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && !p.withhold) {
      // a weight tile serves the token tiles running beside it; an activation tile serves
      // every weight tile over the whole run
      const uint64_t pol_w = l2_evict_normal_policy();
      const uint64_t pol_a = l2_evict_last_policy();
      uint32_t ia = 0, pa = 0, ip = 0, pp = 0;
      int a_issued = 0, p_issued = 0;  // copies issued (for the drain after a timeout)
      bool ok = true;
      for (int64_t tile = blockIdx.x; ok && tile < T; tile += G) {
        const int64_t nt = tile / mptiles, mt0 = 2 * (tile % mptiles);
        const bool two = mt0 + 1 < mtiles;
        const int64_t rt0 = 2 * nt;
        const int nrt = (RT - rt0) >= 2 ? 2 : 1;
        for (int64_t kt = 0; kt < KT; ++kt) {
          if (!(ok = pf_wait(a_empty + 8 * ia, pa ^ 1u, abort, p.wait_ns))) break;
          mbar_expect_tx(a_full + 8 * ia, two ? 2 * kABytes : kABytes);
          tma_load_2d(sA + ia * kAStageBytes, &tmA, (int)(kt * kTileK), (int)(mt0 * kBM),
                      a_full + 8 * ia, pol_a);
          if (two)
            tma_load_2d(sA + ia * kAStageBytes + kABytes, &tmA, (int)(kt * kTileK),
                        (int)((mt0 + 1) * kBM), a_full + 8 * ia, pol_a);
          ++a_issued;
          if (++ia == kAStages) { ia = 0; pa ^= 1u; }
          if (!(ok = pf_wait(p_empty + 8 * ip, pp ^ 1u, abort, p.wait_ns))) break;
          mbar_expect_tx(p_full + 8 * ip, (uint32_t)(nrt * TB));
          for (int r = 0; r < nrt; ++r)
            bulk_g2s(sP + (ip * 2 + r) * TB, p.tiles + ((rt0 + r) * KT + kt) * TB, TB,
                     p_full + 8 * ip, pol_w);
          ++p_issued;
          if (++ip == kPStages) { ip = 0; pp ^= 1u; }
        }
      }
      if (!ok) {
        atomicExch(p.status, 5);
        // Let the copies already issued land before the CTA's shared memory is released:
        // the most recent issue on each slot completes that slot's current phase.
        for (int k = 0; k < kAStages && k < a_issued; ++k) {
          ia = ia == 0 ? kAStages - 1 : ia - 1;
          if (ia == kAStages - 1) pa ^= 1u;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a_full + 8 * ia, pa) && globaltimer_ns() - t0 < kPfWaitNs) {}
        }
        for (int k = 0; k < kPStages && k < p_issued; ++k) {
          ip = ip == 0 ? kPStages - 1 : ip - 1;
          if (ip == kPStages - 1) pp ^= 1u;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(p_full + 8 * ip, pp) && globaltimer_ns() - t0 < kPfWaitNs) {}
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = (FMT == FMT_MX && p.hdr->wide) ? kIdescBF16 : kIdesc;
      uint32_t ia = 0, pa = 0, ib = 0, pb = 0, pab = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; ok && tile < T; tile += G) {
        const bool two = 2 * (tile % mptiles) + 1 < mtiles;
        // both accumulators are free once the epilogue has read the previous tile's
        if (!(ok = pf_wait(acc_empty, pab ^ 1u, abort, p.wait_ns))) break;
        tc_fence_after();
        for (int64_t kt = 0; kt < KT; ++kt) {
          if (!(ok = pf_wait(a_full + 8 * ia, pa, abort, p.wait_ns))) break;
          if (!(ok = pf_wait(b_full + 8 * ib, pb, abort, p.wait_ns))) break;
          tc_fence_after();
          const uint64_t ad0 = desc_sw128(sA + ia * kAStageBytes);
          const uint64_t ad1 = desc_sw128(sA + ia * kAStageBytes + kABytes);
          const uint64_t bd = desc_sw128(sB + ib * kBBytes);
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk) {  // +32 bytes per 16-element k step
            const uint32_t acc = (kt > 0 || kk > 0) ? 1u : 0u;
            mma_f16(tmem, ad0 + 2 * kk, bd + 2 * kk, idesc, acc);
            if (two) mma_f16(tmem + kBN, ad1 + 2 * kk, bd + 2 * kk, idesc, acc);
          }
          mma_commit(a_empty + 8 * ia);
          mma_commit(b_empty + 8 * ib);
          if (++ia == kAStages) { ia = 0; pa ^= 1u; }
          if (++ib == kBStages) { ib = 0; pb ^= 1u; }
        }
        if (!ok) break;
        mma_commit(acc_full);
        pab ^= 1u;
      }
      if (!ok) atomicExch(p.status, 5);
      // every MMA issued has completed once this commit arrives
      mma_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kPfWaitNs) {}
    }
  } else if (warp < 2 + kDeqWarps) {
    // ------------------------------------------------------------ dequantisers
    // Warp d handles row block j = d (16 rows) of both packed row tiles: lane (g, t) holds
    // rows 16d+g and 16d+g+8 for physical k [16t, 16t+16) of the k tile (one scale each).
    const int d = warp - 2, g = lane >> 2, t = lane & 3;
    const int soff = scale_offset(FMT, d, g, t);
    // wide MXFP4 weight: the raw E8M0 bytes give exact bf16 tiles c * 2^(e - 127)
    const bool wide = FMT == FMT_MX && p.hdr->wide != 0;
    uint32_t ip = 0, pp = 0, ib = 0, pb = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; ok && tile < T; tile += G) {
      const int64_t nt = tile / mptiles;
      const int nrt = (RT - 2 * nt) >= 2 ? 2 : 1;
      for (int64_t kt = 0; kt < KT; ++kt) {
        if (!(ok = pf_wait(p_full + 8 * ip, pp, abort, p.wait_ns))) break;
        int4 cw[2];
        uint32_t sc[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (r < nrt) {
            const uint32_t tb = sP + (ip * 2 + r) * TB;
            cw[r] = ld_shared_v4(tb + d * 512 + lane * 16);
            sc[r] = ld_shared_u16(tb + soff);
          } else {
            cw[r] = make_int4(0, 0, 0, 0);
            sc[r] = 0;
          }
        }
        // convert: row g words in k order, row g+8 likewise (8 x f16x2 each)
        uint32_t og[2][8], o8[2][8];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (FMT == FMT_MX && wide) {
            // c (exact in f16) -> fp32, times the exact group scale, -> bf16 (exact: at most
            // two significant bits, >= 2^-128; 6 * 2^127 overflows to inf as in fp32)
            const float wg = e8m0_to_f32(sc[r] & 0xFFu), wg8 = e8m0_to_f32((sc[r] >> 8) & 0xFFu);
            const uint32_t words[4] = {(uint32_t)cw[r].x, (uint32_t)cw[r].y, (uint32_t)cw[r].z,
                                       (uint32_t)cw[r].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t c4[4];
              e2m1x8_to_f16x8(words[q], c4[0], c4[1], c4[2], c4[3]);
              uint32_t o4[4];
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const __half2 hc = *reinterpret_cast<const __half2*>(&c4[b]);
                const float sw = (b & 1) ? wg8 : wg;
                const __nv_bfloat162 hb =
                    __floats2bfloat162_rn(__low2float(hc) * sw, __high2float(hc) * sw);
                o4[b] = *reinterpret_cast<const uint32_t*>(&hb);
              }
              og[r][2 * q] = o4[0];
              og[r][2 * q + 1] = o4[2];
              o8[r][2 * q] = o4[1];
              o8[r][2 * q + 1] = o4[3];
            }
            continue;
          }
          const uint32_t s2 = (FMT == FMT_NV) ? e4m3x2_to_f16x2(sc[r]) : mxenc2_to_f16x2(sc[r]);
          const __half2 sh = *reinterpret_cast<const __half2*>(&s2);
          const __half2 sg = __low2half2(sh), sg8 = __high2half2(sh);
          const uint32_t words[4] = {(uint32_t)cw[r].x, (uint32_t)cw[r].y, (uint32_t)cw[r].z,
                                     (uint32_t)cw[r].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t r0, r1, r2, r3;
            e2m1x8_to_f16x8(words[q], r0, r1, r2, r3);
            __half2 h0 = __hmul2(*reinterpret_cast<__half2*>(&r0), sg);
            __half2 h1 = __hmul2(*reinterpret_cast<__half2*>(&r1), sg8);
            __half2 h2 = __hmul2(*reinterpret_cast<__half2*>(&r2), sg);
            __half2 h3 = __hmul2(*reinterpret_cast<__half2*>(&r3), sg8);
            og[r][2 * q] = *reinterpret_cast<uint32_t*>(&h0);
            og[r][2 * q + 1] = *reinterpret_cast<uint32_t*>(&h2);
            o8[r][2 * q] = *reinterpret_cast<uint32_t*>(&h1);
            o8[r][2 * q + 1] = *reinterpret_cast<uint32_t*>(&h3);
          }
        }
        // The packed stage is released only now that every lane has used the values it
        // loaded: an arrive right after issuing the shared-memory loads let the next copy
        // into the stage overwrite data some loads had not read yet (one warp's 32 weight
        // rows of a k tile wrong, seen with MXFP4 tiles when a CTA ran many tiles).
        __syncwarp();
        if (lane == 0) mbar_arrive(p_empty + 8 * ip);
        if (++ip == kPStages) { ip = 0; pp ^= 1u; }
        if (!(ok = pf_wait(b_empty + 8 * ib, pb ^ 1u, abort, p.wait_ns))) break;
        const uint32_t bt = sB + ib * kBBytes;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (r < nrt) {
            const int row = r * 128 + 16 * d + g;  // row & 7 == g, and (row + 8) & 7 == g
            const uint32_t c0 = (uint32_t)(((2 * t) ^ g) << 4), c1 = (uint32_t)(((2 * t + 1) ^ g) << 4);
            const uint32_t rg = bt + row * 128, r8 = bt + (row + 8) * 128;
            st_shared_v4(rg + c0, og[r][0], og[r][1], og[r][2], og[r][3]);
            st_shared_v4(rg + c1, og[r][4], og[r][5], og[r][6], og[r][7]);
            st_shared_v4(r8 + c0, o8[r][0], o8[r][1], o8[r][2], o8[r][3]);
            st_shared_v4(r8 + c1, o8[r][4], o8[r][5], o8[r][6], o8[r][7]);
          }
        }
        fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(b_full + 8 * ib);
        if (++ib == kBStages) { ib = 0; pb ^= 1u; }
      }
    }
    if (!ok && lane == 0) atomicExch(p.status, 5);
  } else {
    // ------------------------------------------------------------ epilogue
    const int qd = warp & 3;  // TMEM lane quarter this warp may access
    const float f0 = p.hdr->factor[0], f1 = p.hdr->factor[1];
    uint32_t pab = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; ok && tile < T; tile += G) {
      const int64_t nt = tile / mptiles, mp = tile % mptiles;
      if (!(ok = pf_wait(acc_full, pab, abort, p.wait_ns))) break;
      tc_fence_after();
      for (int h = 0; h < kPair; ++h) {  // the tile's two token tiles, accumulator h
      const int64_t mt = 2 * mp + h;
      if (mt >= mtiles) break;  // warp-uniform
      const uint32_t ab = (uint32_t)h;
      const int64_t m = mt * kBM + qd * 32 + lane;
      const bool live = m < p.M;
      const float rs = live ? p.rowscale[m] : 0.0f;
      __nv_bfloat16* crow = p.C + (live ? m : 0) * p.ldc;
      if (p.silu) {
        // paired tiles: in each 128-column half, columns [0, 64) are gate rows 64r + j and
        // [64, 128) the matching up rows; chunk c (32 columns) pairs with chunk c + 2
        for (int c = 0; c < kBN / 32; ++c) {
          if (c & 2) continue;
          const int64_t i0 = (nt * 2 + (c >> 2)) * 64 + (c & 1) * 32;  // first output column
          if (i0 >= p.seg_split) continue;  // warp-uniform
          uint32_t vg[32], vu[32];
          tmem_ld32(tmem + ab * kBN + c * 32 + ((uint32_t)(qd * 32) << 16), vg);
          tmem_ld32(tmem + ab * kBN + (c + 2) * 32 + ((uint32_t)(qd * 32) << 16), vu);
          if (!live) continue;
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float ya = silu_f(__uint_as_float(vg[2 * e]) * rs * f0) *
                             (__uint_as_float(vu[2 * e]) * rs * f1);
            const float yb = silu_f(__uint_as_float(vg[2 * e + 1]) * rs * f0) *
                             (__uint_as_float(vu[2 * e + 1]) * rs * f1);
            __nv_bfloat162 h = __floats2bfloat162_rn(ya, yb);
            o[e] = *reinterpret_cast<uint32_t*>(&h);
          }
          if (p.vec_store && i0 + 32 <= p.seg_split) {
            uint4* dst = reinterpret_cast<uint4*>(crow + i0);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int64_t i = i0 + 2 * e;
              if (p.pair_store && i + 1 < p.seg_split) {
                *reinterpret_cast<uint32_t*>(crow + i) = o[e];
              } else {
                if (i < p.seg_split) *reinterpret_cast<uint16_t*>(crow + i) = (uint16_t)(o[e] & 0xFFFFu);
                if (i + 1 < p.seg_split) *reinterpret_cast<uint16_t*>(crow + i + 1) = (uint16_t)(o[e] >> 16);
              }
            }
          }
        }
      }
      if (!p.silu && p.layout != kLayoutPaired && p.vec_store) {
        // Plain layout with vector stores: chunk c + 1's TMEM load is in flight while chunk
        // c is scaled, rounded and stored (32 columns of this lane's token row per chunk).
        const int64_t ncol = p.N - nt * kBN;  // valid columns of the tile, > 0
        const int nch = ncol >= kBN ? kBN / 32 : (int)((ncol + 31) / 32);
        const uint32_t tb = tmem + ab * kBN + ((uint32_t)(qd * 32) << 16);
        auto chunk = [&](const uint32_t (&v)[32], int c) {
          if (!live) return;
          const int64_t n0 = nt * kBN + c * 32;
          uint32_t o[16];
          if (n0 + 32 <= p.seg_split || n0 >= p.seg_split) {  // one global for the chunk
            const float f = n0 < p.seg_split ? f0 : f1;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * rs * f,
                                                       __uint_as_float(v[2 * i + 1]) * rs * f);
              o[i] = *reinterpret_cast<uint32_t*>(&h);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int64_t n = n0 + 2 * i;
              const float fa = n < p.seg_split ? f0 : f1, fb = (n + 1) < p.seg_split ? f0 : f1;
              __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * rs * fa,
                                                       __uint_as_float(v[2 * i + 1]) * rs * fb);
              o[i] = *reinterpret_cast<uint32_t*>(&h);
            }
          }
          if (n0 + 32 <= p.N) {
            if (p.vec32_store) {
              st_global_v8(crow + n0, o);
              st_global_v8(crow + n0 + 16, o + 8);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(crow + n0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int64_t n = n0 + 2 * i;
              if (n + 1 < p.N) {
                *reinterpret_cast<uint32_t*>(crow + n) = o[i];
              } else if (n < p.N) {
                *reinterpret_cast<uint16_t*>(crow + n) = (uint16_t)(o[i] & 0xFFFFu);
              }
            }
          }
        };
        // Straight-line over the 8 chunks, every load issued (the columns past N are TMEM
        // of this accumulator and are not stored): an issued load's registers are written
        // asynchronously, so no branch merge or loop edge may carry them to their wait.
        uint32_t va[32], vb[32];
        tmem_ld32_issue(tb, va);
#pragma unroll
        for (int c = 0; c < kBN / 32; c += 2) {
          tmem_ld_wait(va);
          tmem_ld32_issue(tb + (uint32_t)(c + 1) * 32, vb);
          if (c < nch) chunk(va, c);
          tmem_ld_wait(vb);
          if (c + 2 < kBN / 32) tmem_ld32_issue(tb + (uint32_t)(c + 2) * 32, va);
          if (c + 1 < nch) chunk(vb, c + 1);
        }
      } else
      for (int c = 0; c < (p.silu ? 0 : kBN / 32); ++c) {
        const int64_t n0 = nt * kBN + c * 32;
        // warp-uniform; paired tiles map columns past N onto valid up rows, so they check
        // each column instead
        if (p.layout != kLayoutPaired && n0 >= p.N) break;
        uint32_t v[32];
        tmem_ld32(tmem + ab * kBN + c * 32 + ((uint32_t)(qd * 32) << 16), v);
        if (!live) continue;
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t n = n0 + 2 * i;
          const float fa = n < p.seg_split ? f0 : f1, fb = (n + 1) < p.seg_split ? f0 : f1;
          const float ya = __uint_as_float(v[2 * i]) * rs * fa;
          const float yb = __uint_as_float(v[2 * i + 1]) * rs * fb;
          __nv_bfloat162 h = __floats2bfloat162_rn(ya, yb);
          o[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        if (p.layout == kLayoutPaired) {
          // each column is mapped to its weight row (gate-over-up order), one at a time
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int64_t n = packed_to_row(p.layout, n0 + e, p.N, p.seg_split);
            if (n >= 0) {
              const float f = n < p.seg_split ? f0 : f1;
              crow[n] = __float2bfloat16_rn(__uint_as_float(v[e]) * rs * f);
            }
          }
        } else if (p.vec_store && n0 + 32 <= p.N) {
          uint4* dst = reinterpret_cast<uint4*>(crow + n0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int64_t n = n0 + 2 * i;
            if (p.pair_store && n + 1 < p.N) {
              *reinterpret_cast<uint32_t*>(crow + n) = o[i];
            } else {
              if (n < p.N) *reinterpret_cast<uint16_t*>(crow + n) = (uint16_t)(o[i] & 0xFFFFu);
              if (n + 1 < p.N) *reinterpret_cast<uint16_t*>(crow + n + 1) = (uint16_t)(o[i] >> 16);
            }
          }
        }
      }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      pab ^= 1u;
    }
    if (!ok && lane == 0) atomicExch(p.status, 5);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------- activation pre-pass
// A[m][k] (bf16) -> A'[m][k] = A * 2^-p (f16), p = (exponent of the row's largest
// magnitude) - 14, clamped to [-120, 113]; rowscale[m] = 2^p.  One CTA per token row.  For
// a wide MXFP4 weight (bf16 tiles) A' is A itself (bf16) and rowscale 1.
constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads) k_prep_rows(const __nv_bfloat16* __restrict__ A,
                                                           int64_t lda, int64_t K, int64_t ldp,
                                                           __half* __restrict__ Ap,
                                                           float* __restrict__ rowscale,
                                                           const PackedHeader* __restrict__ hdr) {
  __shared__ int s_max[kRowThreads / 32];
  const int64_t m = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(A + m * lda);
  const int64_t ng = K / 8;
  if (hdr->fmt == FMT_MX && hdr->wide) {
    uint4* dst = reinterpret_cast<uint4*>(Ap + m * ldp);
    for (int64_t i = threadIdx.x; i < ng; i += kRowThreads) dst[i] = __ldg(row + i);
    if (threadIdx.x == 0) rowscale[m] = 1.0f;
    return;
  }
  int mx = 0;
  for (int64_t i = threadIdx.x; i < ng; i += kRowThreads) {
    const uint4 v = __ldg(row + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    mx = max(mx, act_maxmag8(w));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0;
#pragma unroll
  for (int i = 0; i < kRowThreads / 32; ++i) mx = max(mx, s_max[i]);
  const int p = act_pow2(mx);
  uint4* dst = reinterpret_cast<uint4*>(Ap + m * ldp);
  for (int64_t i = threadIdx.x; i < ng; i += kRowThreads) {
    const uint4 v = __ldg(row + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    dst[i] = act_granule_f16(w, p);
  }
  if (threadIdx.x == 0) rowscale[m] = ldexpf(1.0f, p);
}

// W4A4: the activations quantised to the weight's block format (fp32 decisions, actq.cuh)
// and written as their exact dequantised values: NVFP4 A' = c * s, rowscale = alpha; MXFP4
// A' = c * 2^(e - p), p = (the row's largest group exponent) - 12, at least -126,
// rowscale = 2^p; for a wide MXFP4 weight (bf16 tiles) A' = c * 2^e in bf16, rowscale 1.
// One CTA per token row, one group per thread; a group holding an inf or NaN is written as
// NaN.
template <int FMT>
__global__ void __launch_bounds__(kRowThreads) k_prep_rows4(const __nv_bfloat16* __restrict__ A,
                                                            int64_t lda, int64_t K, int64_t ldp,
                                                            __half* __restrict__ Ap,
                                                            float* __restrict__ rowscale,
                                                            float alpha, float alpha6,
                                                            const PackedHeader* __restrict__ hdr) {
  constexpr int G = FMT == FMT_NV ? 16 : 32, NG = G / 8;
  const int64_t m = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(A + m * lda);
  const int64_t ngr = K / G;
  int p = 0;
  if (FMT == FMT_MX && hdr->wide) {
    uint4* dst = reinterpret_cast<uint4*>(Ap + m * ldp);
    for (int64_t grp = threadIdx.x; grp < ngr; grp += kRowThreads) {
      uint32_t w[NG][4];
      int mg = 0;
#pragma unroll
      for (int v = 0; v < NG; ++v) {
        const uint4 x = __ldg(row + grp * NG + v);
        w[v][0] = x.x;
        w[v][1] = x.y;
        w[v][2] = x.z;
        w[v][3] = x.w;
        mg = max(mg, act_maxmag8(w[v]));
      }
      const bool bad = mg >= 0x7F80;
      const int e = aq_mx_exp(__uint_as_float((uint32_t)(bad ? 0 : mg) << 16));
#pragma unroll
      for (int v = 0; v < NG; ++v) dst[grp * NG + v] = aq_mx_granule_bf16(w[v], e, bad);
    }
    if (threadIdx.x == 0) rowscale[m] = 1.0f;
    return;
  }
  if constexpr (FMT == FMT_MX) {
    __shared__ int s_max[kRowThreads / 32];
    int mx = 0;
    for (int64_t i = threadIdx.x; i < K / 8; i += kRowThreads) {
      const uint4 v = __ldg(row + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      mx = max(mx, min(act_maxmag8(w), 0x7F7F));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0;
#pragma unroll
    for (int i = 0; i < kRowThreads / 32; ++i) mx = max(mx, s_max[i]);
    p = max(aq_mx_exp(__uint_as_float((uint32_t)mx << 16)) - 12, -126);
  }
  uint4* dst = reinterpret_cast<uint4*>(Ap + m * ldp);
  for (int64_t grp = threadIdx.x; grp < ngr; grp += kRowThreads) {
    uint32_t w[NG][4];
    int mg = 0;
#pragma unroll
    for (int v = 0; v < NG; ++v) {
      const uint4 x = __ldg(row + grp * NG + v);
      w[v][0] = x.x;
      w[v][1] = x.y;
      w[v][2] = x.z;
      w[v][3] = x.w;
      mg = max(mg, act_maxmag8(w[v]));
    }
    const bool bad = mg >= 0x7F80;
    const float amax = __uint_as_float((uint32_t)(bad ? 0 : mg) << 16);
    if constexpr (FMT == FMT_NV) {
      const AqNvGroup g = aq_nv_group(amax, alpha, alpha6);
#pragma unroll
      for (int v = 0; v < NG; ++v) dst[grp * NG + v] = aq_nv_granule(w[v], g, bad, nullptr);
    } else {
      const int e = aq_mx_exp(amax);
#pragma unroll
      for (int v = 0; v < NG; ++v) dst[grp * NG + v] = aq_mx_granule(w[v], e, p, bad, nullptr);
    }
  }
  if (threadIdx.x == 0) rowscale[m] = FMT == FMT_NV ? alpha : ldexpf(1.0f, p);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

template <int FMT>
cudaError_t launch_main(const CUtensorMap& tm, const PrefillParams& pp,
                        int grid, cudaStream_t s) {
  static int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int smem = prefill_smem(FMT);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(k_prefill<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    done[dev] = 1;
  }
  k_prefill<FMT><<<grid, kPfThreads, smem, s>>>(tm, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t s, int* launches, int* grid_out,
                           int64_t* tiles_out) {
  if (launches) *launches = 0;
  const int64_t Kp = L.KT * kTileK;
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  // the activation pre-pass writes A' rows [0, M) with row stride Kp
  const __nv_bfloat16* a = reinterpret_cast<const __nv_bfloat16*>(L.A);
  __half* ap = reinterpret_cast<__half*>(L.Ap);
  const PackedHeader* hdr = reinterpret_cast<const PackedHeader*>(L.packed);
  if (!L.w4a4)
    k_prep_rows<<<(unsigned)L.M, kRowThreads, 0, s>>>(a, L.lda, L.K, Kp, ap, L.rowscale, hdr);
  else if (L.fmt == FMT_NV)
    k_prep_rows4<FMT_NV><<<(unsigned)L.M, kRowThreads, 0, s>>>(a, L.lda, L.K, Kp, ap, L.rowscale,
                                                              L.alpha, 6.0f * L.alpha, hdr);
  else
    k_prep_rows4<FMT_MX><<<(unsigned)L.M, kRowThreads, 0, s>>>(a, L.lda, L.K, Kp, ap, L.rowscale,
                                                              L.alpha, 6.0f * L.alpha, hdr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // A' as a 2-D tensor {K, M}: reads past K or M return zeros
  CUtensorMap tm;
  const cuuint64_t dims[2] = {(cuuint64_t)L.K, (cuuint64_t)L.M};
  const cuuint64_t strides[1] = {(cuuint64_t)Kp * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)kBM};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, L.Ap, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  PrefillParams pp;
  pp.tiles = reinterpret_cast<const uint8_t*>(L.packed) + kHeaderBytes;
  pp.hdr = reinterpret_cast<const PackedHeader*>(L.packed);
  pp.N = L.N;
  pp.RT = L.RT;
  pp.KT = L.KT;
  pp.M = L.M;
  pp.ldc = L.ldc;
  pp.seg_split = L.seg_split;
  pp.mtiles = (L.M + kBM - 1) / kBM;
  pp.mptiles = (pp.mtiles + kPair - 1) / kPair;
  const int64_t ntiles = (L.RT + 1) / 2;
  pp.tiles_total = pp.mptiles * ntiles;
  pp.rowscale = L.rowscale;
  pp.C = reinterpret_cast<__nv_bfloat16*>(L.C);
  pp.status = L.status;
  pp.vec_store = ((uintptr_t)L.C % 16 == 0) && (L.ldc % 8 == 0);
  pp.vec32_store = ((uintptr_t)L.C % 32 == 0) && (L.ldc % 16 == 0);
  pp.pair_store = ((uintptr_t)L.C % 4 == 0) && (L.ldc % 2 == 0);
  pp.wait_ns = L.wait_ns ? L.wait_ns : 2000000000ull;
  pp.withhold = L.withhold;
  pp.layout = L.layout;
  pp.silu = L.silu;
  int64_t grid = L.grid > 0 ? L.grid : 1;
  if (grid > pp.tiles_total) grid = pp.tiles_total;
  e = (L.fmt == FMT_NV) ? launch_main<FMT_NV>(tm, pp, (int)grid, s)
                        : launch_main<FMT_MX>(tm, pp, (int)grid, s);
  if (e != cudaSuccess) return e;
  if (launches) *launches = 2;
  if (grid_out) *grid_out = (int)grid;
  if (tiles_out) *tiles_out = pp.tiles_total;
  return cudaSuccess;
}

}  // namespace vt
