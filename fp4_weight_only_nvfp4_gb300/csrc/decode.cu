// Decode GEMM (M <= 16): C[M][N] = A[M][K] . W[N][K]^T with W streamed from the packed
// tile layout.  Sources: "keep the ModelOpt NVFP4 lm_head packed" (vllm.cpp PR #263),
// "Why this row matters" (W4A16 decode is pure weight traffic); "re-verify 27B NVFP4"
// (PR #178), "Attribution" (the FP4 MLP GEMM at ~68% of the bandwidth roof is the lever);
// "MXFP4 decode-graph + gate_up FUSION" (PR #54), "Step 3" (the CTA count per SM decides the
// residual; a regrouped fp32 reduce moves bf16 ULPs, so reductions here have a fixed
// order); "re-verify 27B NVFP4" (PR #178): a split-K workspace whose spin-locks were not
// zeroed hung the GPU, so every wait here is bounded and the counters are zeroed by each
// call's pre-pass (or left at zero by the previous call's reducers).
//
// Design (GB300): one persistent CTA per SM with 16 consumer warps, one producer warp and
// one publisher warp.  Work items are (128-row tile, 64-k tile) pairs in row-tile-major
// order; CTA c owns items [c*I/G, (c+1)*I/G).  The producer thread streams the CTA's items
// through a ring of shared-memory stages with 1-D TMA bulk copies (up to KS consecutive k
// tiles of weights per copy, plus the matching activation slices and scales, unless the
// activations are resident).  Consumers dequantise in registers (E2M1 -> f16 by cvt, times
// the group scale in f16, both exact) and accumulate with m16n8k16 MMAs in fp32.  At the
// end of each row-tile segment the warps' partial sums are added in a fixed order through
// shared memory; a row tile shared by several CTAs is finished by its first contributor
// (see k_decode), which adds the others' partials in CTA order.
#include <cuda_bf16.h>

#include <type_traits>

#include "actq.cuh"
#include "common.cuh"
#include "kernels.h"

namespace vt {

constexpr int kAScaleStride = 16;   // floats per k tile in the activation-scale array
constexpr int kConsumerWarps = 16;
// Group table of the mixture-of-experts mode (ints, in the workspace): the number of
// problems P; per problem its expert, token count, first row in the gathered activations,
// and the output row of each of its (up to 16) tokens.
constexpr int kGtMaxProblems = 128;
constexpr int kGtP = 0;
constexpr int kGtExpert = 1;
constexpr int kGtCount = kGtExpert + kGtMaxProblems;
constexpr int kGtRowsum = kGtCount + kGtMaxProblems;
constexpr int kGtPair = kGtRowsum + kGtMaxProblems;
constexpr int kGtInts = kGtPair + kGtMaxProblems * 16;
static_assert(kGtInts == kGroupTableInts, "group table size differs from the workspace layout's");
constexpr int kSlotPad = 36;        // floats per token row of a warp's reduction slot
#ifndef VT_DECODE_PREFETCH
#define VT_DECODE_PREFETCH 2
#endif
constexpr int kPrefetchStages = VT_DECODE_PREFETCH;  // stages requested before the pre-pass ends
#ifndef VT_RESIDENT_PREFETCH
#define VT_RESIDENT_PREFETCH 2
#endif
constexpr int kResidentPrefetch = VT_RESIDENT_PREFETCH;  // resident mode: stages before A is in
#ifndef VT_GROUPED_PREFETCH
#define VT_GROUPED_PREFETCH 2
#endif
constexpr int kGroupedPrefetch = VT_GROUPED_PREFETCH;  // grouped mode: stages before the pre-pass ends
#ifndef VT_GROUPED_RESIDENT_PREFETCH
#define VT_GROUPED_RESIDENT_PREFETCH 2
#endif
constexpr int kGroupedResidentPrefetch = VT_GROUPED_RESIDENT_PREFETCH;  // grouped resident mode

int decode_mt(int M) { return M <= 8 ? 8 : 16; }

// Dynamic shared memory of the decode kernel: `stages` stages of `ks` k tiles (weights, M
// activation rows and the activation scales each), the consumer warps' reduction slots and
// the barriers.
size_t decode_smem_bytes(int fmt, int M, int ks, int stages, int64_t resident_kt) {
  const size_t mt = (size_t)decode_mt(M);
  const size_t stage = resident_kt ? (size_t)ks * tile_bytes(fmt)
                                   : (size_t)ks * (tile_bytes(fmt) + (size_t)M * 128 + kAScaleStride * 4);
  return (size_t)stages * stage + kConsumerWarps * mt * kSlotPad * 4 + mt * 128 * 4 +
         decode_resident_bytes(M, resident_kt) + (size_t)stages * 16 + 128;
}

bool decode_resident_ok(int M, int64_t KT, int64_t RT) {
  // measured: converting in every CTA pays off up to about 16 KB of activations (M = 1
  // at K = 8192, M = 2 at K = 4096); beyond that the pre-pass is faster
  return M >= 1 && M <= kResidentMaxM && RT <= kFixedCounterTiles &&
         (size_t)M * KT * 128 <= kResidentMaxBytes;
}

// ------------------------------------------------------------- activation pre-pass
// A[m][k] (bf16) -> A'[kt][m][64] (f16) with one power-of-two scale per (token m, 64-wide
// k tile kt): A' = A * 2^-p, ascale[kt][m] = 2^p, p chosen from the tile's largest
// magnitude so that every value lands below 2^15 (no f16 overflow) and values down to
// 2^-31 of that maximum stay exact.  The GEMM multiplies each k tile's partial sums by
// its ascale.  The 16-byte granules of each 128-byte row are stored XOR-swizzled by
// (m & 7) so that the MMA fragment reads from shared memory are free of bank conflicts.
// Grid (M, ceil(KT / 8)); 64 threads = 8 k tiles x 8 granules, one granule each.
constexpr int kPrepThreads = 64;
constexpr int kPrepTiles = 8;

// Zeroes the split-K counters of this call's decode kernel.  The pre-pass runs after the
// previous call has finished (griddepcontrol.wait) and before this call's decode kernel
// counts, so the counters start at zero even when one workspace serves weights of other
// shapes, whose activation and partial-sum regions overlap this weight's counters.
__device__ __forceinline__ void zero_counters(int* counters, int64_t n) {
  const int64_t nb = (int64_t)gridDim.x * gridDim.y;
  const int64_t b = (int64_t)blockIdx.y * gridDim.x + blockIdx.x;
  for (int64_t i = b * blockDim.x + threadIdx.x; i < n; i += nb * blockDim.x) counters[i] = 0;
}

__global__ void __launch_bounds__(kPrepThreads) k_prep_a(const __nv_bfloat16* __restrict__ A,
                                                         int64_t lda, int64_t K, int64_t KT,
                                                         int rows, __half* __restrict__ Ap,
                                                         float* __restrict__ ascale,
                                                         int* __restrict__ counters,
                                                         int64_t ncounters) {
  // Let the GEMM kernel launch (it starts streaming weights), then wait for whatever
  // produced A (and for the previous GEMM, which may still read the workspace).
  pdl_launch_dependents();
  pdl_wait();
  zero_counters(counters, ncounters);
  const int m = blockIdx.x;
  const int64_t kt = (int64_t)blockIdx.y * kPrepTiles + (threadIdx.x >> 3);
  const int gi = threadIdx.x & 7;
  const int64_t k0 = kt * 64 + gi * 8;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (kt < KT && k0 < K) v = __ldg(reinterpret_cast<const uint4*>(A + m * lda + k0));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  int mx = act_maxmag8(w);
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (kt >= KT) return;
  const int p = act_pow2(mx);
  *reinterpret_cast<uint4*>(Ap + ((kt * rows + m) * 64 + ((gi ^ (m & 7)) * 8))) =
      act_granule_f16(w, p);
  if (gi == 0) ascale[kt * kAScaleStride + m] = pow2f(p);
}

// W4A4: the same pre-pass with the activations quantised to the weight's block format
// (fp32 decisions, actq.cuh) and written as their exact dequantised values: NVFP4 c * s with
// ascale = alpha; MXFP4 c * 2^(e - p) with p = (largest group exponent of the k tile) - 12,
// at least -126, and ascale = 2^p.  A group holding an inf or NaN is written as NaN.
template <int FMT>
__global__ void __launch_bounds__(kPrepThreads) k_prep_a4(const __nv_bfloat16* __restrict__ A,
                                                          int64_t lda, int64_t K, int64_t KT,
                                                          int rows, __half* __restrict__ Ap,
                                                          float* __restrict__ ascale,
                                                          float alpha, float alpha6,
                                                          int* __restrict__ counters,
                                                          int64_t ncounters) {
  pdl_launch_dependents();
  pdl_wait();
  zero_counters(counters, ncounters);
  const int m = blockIdx.x;
  const int64_t kt = (int64_t)blockIdx.y * kPrepTiles + (threadIdx.x >> 3);
  const int gi = threadIdx.x & 7;
  const int64_t k0 = kt * 64 + gi * 8;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (kt < KT && k0 < K) v = __ldg(reinterpret_cast<const uint4*>(A + m * lda + k0));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  // the group's largest magnitude: 2 granules (NVFP4) or 4 (MXFP4) in adjacent lanes
  int mg = act_maxmag8(w);
  mg = max(mg, __shfl_xor_sync(0xffffffffu, mg, 1));
  if constexpr (FMT == FMT_MX) mg = max(mg, __shfl_xor_sync(0xffffffffu, mg, 2));
  const int mt = max(min(mg, 0x7F7F), __shfl_xor_sync(0xffffffffu, min(mg, 0x7F7F), 4));
  if (kt >= KT) return;
  const bool bad = mg >= 0x7F80;
  const float amax = __uint_as_float((uint32_t)(bad ? 0 : mg) << 16);
  uint4 o;
  float sc;
  if constexpr (FMT == FMT_NV) {
    o = aq_nv_granule(w, aq_nv_group(amax, alpha, alpha6), bad, nullptr);
    sc = alpha;
  } else {
    const int et = aq_mx_exp(__uint_as_float((uint32_t)mt << 16));
    const int p = max(et - 12, -126);
    o = aq_mx_granule(w, aq_mx_exp(amax), p, bad, nullptr);
    sc = pow2f(p);
  }
  *reinterpret_cast<uint4*>(Ap + ((kt * rows + m) * 64 + ((gi ^ (m & 7)) * 8))) = o;
  if (gi == 0) ascale[kt * kAScaleStride + m] = sc;
}

// ------------------------------------------------------------------- main kernel
struct DecodeParams {
  const uint8_t* tiles;
  const PackedHeader* hdr;
  int64_t N, KT, items, seg_split, ldc;
  int M, stages;
  const __half* Ap;
  const float* ascale;  // [KT][16]
  __nv_bfloat16* C;
  float* partials;
  int* counters;
  int* status;
  uint64_t wait_ns;  // limit of every bounded wait
  int withhold;      // test hook: issue no copies (the waits then run out)
  // greedy head (g_idx != nullptr): no output is written; per token the largest bf16
  // output and its lowest index are kept as one 64-bit key, then written to g_idx/g_val
  int32_t* g_idx;
  float* g_val;
  unsigned long long* g_keys;  // [16], zero between calls
  unsigned int* g_done;        // CTAs finished, zero between calls
  uint32_t layout;             // packed row order (kLayoutRows / kLayoutPaired)
  int silu;                    // paired gate_up: write silu(gate) * up, C is [M][I]
  // grouped (mixture-of-experts) mode: problems = experts in use, from the pre-pass
  const int* gtab;             // group table (see kGt*)
  const __nv_bfloat16* A;      // resident mode: the bf16 activations [M][lda]
  int64_t lda, K;
  const uint8_t* gbase;        // expert e's packed weight at gbase + e * expert_bytes
  int64_t expert_bytes, RT;    // bytes per expert; 128-row tiles per expert
  const int32_t* topk_ids;     // grouped mode: the routing, grouped again by the kernel itself
  int npairs, E;
  int Mtok, topk;              // grouped resident mode: tokens of A, slots per token
};

// SiLU(x) = x / (1 + e^-x) in fp32 (e^-x overflowing to infinity gives -0 for large -x).
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// Greedy key of output value h at index n: larger value -> larger key; equal values ->
// the lower index gives the larger key (ties to the lowest index, "re-verify 27B NVFP4",
// "Correctness -- resolved, not fixed"); -0 equals +0; NaN above every number.  A max over
// keys is order-independent, so CTAs may combine them with atomicMax in any order.  Key 0
// means "no candidate".
__device__ __forceinline__ unsigned long long greedy_key(__nv_bfloat16 h, int64_t n) {
  const float v = __bfloat162float(h);
  uint32_t k;
  if (v != v) {
    k = 0xFFFFFFFFu;
  } else {
    const uint32_t b = (v == 0.0f) ? 0u : __float_as_uint(v);
    k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  return ((unsigned long long)k << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)n);
}

__device__ __forceinline__ float greedy_value(unsigned long long key) {
  const uint32_t k = (uint32_t)(key >> 32);
  if (k == 0xFFFFFFFFu) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Warp-wide max of the lanes' keys (all 32 lanes take part); lane 0 folds it into the
// CTA's key of token m in shared memory (keys of one warp always belong to one token m).
// The 64-bit max is taken as two 32-bit warp reductions: the largest high word, then the
// largest low word among the lanes that hold it.
__device__ __forceinline__ void greedy_fold(unsigned long long key, unsigned long long* keys,
                                            int m) {
  const uint32_t hi = (uint32_t)(key >> 32), lo = (uint32_t)key;
  const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
  key = ((unsigned long long)mhi << 32) | mlo;
  if ((threadIdx.x & 31) == 0 && key) atomicMax(keys + m, key);  // shared-memory atomic
}

__device__ __forceinline__ int64_t owner_of(int64_t i, int64_t I, int64_t G) {
  return ((i + 1) * G - 1) / I;  // the CTA c with c*I/G <= i < (c+1)*I/G
}

// Arrival on a grid-wide counter: one atomic add with acquire-release semantics at GPU
// scope.  Preceded by a CTA barrier, it publishes every write the CTA made before the
// barrier, and the CTA that sees the final count also sees every other CTA's writes.
__device__ __forceinline__ unsigned int arrive_acq_rel(unsigned int* ctr) {
  unsigned int prev;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(prev) : "l"(ctr) : "memory");
  return prev;
}

// Publication of a partial sum: a release add at GPU scope (the writes it publishes reach
// this thread through a CTA-scope barrier first); the issuing thread does not wait for it.
__device__ __forceinline__ void publish_release(unsigned int* ctr) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* ctr) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
  return v;
}

// Bounded wait until *ctr == target (acquire); false once `limit_ns` of wall time passed.
__device__ __forceinline__ bool wait_count(const unsigned int* ctr, unsigned int target,
                                           uint64_t limit_ns) {
  if (ld_acquire_gpu(ctr) == target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(100);
    if (ld_acquire_gpu(ctr) == target) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- routing grouping
// Mixture-of-experts decode groups the (token m, slot j) pairs of topk_ids[M][topk] into
// problems, one per expert in use, in increasing expert order, with each problem's pairs in
// increasing pair order (m * topk + j), so that the grouping, and every output bit, does not
// depend on the routing's order.  The first 128 threads of a block compute it, one pair per
// thread: a rank sort of the keys (expert << 8 | pair; an id outside [0, E) sorts last),
// then scans for each pair's problem, its slot in the problem and the problem's first row.
// A pair at slot >= cap (the decode kernel's token tile; only a token naming one expert
// several times can get there, since M <= cap) is not kept.  Both the activation pre-pass
// and the grouped decode kernel compute it, from the same ids, to the same result.
constexpr int kGroupThreads = 128;  // one pair per thread: M * topk <= 128

// Barrier over the block's first 128 threads: named barrier BAR (0 = the whole block, when it
// has exactly 128 threads).
template <int BAR>
__device__ __forceinline__ void group_sync() {
  asm volatile("bar.sync %0, 128;" ::"n"(BAR) : "memory");
}

// Inclusive scan (sum or max) over the 128 threads' values.
template <int BAR, bool MAX>
__device__ __forceinline__ int group_scan(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = MAX ? max(v, u) : v + u;
  }
  if (lane == 31) s_warp[w] = v;
  group_sync<BAR>();
  for (int q = 0; q < w; ++q) v = MAX ? max(v, s_warp[q]) : v + s_warp[q];
  group_sync<BAR>();
  return v;
}

__device__ __forceinline__ uint32_t pair_key(int e, int i, int E) {
  return (e >= 0 && e < E) ? (((uint32_t)e << 8) | (uint32_t)i) : 0xFFFFFFFFu;
}

// Thread t's result describes sorted position t: its pair, expert, problem, slot, whether it
// is kept, heads its problem (then rsum = the problem's first row) or is its problem's last
// kept pair; prob + 1 at t = 127 is the number of problems.
struct PairPlace {
  int e, pair, prob, slot, rsum;
  bool valid, kept, head, last;
};

// Threads at positions >= n hold the invalid key: only the first n keys need comparing (an
// invalid key at position j >= n sorts after every key before it and before the others).
template <int BAR>
__device__ __forceinline__ PairPlace group_pairs(uint32_t key, int n, int cap, uint32_t* s_in,
                                                 uint32_t* s_key, int* s_warp) {
  const int tid = threadIdx.x;
  s_in[tid] = key;
  group_sync<BAR>();
  int rank = tid < n ? 0 : tid - n;  // smaller keys, ties (the invalid ones) broken by position
#pragma unroll 4
  for (int j = 0; j < n; ++j) {
    const uint32_t x = s_in[j];
    rank += (x < key) | ((x == key) & (j < tid));
  }
  s_key[rank] = key;
  group_sync<BAR>();
  PairPlace q;
  key = s_key[tid];
  q.valid = key != 0xFFFFFFFFu;
  q.e = (int)(key >> 8);
  q.pair = (int)(key & 0xFFu);
  q.head = q.valid && (tid == 0 || (s_key[tid - 1] >> 8) != key >> 8);
  const int first = group_scan<BAR, true>(q.head ? tid : 0, s_warp);
  q.slot = tid - first;
  q.kept = q.valid && q.slot < cap;
  // problems so far (low half) and kept pairs so far (high half) in one scan
  const int cnt = group_scan<BAR, false>((q.head ? 1 : 0) | (q.kept ? 1 << 16 : 0), s_warp);
  q.prob = (cnt & 0xFFFF) - 1;
  q.rsum = (cnt >> 16) - 1;  // kept pairs before this one
  q.last = q.kept && (tid + 1 == kGroupThreads || !(s_key[tid + 1] != 0xFFFFFFFFu &&
                                                   (s_key[tid + 1] >> 8) == key >> 8 &&
                                                   q.slot + 1 < cap));
  return q;
}

// CTA layout: 16 consumer warps, one producer warp and one publisher warp.  A stage holds
// up to KS consecutive k tiles of one 128-row tile (one TMA bulk copy of the weights, one
// of the matching activation slices, one of their scales); consumer warp w owns the
// row-block pair w % 4 (32 rows) and the stage's k tiles w / 4, w / 4 + 4, ... .  The
// producer is one thread.
//
// Row tiles shared by several CTAs (stream-K): the tile's first contributor c_lo -- for
// which the tile is its last segment -- reduces it; every later contributor meets the tile
// as its first segment, writes its partial sums, and the publisher warp announces them with
// a release add on the tile's counter, so that no consumer waits on a global round trip in
// the middle of a call.  c_lo waits (bounded) for the count, adds the partials in
// contributor order to its own and resets the counter for the next call.  When exactly one
// later CTA shares the tile, c_lo's publisher warp does that wait while c_lo's consumers
// still stream and copies the partial into shared memory, so the reduction at the end of
// the call makes no global round trip.
//
// Resident mode (RA, small M * K): the kernel converts the whole activation matrix into
// shared memory itself after griddepcontrol.wait (no pre-pass kernel), the stages carry
// weights only, and the producer fills the whole ring at once, since no activation copy
// can queue behind the weights.  The split-K counters then rely on being left at zero by
// the previous call (each reducer resets its counter; the workspace keeps the counters in a
// fixed region that no other data of any weight overlaps).
template <int FMT, int MT, int KS, bool GRP, bool RA, bool EPI>
__global__ void __launch_bounds__(kConsumerWarps * 32 + 64, 1) k_decode(const DecodeParams p) {
  constexpr int TB = tile_bytes(FMT);
  constexpr int NJ = MT / 8;           // n8 MMA column blocks
  constexpr int CW = kConsumerWarps;
  constexpr int CT = CW * 32;          // consumer threads
  constexpr int SLOT = MT * kSlotPad;  // floats per warp reduction slot (32 rows + pad)
  constexpr int WBYTES = KS * TB;      // weight bytes of a full stage
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_flag, s_ncon, s_pre;
  __shared__ unsigned long long s_gkey[16];  // greedy head: this CTA's best key per token
  __shared__ int64_t s_clo;
  // The next kernel in the stream may launch now: it only waits (griddepcontrol.wait)
  // for this grid to finish before it touches anything this grid reads or writes.
  pdl_launch_dependents();

  // Grouped mode: the weights to stream depend on the routing, so the block's first 128
  // threads group the pairs first, from topk_ids (complete: the pre-pass lets this kernel
  // launch only after its own wait), as the pre-pass does; the producer can then request
  // weights while the pre-pass still converts the activations.
  __shared__ uint32_t s_rin[GRP ? kGroupThreads : 1], s_rkey[GRP ? kGroupThreads : 1];
  __shared__ int s_rwarp[4], s_rP;
  __shared__ int s_rexp[GRP ? kGtMaxProblems : 1], s_rcnt[GRP ? kGtMaxProblems : 1];
  __shared__ int s_rrsum[GRP ? kGtMaxProblems : 1];
  __shared__ int s_rfirst[GRP ? kGtMaxProblems : 1];  // a problem's first sorted position
  if constexpr (GRP) {
    if (threadIdx.x < kGroupThreads) {
      // Without a pre-pass (grouped resident mode) nothing has waited for the kernel that
      // may have written topk_ids: wait here, before reading them.
      if constexpr (RA) pdl_wait();
      const int tid = threadIdx.x;
      const uint32_t key = tid < p.npairs ? pair_key(__ldcg(p.topk_ids + tid), tid, p.E) : 0xFFFFFFFFu;
      const PairPlace q = group_pairs<2>(key, p.npairs, MT, s_rin, s_rkey, s_rwarp);
      if (q.kept && q.head) {
        s_rexp[q.prob] = q.e;
        s_rrsum[q.prob] = q.rsum;
        s_rfirst[q.prob] = tid;
      }
      if (q.last) s_rcnt[q.prob] = q.slot + 1;
      if (tid == kGroupThreads - 1) s_rP = q.prob + 1;
      // the pre-pass's report, made here when there is none: an id outside [0, E), or a pair
      // beyond its expert's token tile, was skipped (status 6)
      if (RA && blockIdx.x == 0 &&
          ((tid < p.npairs && key == 0xFFFFFFFFu) || (q.valid && !q.kept)))
        atomicExch(p.status, 6);
    }
    __syncthreads();
  }
  const int S = p.stages;
  const int M = GRP ? MT : p.M;  // rows of the stage's activation area
  // stage: weights | activation slices (M rows of 128 B per k tile) | activation scales;
  // resident mode: weights only
  const int SCALES_OFF = WBYTES + KS * M * 128;
  const int STAGE = RA ? WBYTES : SCALES_OFF + KS * kAScaleStride * 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t G = gridDim.x, c = blockIdx.x, KT = p.KT;
  const int64_t I = GRP ? (int64_t)s_rP * p.RT * KT : p.items;
  const int64_t i0 = c * I / G, i1 = (c + 1) * I / G;

  float* slots = reinterpret_cast<float*>(smem + (size_t)S * STAGE);
  // the reducer's copy [MT][128] of the partial of its last tile's one later contributor
  float* pre = slots + (size_t)CW * SLOT;
  // resident mode: activations [KT][M][64] f16 (the pre-pass layout) and scales [KT][8]
  uint8_t* res = smem + (size_t)S * STAGE + (size_t)CW * SLOT * 4 + (size_t)MT * 128 * 4;
  const size_t res_bytes = RA ? decode_resident_bytes(M, KT) : 0;
  const uint32_t res_u = smem_u32(res), rscale_u = res_u + (uint32_t)(M * KT * 128);
  uint64_t* full = reinterpret_cast<uint64_t*>(res + res_bytes);
  uint64_t* empty = full + S;
  const uint32_t ring_u = smem_u32(smem), full_u = smem_u32(full), empty_u = smem_u32(empty);
  const uint32_t pub_u = smem_u32(empty + S);  // consumers -> publisher: partial written
  const uint32_t aready_u = smem_u32(empty + S + 1);  // resident mode: activations converted
  const uint32_t pre_u = smem_u32(empty + S + 2);  // publisher -> reducer: later partials in
  // EPI, per row-block group jp: the group's other three warps have written their slots
  // (gfull), the group's reducing warp has read them (gfree)
  [[maybe_unused]] const uint32_t gfull_u = smem_u32(empty + S + 3);
  [[maybe_unused]] const uint32_t gfree_u = smem_u32(empty + S + 7);

  // Stages walk the CTA's items in order; all loop state advances incrementally.
  const int kt_first = (int)(i0 % KT);
  const int KTi = (int)KT;
  auto stage_len = [&](int64_t pos, int kt) -> int {
    int n = KS;
    if (n > KTi - kt) n = KTi - kt;
    if ((int64_t)n > i1 - pos) n = (int)(i1 - pos);
    return n;
  };

  if (threadIdx.x < 16) s_gkey[threadIdx.x] = 0ull;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_u + 8 * s, 1);
      mbar_init(empty_u + 8 * s, CW);
    }
    mbar_init(pub_u, CW);
    mbar_init(aready_u, 1);
    mbar_init(pre_u, 1);
    if constexpr (EPI) {
      for (int j = 0; j < 4; ++j) {
        mbar_init(gfull_u + 8 * j, 3);
        mbar_init(gfree_u + 8 * j, 1);
      }
    }
  }
  fence_mbar_init();
  __syncthreads();

  if (warp == CW + 1) {
    // ------------------------------------------------------------- publisher
    // A CTA whose range starts inside a row tile shares that tile with the CTA before it:
    // publish this CTA's partial of it once the consumers have written it.
    if (lane == 0 && i0 < i1 && i0 % KT != 0) {
      if (mbar_wait_bounded(pub_u, 0, p.wait_ns))
        publish_release(reinterpret_cast<unsigned int*>(&p.counters[i0 / KT]));
      else
        atomicExch(p.status, 5);
    }
    // A CTA whose last segment starts a row tile that exactly one later CTA shares reduces
    // that tile, and that CTA's partial is its first segment, published early: wait for it
    // here, while the consumers still stream, copy it into shared memory and reset the
    // counter.  s_pre: 2 the partial is in `pre`, 0 the wait ran out.  (Tiles shared by more
    // CTAs end in middle CTAs that finish with this one; their reducer's consumers wait for
    // them themselves.)  The counters are the previous call's until that grid has finished:
    // wait for it first.
    const int64_t rl = i0 < i1 ? (i1 - 1) / KT : 0;
    if (i0 < i1 && rl * KT >= i0 && rl * KT + KT > i1 && owner_of(rl * KT + KT - 1, I, G) == c + 1) {
      pdl_wait();
      unsigned int* ctr = reinterpret_cast<unsigned int*>(&p.counters[rl]);
      bool got = false;
      if (lane == 0) got = wait_count(ctr, 1u, p.wait_ns);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (got) {
        (void)ld_acquire_gpu(ctr);  // every lane acquires the contributor's writes
        const int mrows = GRP ? s_rcnt[(int)(rl / p.RT)] : M;
        const float* src = p.partials + (size_t)(c + 1) * 2 * MT * 128;
        for (int i = lane; i < mrows * 128; i += 32) pre[i] = __ldcg(src + i);
        __syncwarp();
        if (lane == 0) *ctr = 0;  // the contributor has arrived: reset for the next call
      } else if (lane == 0) {
        atomicExch(p.status, 5);
      }
      __syncwarp();
      if (lane == 0) {
        s_pre = got ? 2 : 0;
        mbar_arrive(pre_u);
      }
    }
    return;
  }

  if constexpr (GRP && RA) {
    if (warp == CW) {
      // ------------------------------------------------ producer (grouped, resident)
      // weights only (the consumers convert the activations themselves): the first stages
      // at once, the rest once the activations are in shared memory
      if (lane == 0 && !p.withhold) {
        const uint64_t pol = l2_evict_first_policy();
        int64_t pos = i0, rtl = 0;
        int kt = kt_first, issued = 0, slot = 0;
        int prob = (int)((i0 / KT) / p.RT), e = 0;
        rtl = i0 / KT - (int64_t)prob * p.RT;
        if (pos < i1) e = s_rexp[prob];
        while (pos < i1) {
          if (issued == kGroupedResidentPrefetch && !mbar_wait_bounded(aready_u, 0, p.wait_ns)) {
            atomicExch(p.status, 5);
            break;
          }
          if (issued >= S &&
              !mbar_wait_bounded(empty_u + 8 * slot, (uint32_t)((issued / S - 1) & 1), p.wait_ns)) {
            atomicExch(p.status, 5);
            break;
          }
          const int n = stage_len(pos, kt);
          mbar_expect_tx(full_u + 8 * slot, (uint32_t)(n * TB));
          bulk_g2s(ring_u + slot * STAGE,
                   p.gbase + e * p.expert_bytes + kHeaderBytes + (rtl * KT + kt) * TB,
                   (uint32_t)(n * TB), full_u + 8 * slot, pol);
          pos += n;
          kt += n;
          if (kt == KTi) {
            kt = 0;
            if (++rtl == p.RT && pos < i1) {
              rtl = 0;
              e = s_rexp[++prob];
            }
          }
          ++issued;
          if (++slot == S) slot = 0;
        }
      }
      return;
    }
  }

  if constexpr (GRP && !RA) {
    if (warp == CW) {
      // --------------------------------------------------------- producer (grouped)
      // virtual row tile rt = problem * RT + rt_l; the weights of expert e = expert[problem].
      // As in the dense producer, the first stages' weights are requested before the
      // activation pre-pass has finished and their activation copies once it has.
      if (lane == 0 && !p.withhold) {
        const uint64_t pol = l2_evict_first_policy();
        const uint64_t pol_a = l2_evict_last_policy();
        int64_t pos = i0, rt = i0 / KT;
        int kt = kt_first, slot = 0, issued = 0;
        uint32_t par = 0;
        int prob = (int)(rt / p.RT);
        int64_t rtl = rt - (int64_t)prob * p.RT;
        int e = 0, cnt = 0, rsum = 0;
        if (pos < i1) {
          e = s_rexp[prob];
          cnt = s_rcnt[prob];
          rsum = s_rrsum[prob];
        }
        // the activation slices and scales of a stage (pre-pass layout of problem pr)
        auto act_copies = [&](int sl, int n, int ktv, int pr, int cn, int rs) {
          const uint32_t dst = ring_u + sl * STAGE;
          bulk_g2s(dst + WBYTES, p.Ap + ((int64_t)rs * KT + (int64_t)ktv * cn) * 64,
                   (uint32_t)(n * cn * 128), full_u + 8 * sl, pol_a);
          bulk_g2s(dst + SCALES_OFF, p.ascale + ((int64_t)pr * KT + ktv) * kAScaleStride,
                   (uint32_t)(n * kAScaleStride * 4), full_u + 8 * sl, pol_a);
        };
        const int PF = S < kGroupedPrefetch ? S : kGroupedPrefetch;
        int pf_n[kGroupedPrefetch], pf_kt[kGroupedPrefetch], pf_pr[kGroupedPrefetch];
        int pf_cnt[kGroupedPrefetch], pf_rs[kGroupedPrefetch];
        bool waited = false;
        auto finish_prefetch = [&]() {
          pdl_wait();
          fence_proxy_async_all();
          waited = true;
          for (int s2 = 0; s2 < issued && s2 < PF; ++s2)
            act_copies(s2, pf_n[s2], pf_kt[s2], pf_pr[s2], pf_cnt[s2], pf_rs[s2]);
        };
        while (pos < i1) {
          if (!waited && issued == PF) finish_prefetch();
          if (issued >= S && !mbar_wait_bounded(empty_u + 8 * slot, par ^ 1u, p.wait_ns)) {
            atomicExch(p.status, 5);
            break;
          }
          const int n = stage_len(pos, kt);
          const uint32_t dst = ring_u + slot * STAGE;
          mbar_expect_tx(full_u + 8 * slot, (uint32_t)(n * (TB + cnt * 128 + kAScaleStride * 4)));
          bulk_g2s(dst, p.gbase + e * p.expert_bytes + kHeaderBytes + (rtl * KT + kt) * TB,
                   (uint32_t)(n * TB), full_u + 8 * slot, pol);
          if (waited) {
            act_copies(slot, n, kt, prob, cnt, rsum);
          } else {  // slot == issued here
            pf_n[issued] = n;
            pf_kt[issued] = kt;
            pf_pr[issued] = prob;
            pf_cnt[issued] = cnt;
            pf_rs[issued] = rsum;
          }
          ++issued;
          pos += n;
          kt += n;
          if (kt == KTi) {
            kt = 0;
            if (++rtl == p.RT && pos < i1) {
              rtl = 0;
              ++prob;
              e = s_rexp[prob];
              cnt = s_rcnt[prob];
              rsum = s_rrsum[prob];
            }
          }
          if (++slot == S) {
            slot = 0;
            par ^= 1u;
          }
        }
        if (!waited) finish_prefetch();
      }
      return;
    }
  }

  if (RA && warp == CW) {
    // ------------------------------------------------------------- producer (resident)
    // weights only; the first stages are requested at once, the rest once the consumers
    // have the activations (weight requests queued ahead would delay the activation loads)
    if (lane == 0 && !p.withhold) {
      const uint64_t pol = l2_evict_first_policy();
      int64_t pos = i0;
      int kt = kt_first, issued = 0, slot = 0;
      while (pos < i1) {
        if (issued == kResidentPrefetch && !mbar_wait_bounded(aready_u, 0, p.wait_ns)) {
          atomicExch(p.status, 5);
          break;
        }
        if (issued >= S &&
            !mbar_wait_bounded(empty_u + 8 * slot, (uint32_t)((issued / S - 1) & 1), p.wait_ns)) {
          atomicExch(p.status, 5);
          break;
        }
        const int n = stage_len(pos, kt);
        mbar_expect_tx(full_u + 8 * slot, (uint32_t)(n * TB));
        bulk_g2s(ring_u + slot * STAGE, p.tiles + pos * TB, (uint32_t)(n * TB), full_u + 8 * slot,
                 pol);
        pos += n;
        kt += n;
        if (kt == KTi) kt = 0;
        ++issued;
        if (++slot == S) slot = 0;
      }
    }
    return;
  }

  if (warp == CW) {
    // ------------------------------------------------------------- producer
    if (lane == 0 && !p.withhold) {
      const uint64_t pol = l2_evict_first_policy();   // weights: streamed once
      const uint64_t pol_a = l2_evict_last_policy();  // activations: re-read by every CTA
      const uint32_t per_tile = (uint32_t)(TB + M * 128 + kAScaleStride * 4);
      // The weights do not depend on the activation pre-pass: the first stages' weights are
      // requested before waiting for it.  Only a few: the consumers run at about the HBM
      // rate, so a deeper head start does not shorten the call, while every weight byte
      // queued ahead delays the first activation copies behind it.
      const int P = S < kPrefetchStages ? S : kPrefetchStages;
      int64_t pos = i0;
      int kt = kt_first, issued = 0;
      for (; issued < P && pos < i1; ++issued) {
        const int n = stage_len(pos, kt);
        mbar_expect_tx(full_u + 8 * issued, n * per_tile);
        bulk_g2s(ring_u + issued * STAGE, p.tiles + pos * TB, (uint32_t)(n * TB),
                 full_u + 8 * issued, pol);
        pos += n;
        kt += n;
        if (kt == KTi) kt = 0;
      }
      pdl_wait();
      fence_proxy_async_all();
      {
        int64_t pos2 = i0;
        int kt2 = kt_first;
        for (int s2 = 0; s2 < issued; ++s2) {
          const int n = stage_len(pos2, kt2);
          bulk_g2s(ring_u + s2 * STAGE + WBYTES, p.Ap + (int64_t)kt2 * M * 64,
                   (uint32_t)(n * M * 128), full_u + 8 * s2, pol_a);
          bulk_g2s(ring_u + s2 * STAGE + SCALES_OFF, p.ascale + (int64_t)kt2 * kAScaleStride,
                   (uint32_t)(n * kAScaleStride * 4), full_u + 8 * s2, pol_a);
          pos2 += n;
          kt2 += n;
          if (kt2 == KTi) kt2 = 0;
        }
      }
      // then whole stages; slot issued % S, reused once its previous use has been consumed
      int slot = issued % S;
      while (pos < i1) {
        if (issued >= S &&
            !mbar_wait_bounded(empty_u + 8 * slot, (uint32_t)((issued / S - 1) & 1), p.wait_ns)) {
          atomicExch(p.status, 5);
          break;
        }
        const int n = stage_len(pos, kt);
        const uint32_t dst = ring_u + slot * STAGE;
        mbar_expect_tx(full_u + 8 * slot, n * per_tile);
        bulk_g2s(dst, p.tiles + pos * TB, (uint32_t)(n * TB), full_u + 8 * slot, pol);
        bulk_g2s(dst + WBYTES, p.Ap + (int64_t)kt * M * 64, (uint32_t)(n * M * 128),
                 full_u + 8 * slot, pol_a);
        bulk_g2s(dst + SCALES_OFF, p.ascale + (int64_t)kt * kAScaleStride,
                 (uint32_t)(n * kAScaleStride * 4), full_u + 8 * slot, pol_a);
        pos += n;
        kt += n;
        if (kt == KTi) kt = 0;
        ++issued;
        if (++slot == S) slot = 0;
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  // Grouped resident mode: the grouping threads have waited already, and the block barrier
  // after the grouping orders every thread after that wait (griddepcontrol.wait makes the
  // earlier grids' memory visible to the whole grid); a second wait would only add its
  // release latency.
  if constexpr (!(GRP && RA)) pdl_wait();
  if constexpr (RA) {
    // The activation conversion of the pre-pass, done here into shared memory: A[m][k]
    // (bf16) -> A'[kt][m][64] (f16) = A * 2^-p with one power of two p per (token m, 64-wide
    // k tile kt) from the tile's largest magnitude, scales[kt][m] = 2^p; 16-byte granules
    // XOR-swizzled by (m & 7).  Eight consecutive threads hold one (m, kt) tile row; the
    // loop runs the same number of times in every warp (the shuffles need all lanes).
    // Grouped: only the call's tokens are converted; a slot reads its token's row, so the
    // tile's rows past the tokens are never read.
    const int Mrows = GRP ? p.Mtok : M;
    const int64_t total = (int64_t)Mrows * KT * 8;
    const __nv_bfloat16* A = p.A;
    // granule idx (loaded as v) converted and stored; a whole warp calls it (shuffles)
    auto put = [&](int64_t idx, uint4 v, int64_t ktr, int m) {
      const bool valid = idx < total;
      const int gi = (int)(idx & 7);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      int mx = act_maxmag8(w);
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (valid) {
        const int pe = act_pow2(mx);
        const uint4 o = act_granule_f16(w, pe);
        st_shared_v4(res_u + (uint32_t)(((ktr * M + m) * 64 + ((gi ^ (m & 7)) * 8)) * 2),
                     o.x, o.y, o.z, o.w);
        if (gi == 0) st_shared_f32(rscale_u + (uint32_t)((ktr * kResScaleStride + m) * 4), pow2f(pe));
      }
    };
    if constexpr (GRP) {
      // up to 8 tokens of up to 62 k tiles: a thread's granules are loaded together first,
      // so that their loads are in flight at once
      constexpr int CU = 4;
      for (int64_t base = 0; base < total; base += CU * CT) {
        uint4 v[CU];
        int64_t kr[CU];
        int mm[CU];
#pragma unroll
        for (int j = 0; j < CU; ++j) {
          const int64_t idx = base + j * CT + threadIdx.x;
          const int64_t r = idx >> 3;
          kr[j] = r / Mrows;
          mm[j] = (int)(r - kr[j] * Mrows);
          const int64_t k0 = kr[j] * 64 + (idx & 7) * 8;
          v[j] = make_uint4(0, 0, 0, 0);
          if (idx < total && k0 < p.K)
            v[j] = __ldg(reinterpret_cast<const uint4*>(A + mm[j] * p.lda + k0));
        }
#pragma unroll
        for (int j = 0; j < CU; ++j) put(base + j * CT + threadIdx.x, v[j], kr[j], mm[j]);
      }
    } else {
      for (int64_t base = 0; base < total; base += CT) {
        const int64_t idx = base + threadIdx.x;
        const int64_t r = idx >> 3;
        const int64_t ktr = r / Mrows;
        const int m = (int)(r - ktr * Mrows);
        const int64_t k0 = ktr * 64 + (int)(idx & 7) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (idx < total && k0 < p.K)
          v = __ldg(reinterpret_cast<const uint4*>(A + m * p.lda + k0));
        put(idx, v, ktr, m);
      }
    }
    // scales of the token columns past M (read by the fragments of absent tokens)
    for (int64_t i = threadIdx.x; i < KT * kResScaleStride; i += CT)
      if ((int)(i % kResScaleStride) >= M) st_shared_f32(rscale_u + (uint32_t)(i * 4), 0.0f);
    consumer_sync(CT);
    if (threadIdx.x == 0) mbar_arrive(aready_u);
  }
  const int jp = warp & 3, kq = warp >> 2;  // row blocks 2jp, 2jp+1; k tiles kq, kq+4
  float f0 = p.hdr->factor[0], f1 = p.hdr->factor[1];
  // wide MXFP4 weight: raw E8M0 bytes in the tiles, each group's exact scale applied in fp32
  bool wide = FMT == FMT_MX && p.hdr->wide != 0;
  // grouped mode: the current problem's token count, output rows and expert factor
  int Mc = M, gprob = -1;
  const int* grow = nullptr;
  // grouped resident mode: the problem's first sorted position; this lane's token rows
  int gfirst = 0, tok_g = 0, tok_a0 = 0, tok_a1 = 0;
  // the output row of slot m: the token itself, or (grouped) its (token, slot) pair
  auto out_row = [&](int m) -> int64_t {
    if constexpr (!GRP) return m;
    else if constexpr (RA) return (int64_t)(s_rkey[gfirst + m] & 0xFFu);
    else return (int64_t)grow[m];
  };
  const int soff = scale_offset(FMT, 2 * jp, g, t);
  float acc[2][NJ][4];
  // Greedy head, 8-token tile: the CTA-wide epilogues give thread x the outputs x + j CT
  // (j < 2, token (x + j CT) / 128) of every tile, so each thread keeps the best key of its
  // two outputs in registers across tiles and folds them into the CTA's keys once, after its
  // last tile.  (The 16-token tile folds every tile's keys at once.)
  constexpr int kEpiIters = (MT * 128 + CT - 1) / CT;
  [[maybe_unused]] unsigned long long gk_run[kEpiIters];
#pragma unroll
  for (int j = 0; j < kEpiIters; ++j) gk_run[j] = 0ull;
  auto greedy_note = [&](unsigned long long key, int j, int m) {
    if constexpr (MT == 8) gk_run[j] = key > gk_run[j] ? key : gk_run[j];
    else greedy_fold(key, s_gkey, m);
  };
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int u = 0; u < NJ; ++u)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[b][u][r] = 0.0f;

  // The stage loop, compiled twice for plain MXFP4 weights at the 8-token tile: once for the
  // narrow scale encoding and once for wide weights (WIDE), so that each copy gets its own
  // register allocation.  The grouped kernel, whose experts may differ, and the 16-token tile
  // (where two copies in one kernel cost more registers than one) decide inside one copy.
  auto consume = [&](auto wide_tag) -> bool {
  constexpr bool WIDE = decltype(wide_tag)::value;
  bool ok = true;
  int64_t pos = i0;
  int kt = kt_first, slot = 0;
  uint32_t par = 0;
  const int64_t rt_first = i0 / KT;
  int64_t rt = rt_first;  // row tile of the current segment
  [[maybe_unused]] uint32_t nfast = 0;  // EPI: group epilogues so far (every warp meets the same tiles)
  while (pos < i1) {
    const int n = stage_len(pos, kt);
    if constexpr (GRP) {
      const int pr = (int)(rt / p.RT);
      if (pr != gprob) {
        gprob = pr;
        Mc = s_rcnt[pr];
        if constexpr (RA) {
          // slot m of the problem is sorted position gfirst + m; its token is pair / topk
          gfirst = s_rfirst[pr];
          auto tok = [&](int m) { return m < Mc ? (int)((s_rkey[gfirst + m] & 0xFFu) / p.topk) : 0; };
          tok_g = tok(g);
          tok_a0 = tok(2 * t);
          tok_a1 = tok(2 * t + 1);
        } else {
          grow = p.gtab + kGtPair + pr * 16;  // written by the pre-pass (complete: waited above)
        }
        const PackedHeader* he = reinterpret_cast<const PackedHeader*>(
            p.gbase + (int64_t)s_rexp[pr] * p.expert_bytes);
        f0 = f1 = he->factor[0];
        wide = FMT == FMT_MX && he->wide != 0;
      }
    }
    if (ok) ok = mbar_wait_bounded(full_u + 8 * slot, par, p.wait_ns);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      const uint32_t sbase = ring_u + slot * STAGE;
      // one k tile of this warp's work; W: the exact path of a wide MXFP4 weight
      auto ktile = [&](int kh, auto w_tag) {
        constexpr bool W = decltype(w_tag)::value;
        const uint32_t tb = sbase + kh * TB;
        const uint32_t ab = RA ? res_u + (uint32_t)((kt + kh) * M * 128)
                               : sbase + WBYTES + kh * Mc * 128;
        // activation fragments (B operand) of token block u: token rows g (+8), physical
        // k 16t .. 16t+15
        auto load_b = [&](int u, uint32_t (&bf)[4][2]) {
          const int m = g + 8 * u;
          if (m < Mc) {
            const int r = (GRP && RA) ? tok_g : m;  // grouped resident: the slot's token row
            const uint32_t rowa = ab + r * 128;
            const int4 v0 = ld_shared_v4(rowa + (((2 * t) ^ (r & 7)) << 4));
            const int4 v1 = ld_shared_v4(rowa + (((2 * t + 1) ^ (r & 7)) << 4));
            bf[0][0] = v0.x; bf[0][1] = v0.y;
            bf[1][0] = v0.z; bf[1][1] = v0.w;
            bf[2][0] = v1.x; bf[2][1] = v1.y;
            bf[3][0] = v1.z; bf[3][1] = v1.w;
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) bf[q][0] = bf[q][1] = 0u;
          }
        };
        // activation scales of this k tile for the tokens of this lane's accumulators
        auto load_as = [&](int u, float (&a)[2]) {
          if constexpr (GRP && RA) {  // the tokens of slots 2t and 2t + 1 (8-token tile)
            const uint32_t sr = rscale_u + (uint32_t)((kt + kh) * kResScaleStride * 4);
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(a[0]) : "r"(sr + tok_a0 * 4));
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(a[1]) : "r"(sr + tok_a1 * 4));
          } else {
            const uint32_t sa =
                RA ? rscale_u + (uint32_t)(((kt + kh) * kResScaleStride + 2 * t + 8 * u) * 4)
                   : sbase + SCALES_OFF + kh * kAScaleStride * 4 + (2 * t + 8 * u) * 4;
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(a[0]), "=f"(a[1]) : "r"(sa));
          }
        };
        if constexpr (W) {
          // Exact MXFP4 over the whole E8M0 range: lane t's k lie in group t >> 1 of the
          // k tile, so one MMA takes the lanes of group 0 (the others' weights zeroed) and
          // a second those of group 1; each group's fp32 sums are multiplied by the token's
          // activation scale and then by the group's exact scale 2^(e - 127).  The weights
          // enter the MMA as the E2M1 values themselves (exact in f16).  One row block and
          // one token block at a time, to keep few registers live.
          const uint2 sc8 = ld_shared_v2(tb + kCodeBytes + jp * 64 + g * 8);
          const uint32_t gm = (t < 2) ? 0xFFFFFFFFu : 0u;
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const int j = 2 * jp + b;
            const int4 wv = ld_shared_v4(tb + j * 512 + lane * 16);
            // scale bytes: group h, row g (low byte) and row g + 8 (high byte) of block j
            const uint32_t s0 = sc8.x >> (16 * b), s1 = sc8.y >> (16 * b);
            const float fg0 = e8m0_to_f32(s0 & 0xFFu), fg80 = e8m0_to_f32((s0 >> 8) & 0xFFu);
            const float fg1 = e8m0_to_f32(s1 & 0xFFu), fg81 = e8m0_to_f32((s1 >> 8) & 0xFFu);
            const uint32_t words[4] = {(uint32_t)wv.x, (uint32_t)wv.y, (uint32_t)wv.z,
                                       (uint32_t)wv.w};
#pragma unroll
            for (int u = 0; u < NJ; ++u) {
              uint32_t bf[4][2];
              float a2[2];
              load_b(u, bf);
              load_as(u, a2);
              float t0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, t1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint32_t r0, r1, r2, r3;
                e2m1x8_to_f16x8(words[q], r0, r1, r2, r3);
                mma_f16_16816(t0, r0 & gm, r1 & gm, r2 & gm, r3 & gm, bf[q][0], bf[q][1]);
                mma_f16_16816(t1, r0 & ~gm, r1 & ~gm, r2 & ~gm, r3 & ~gm, bf[q][0], bf[q][1]);
              }
              acc[b][u][0] = fmaf(t0[0] * a2[0], fg0, acc[b][u][0]);
              acc[b][u][0] = fmaf(t1[0] * a2[0], fg1, acc[b][u][0]);
              acc[b][u][1] = fmaf(t0[1] * a2[1], fg0, acc[b][u][1]);
              acc[b][u][1] = fmaf(t1[1] * a2[1], fg1, acc[b][u][1]);
              acc[b][u][2] = fmaf(t0[2] * a2[0], fg80, acc[b][u][2]);
              acc[b][u][2] = fmaf(t1[2] * a2[0], fg81, acc[b][u][2]);
              acc[b][u][3] = fmaf(t0[3] * a2[1], fg80, acc[b][u][3]);
              acc[b][u][3] = fmaf(t1[3] * a2[1], fg81, acc[b][u][3]);
            }
          }
        } else {
          uint32_t bfr[NJ][4][2];
          float as[NJ][2];
#pragma unroll
          for (int u = 0; u < NJ; ++u) {
            load_b(u, bfr[u]);
            load_as(u, as[u]);
          }
          uint32_t sc4;
          asm volatile("ld.shared.b32 %0, [%1];" : "=r"(sc4) : "r"(tb + soff));
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const int j = 2 * jp + b;
            const int4 wv = ld_shared_v4(tb + j * 512 + lane * 16);
            const uint32_t two = b ? (sc4 >> 16) : (sc4 & 0xFFFFu);
            const uint32_t sc = (FMT == FMT_NV) ? e4m3x2_to_f16x2(two) : mxenc2_to_f16x2(two);
            const __half2 sc2 = *reinterpret_cast<const __half2*>(&sc);
            const __half2 sg = __low2half2(sc2), sg8 = __high2half2(sc2);
            const uint32_t words[4] = {(uint32_t)wv.x, (uint32_t)wv.y, (uint32_t)wv.z,
                                       (uint32_t)wv.w};
            float tmp[NJ][4];
#pragma unroll
            for (int u = 0; u < NJ; ++u)
#pragma unroll
              for (int r = 0; r < 4; ++r) tmp[u][r] = 0.0f;
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
                mma_f16_16816(tmp[u], a0, a1, a2, a3, bfr[u][q][0], bfr[u][q][1]);
            }
            // this k tile's sums back to the activations' true scale
#pragma unroll
            for (int u = 0; u < NJ; ++u) {
              acc[b][u][0] = fmaf(tmp[u][0], as[u][0], acc[b][u][0]);
              acc[b][u][1] = fmaf(tmp[u][1], as[u][1], acc[b][u][1]);
              acc[b][u][2] = fmaf(tmp[u][2], as[u][0], acc[b][u][2]);
              acc[b][u][3] = fmaf(tmp[u][3], as[u][1], acc[b][u][3]);
            }
          }
        }
      };
      if (FMT == FMT_MX && (WIDE || ((GRP || MT == 16) && wide))) {
#pragma unroll 1
        for (int kh = kq; kh < KS; kh += 4)
          if (kh < n) ktile(kh, std::true_type{});
      } else {
#pragma unroll
        for (int kh = kq; kh < KS; kh += 4)
          if (kh < n) ktile(kh, std::false_type{});
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_u + 8 * slot);
    pos += n;
    kt += n;
    if (++slot == S) {
      slot = 0;
      par ^= 1u;
    }
    if (kt == KTi) kt = 0;
    if (pos != i1 && kt != 0) continue;

    // ---- end of a row-tile segment: warp partials -> slots -> fixed-order sums.  The tile
    // is complete when it lies inside this CTA's item range; otherwise one thread finds the
    // CTAs that share it (64-bit divisions, so once per CTA, not per thread).
    const bool complete = (rt * KT >= i0) && (rt * KT + KT <= i1);
    // shared tile: this CTA reduces it when the tile starts inside its range (then it is
    // this CTA's last segment), else it contributes its first segment's partial
    const bool reducer = !complete && rt * KT >= i0;
    if (reducer && threadIdx.x == 0) {
      const int64_t c_hi = owner_of(rt * KT + KT - 1, I, G);
      s_clo = c;
      s_ncon = (int)(c_hi - c + 1);
    }
    if constexpr (EPI) {
      // the group's last reduction must have read the slots before they are rewritten
      if (nfast > 0 && ok) ok = mbar_wait_bounded(gfree_u + 8 * jp, (nfast - 1) & 1u, p.wait_ns);
    }
    float* my = slots + warp * SLOT;
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int u = 0; u < NJ; ++u) {
        const int m0 = 2 * t + 8 * u;
        const int r0 = b * 16 + g;
        my[m0 * kSlotPad + r0] = acc[b][u][0];
        my[(m0 + 1) * kSlotPad + r0] = acc[b][u][1];
        my[m0 * kSlotPad + r0 + 8] = acc[b][u][2];
        my[(m0 + 1) * kSlotPad + r0 + 8] = acc[b][u][3];
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[b][u][r] = 0.0f;
      }
    if constexpr (EPI) {
      if (complete && !p.silu && Mc <= 2) {
        // Rows 32 jp .. 32 jp + 31 of a complete tile need only the slots of the four warps
        // of row-block group jp: one of them (in turn) sums those rows once the other three
        // have written their slots, and the rest go straight on to the next tile.  The sums
        // and their order are those of the CTA-wide epilogue below.
        __syncwarp();
        if (kq != (int)(nfast & 3u)) {
          if (lane == 0) mbar_arrive(gfull_u + 8 * jp);
        } else {
          if (ok) ok = mbar_wait_bounded(gfull_u + 8 * jp, nfast & 1u, p.wait_ns);
          for (int m = 0; m < Mc; ++m) {  // one token per pass: warp-uniform m
            float sum = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) sum += slots[(q * 4 + jp) * SLOT + m * kSlotPad + lane];
            // grouped: the row within the expert, and the output row of the problem's slot m
            const int64_t prow = (GRP ? rt - (int64_t)gprob * p.RT : rt) * kTileRows + 32 * jp + lane;
            const int64_t n = packed_to_row(p.layout, prow, p.N, p.seg_split);
            if (p.g_idx) {
              unsigned long long key = 0;
              if (n >= 0) key = greedy_key(__float2bfloat16_rn(sum * (n < p.seg_split ? f0 : f1)), n);
              greedy_fold(key, s_gkey, m);
            } else if (n >= 0) {
              const float f = n < p.seg_split ? f0 : f1;
              p.C[out_row(m) * p.ldc + n] = __float2bfloat16_rn(sum * f);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(gfree_u + 8 * jp);
        }
        ++nfast;
        ++rt;
        continue;
      }
    }
    consumer_sync(CT);
    const int nout = Mc * 128;
    if (complete && p.silu) {
      // paired tile: rows j < 64 are gate rows, rows 64 + j the matching up rows
      for (int idx = threadIdx.x; idx < M * 64; idx += CT) {
        const int m = idx >> 6, j = idx & 63;
        float gs = 0.0f, us = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          gs += slots[(q * 4 + (j >> 5)) * SLOT + m * kSlotPad + (j & 31)];
          us += slots[(q * 4 + 2 + (j >> 5)) * SLOT + m * kSlotPad + (j & 31)];
        }
        const int64_t i = rt * 64 + j;
        if (i < p.seg_split)
          p.C[(int64_t)m * p.ldc + i] = __float2bfloat16_rn(silu_f(gs * f0) * (us * f1));
      }
    } else if (!reducer) {  // a reducer adds its slots when the other partials are in
      // output idx (token idx / 128, tile row idx % 128), the thread's j-th of the tile
      auto cta_out = [&](int idx, int j) {
        const int m = idx >> 7, row = idx & 127, pr = row >> 5, rr = row & 31;
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) sum += slots[(q * 4 + pr) * SLOT + m * kSlotPad + rr];
        if (complete) {
          // the weight row (and output column) this tile row holds, -1 for padding; grouped:
          // the row within the expert, and the output row of the problem's token m
          const int64_t prow = GRP ? (rt - (int64_t)gprob * p.RT) * kTileRows + row
                                   : rt * kTileRows + row;
          const int64_t n = packed_to_row(p.layout, prow, p.N, p.seg_split);
          const int64_t crow = out_row(m);
          if (p.g_idx) {  // warp-uniform: a warp's 32 outputs belong to one token
            unsigned long long key = 0;
            if (n >= 0) key = greedy_key(__float2bfloat16_rn(sum * (n < p.seg_split ? f0 : f1)), n);
            greedy_note(key, j, m);
          } else if (n >= 0) {
            const float f = n < p.seg_split ? f0 : f1;
            p.C[crow * p.ldc + n] = __float2bfloat16_rn(sum * f);
          }
        } else if (!reducer) {
          p.partials[((size_t)c * 2 * MT + m) * 128 + row] = sum;
        }
      };
      if constexpr (MT == 8) {
#pragma unroll
        for (int j = 0; j < kEpiIters; ++j) {
          const int idx = threadIdx.x + j * CT;
          if (idx >= nout) break;
          cta_out(idx, j);
        }
      } else {
        for (int idx = threadIdx.x; idx < nout; idx += CT) cta_out(idx, 0);
      }
    }
    if (!complete && !reducer) {
      // this CTA's partial of a tile reduced by an earlier CTA: hand it to the publisher
      __syncwarp();
      if (lane == 0) mbar_arrive(pub_u);
    }
    if (reducer) {
      if (threadIdx.x == 0) {
        int f = 0;
        if (s_ncon == 2) {
          // the publisher warp has the later contributor's partial (and reset the counter)
          if (mbar_wait_bounded(pre_u, 0, p.wait_ns)) f = s_pre;
        } else {
          unsigned int* ctr = reinterpret_cast<unsigned int*>(&p.counters[rt]);
          if (wait_count(ctr, (unsigned int)(s_ncon - 1), p.wait_ns)) {
            *ctr = 0;  // every contributor has arrived: reset for the next call
            f = 1;
          }
        }
        if (!f) atomicExch(p.status, 5);
        s_flag = f;
      }
      consumer_sync(CT);
      if (s_flag) {
        // this CTA's own partial (its slots, in fixed order) first, then the later
        // contributors' partials in contributor order (one: from shared memory; more:
        // loaded in batches of 8)
        const int64_t c_lo = s_clo;
        const int ncon = s_ncon;
        const bool in_smem = s_flag == 2;
        auto tile_sum = [&](int m, int row) -> float {
          const int pr = row >> 5, rr = row & 31;
          float sum = 0.0f;
#pragma unroll
          for (int q = 0; q < 4; ++q) sum += slots[(q * 4 + pr) * SLOT + m * kSlotPad + rr];
          const size_t off = (size_t)m * 128 + row;
          if (in_smem) return sum + pre[off];
          for (int b0 = 1; b0 < ncon; b0 += 8) {
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int64_t cc = c_lo + b0 + q;
              v[q] = (b0 + q < ncon) ? __ldcg(&p.partials[(size_t)cc * 2 * MT * 128 + off]) : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (b0 + q < ncon) sum += v[q];
          }
          return sum;
        };
        if (p.silu) {
          for (int idx = threadIdx.x; idx < M * 64; idx += CT) {
            const int m = idx >> 6, j = idx & 63;
            const float gs = tile_sum(m, j), us = tile_sum(m, 64 + j);
            const int64_t i = rt * 64 + j;
            if (i < p.seg_split)
              p.C[(int64_t)m * p.ldc + i] = __float2bfloat16_rn(silu_f(gs * f0) * (us * f1));
          }
        }
        auto red_out = [&](int idx, int j) {
          const int m = idx >> 7, row = idx & 127;
          const float sum = tile_sum(m, row);
          const int64_t prow = GRP ? (rt - (int64_t)gprob * p.RT) * kTileRows + row
                                   : rt * kTileRows + row;
          const int64_t n = packed_to_row(p.layout, prow, p.N, p.seg_split);
          const int64_t crow = out_row(m);
          if (p.g_idx) {
            unsigned long long key = 0;
            if (n >= 0) key = greedy_key(__float2bfloat16_rn(sum * (n < p.seg_split ? f0 : f1)), n);
            greedy_note(key, j, m);
          } else if (n >= 0) {
            const float f = n < p.seg_split ? f0 : f1;
            p.C[crow * p.ldc + n] = __float2bfloat16_rn(sum * f);
          }
        };
        const int nred = p.silu ? 0 : nout;
        if constexpr (MT == 8) {
#pragma unroll
          for (int j = 0; j < kEpiIters; ++j) {
            const int idx = threadIdx.x + j * CT;
            if (idx >= nred) break;
            red_out(idx, j);
          }
        } else {
          for (int idx = threadIdx.x; idx < nred; idx += CT) red_out(idx, 0);
        }
      }
    }
    consumer_sync(CT);  // slots are rewritten by the next segment
    ++rt;
  }
  return ok;
  };
  bool ok;
  if constexpr (FMT == FMT_MX && !GRP && MT == 8) {
    if (wide) ok = consume(std::true_type{});
    else ok = consume(std::false_type{});
  } else {
    ok = consume(std::false_type{});
  }
  if (!ok && lane == 0) atomicExch(p.status, 5);
  if (p.g_idx) {
    if constexpr (MT == 8) {
      // the running keys of the CTA-wide epilogues (warp-uniform token per j)
#pragma unroll
      for (int j = 0; j < kEpiIters; ++j) {
        const int idx = threadIdx.x + j * CT;
        if (idx < M * 128) greedy_fold(gk_run[j], s_gkey, idx >> 7);
      }
    }
    // One global atomic per token per CTA; the last CTA to finish turns the keys into
    // indices and values and clears them (and the counter) for the next call.
    consumer_sync(CT);
    if (threadIdx.x < M && s_gkey[threadIdx.x]) atomicMax(p.g_keys + threadIdx.x, s_gkey[threadIdx.x]);
    consumer_sync(CT);
    if (threadIdx.x == 0) s_flag = (arrive_acq_rel(p.g_done) == gridDim.x - 1);
    consumer_sync(CT);
    if (s_flag) {
      if (threadIdx.x < M) {
        const unsigned long long key = atomicExch(p.g_keys + threadIdx.x, 0ull);
        p.g_idx[threadIdx.x] = key ? (int32_t)(0xFFFFFFFFu - (uint32_t)key) : -1;
        if (p.g_val) p.g_val[threadIdx.x] = greedy_value(key);
      }
      if (threadIdx.x == 0) atomicExch(p.g_done, 0u);
    }
  }
}

// Raises a kernel's dynamic shared memory limit once per device (the first call on a
// device, made before any graph capture, does it).
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

template <int FMT, int MT, int KS, bool GRP = false, bool RA = false, bool EPI = false>
static cudaError_t launch_t(const DecodeLaunch& L, cudaStream_t s) {
  static int done[64] = {0};
  const size_t smem = decode_smem_bytes(FMT, GRP ? MT : L.M, KS, L.stages, RA ? L.KT : 0);
  cudaError_t e = allow_smem(k_decode<FMT, MT, KS, GRP, RA, EPI>, (int)smem, done);
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
  p.ascale = L.ascale;
  p.C = reinterpret_cast<__nv_bfloat16*>(L.C);
  p.partials = L.partials;
  p.counters = L.counters;
  p.status = L.status;
  p.wait_ns = L.wait_ns ? L.wait_ns : 2000000000ull;
  p.withhold = L.withhold;
  p.g_idx = L.g_idx;
  p.g_val = L.g_val;
  p.g_keys = L.g_keys;
  p.g_done = L.g_done;
  p.layout = L.layout;
  p.silu = L.silu;
  p.gtab = L.gtab;
  p.gbase = reinterpret_cast<const uint8_t*>(L.packed);
  p.expert_bytes = L.expert_bytes;
  p.RT = L.RT;
  p.A = reinterpret_cast<const __nv_bfloat16*>(L.A);
  p.lda = L.lda;
  p.K = L.K;
  p.topk_ids = L.topk_ids;
  p.npairs = L.npairs;
  p.E = L.E;
  p.Mtok = L.Mtok;
  p.topk = L.topk;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)L.grid);
  cfg.blockDim = dim3((unsigned)(kConsumerWarps * 32 + 64));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode<FMT, MT, KS, GRP, RA, EPI>, p);
}

// ------------------------------------------------------------- grouped pre-pass
// Mixture-of-experts decode: each (token m, slot j) pair of topk_ids[M][topk] names an
// expert.  The pairs are grouped into problems, one per expert in use, in increasing
// expert order, with each problem's tokens in increasing pair order (m * topk + j): the
// grouping, and so every output bit, is the same in every run.  Block (b, y) converts the
// activations of problem b's tokens for k tiles 8y .. 8y+7 exactly as k_prep_a does, into
// A'[rowsum_b * KT + kt * count_b + s][64] (granules XOR-swizzled by s & 7) with scales
// ascale[(b * KT + kt) * 16 + s]; block (0, 0) also writes the group table.  A pair whose
// expert id is out of range, or that would be the (cap+1)-th or later pair of its expert (the
// decode kernel's token tile holds `cap` rows; only a token naming one expert several times
// can get there, since M <= cap), sets status 6 and is left out (its output row is not
// written).
__global__ void __launch_bounds__(kGroupThreads) k_group_prep(
    const __nv_bfloat16* __restrict__ A, int64_t lda, int64_t K, int64_t KT,
    const int32_t* __restrict__ topk_ids, int npairs, int topk, int E, int cap,
    __half* __restrict__ Ap, float* __restrict__ ascale, int* __restrict__ gtab,
    int* __restrict__ status, int* __restrict__ counters, int64_t ncounters) {
  // The grouped decode kernel reads topk_ids itself as soon as it starts: it may launch only
  // once whatever wrote them has finished, that is after this wait.
  pdl_wait();
  pdl_launch_dependents();
  zero_counters(counters, ncounters);
  __shared__ uint32_t s_in[kGroupThreads], s_key[kGroupThreads];
  __shared__ int s_warp[kGroupThreads / 32];
  __shared__ int s_P, s_cnt, s_rsum, s_pair[16];
  __shared__ __align__(16) uint4 s_a[16 * kPrepTiles * 8];  // A rows' granules of this block's k tiles
  const int tid = threadIdx.x;
  const bool lead = blockIdx.x == 0 && blockIdx.y == 0;
  const int M = npairs / topk;
  // The activations of every token for this block's k tiles, requested before the grouping
  // (which token rows the block converts is known only after it).
  for (int i = tid; i < M * kPrepTiles * 8; i += kGroupThreads) {
    const int m = i / (kPrepTiles * 8), r = i - m * (kPrepTiles * 8);
    const int64_t k0 = ((int64_t)blockIdx.y * kPrepTiles + (r >> 3)) * 64 + (r & 7) * 8;
    s_a[i] = k0 < K ? __ldg(reinterpret_cast<const uint4*>(A + m * lda + k0)) : make_uint4(0, 0, 0, 0);
  }
  // the grouping (see group_pairs); an invalid id or a pair beyond its expert's token tile
  // is reported (status 6) and left out
  int id = -1;
  if (tid < npairs) id = __ldcg(topk_ids + tid);
  const uint32_t key0 = tid < npairs ? pair_key(id, tid, E) : 0xFFFFFFFFu;
  if (tid < npairs && key0 == 0xFFFFFFFFu && lead) atomicExch(status, 6);
  const PairPlace q = group_pairs<0>(key0, npairs, cap, s_in, s_key, s_warp);
  if (q.valid && !q.kept && lead) atomicExch(status, 6);
  const int prob = q.prob, slot = q.slot, pair = q.pair;
  const bool kept = q.kept, head = q.head, last = q.last;
  if (tid == kGroupThreads - 1) s_P = prob + 1;  // heads among the valid pairs
  if (lead && kept) {
    gtab[kGtPair + prob * 16 + slot] = pair;
    if (head) {
      gtab[kGtExpert + prob] = q.e;
      gtab[kGtRowsum + prob] = q.rsum;
    }
    if (last) gtab[kGtCount + prob] = slot + 1;
  }
  const int b = blockIdx.x;
  if (kept && prob == b) {
    s_pair[slot] = pair;
    if (head) s_rsum = q.rsum;
    if (last) s_cnt = slot + 1;
  }
  __syncthreads();
  const int P = s_P;
  if (lead && tid == 0) gtab[kGtP] = P;
  if (b >= P) return;
  // Convert this problem's tokens for k tiles 8y .. 8y+7 as k_prep_a does: rows
  // rowsum * KT + kt * count + s, granules XOR-swizzled by s & 7; threads 0-63 take the even
  // slots, 64-127 the odd ones.
  const int cnt = s_cnt, rsum = s_rsum;
  const int64_t kt = (int64_t)blockIdx.y * kPrepTiles + ((tid & 63) >> 3);
  const int gi = tid & 7;
  for (int sx = tid >> 6; sx < cnt; sx += 2) {
    const int m = s_pair[sx] / topk;
    const uint4 v = s_a[m * (kPrepTiles * 8) + (tid & 63)];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    int mx = act_maxmag8(w);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (kt >= KT) continue;
    const int pe = act_pow2(mx);
    *reinterpret_cast<uint4*>(Ap + ((rsum * KT + kt * cnt + sx) * 64 + ((gi ^ (sx & 7)) * 8))) =
        act_granule_f16(w, pe);
    if (gi == 0) ascale[((int64_t)b * KT + kt) * kAScaleStride + sx] = pow2f(pe);
  }
}

cudaError_t launch_decode_grouped(const DecodeLaunch& L0, const int32_t* topk_ids, int npairs,
                                  int topk, int E, cudaStream_t s, int* launches) {
  if (npairs > kGroupThreads) return cudaErrorInvalidValue;
  DecodeLaunch L = L0;
  L.topk_ids = topk_ids;
  L.npairs = npairs;
  L.E = E;
  L.topk = topk;
  L.Mtok = npairs / topk;
  cudaError_t e = cudaSuccess;
  if (L.resident) {  // one kernel: it groups the routing and converts the activations itself
    if (decode_mt(L.M) != 8) return cudaErrorInvalidValue;
    // with the per-group epilogue (EPI) for the complete tiles of problems of up to 2 slots,
    // which most problems of a few tokens over many experts are (128 experts of 1536 x 2048,
    // top-8: M = 4 18.73 -> 18.41 us, M = 8 24.57 -> 24.41 us, outputs bit-identical)
    const bool nv = L.fmt == FMT_NV;
    if (L.ks == 16)
      e = nv ? launch_t<FMT_NV, 8, 16, true, true, true>(L, s)
             : launch_t<FMT_MX, 8, 16, true, true, true>(L, s);
    else if (L.ks == 4)
      e = nv ? launch_t<FMT_NV, 8, 4, true, true>(L, s) : launch_t<FMT_MX, 8, 4, true, true>(L, s);
    else
      e = nv ? launch_t<FMT_NV, 8, 8, true, true, true>(L, s)
             : launch_t<FMT_MX, 8, 8, true, true, true>(L, s);
    if (launches) *launches = 1;
    return e;
  }
  {
    const int pmax = npairs < E ? npairs : E;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(pmax > 0 ? pmax : 1),
                       (unsigned)((L.KT + kPrepTiles - 1) / kPrepTiles));
    cfg.blockDim = dim3(kGroupThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_group_prep, reinterpret_cast<const __nv_bfloat16*>(L.A),
                           L.lda, L.K, L.KT, topk_ids, npairs, topk, E, decode_mt(L.M),
                           reinterpret_cast<__half*>(L.Ap), L.ascale, const_cast<int*>(L.gtab),
                           L.status, L.counters, (int64_t)(pmax < kGtMaxProblems ? pmax : kGtMaxProblems) * L.RT);
    if (e != cudaSuccess) return e;
  }
  // token tile: 8 rows when M <= 8 (an expert then gets at most 8 pairs; extra pairs from a
  // token naming one expert twice are skipped by the pre-pass), else 16
  const bool m8 = decode_mt(L.M) == 8;
  if (L.ks == 4)
    e = (L.fmt == FMT_NV) ? (m8 ? launch_t<FMT_NV, 8, 4, true>(L, s) : launch_t<FMT_NV, 16, 4, true>(L, s))
                          : (m8 ? launch_t<FMT_MX, 8, 4, true>(L, s) : launch_t<FMT_MX, 16, 4, true>(L, s));
  else
    e = (L.fmt == FMT_NV) ? (m8 ? launch_t<FMT_NV, 8, 8, true>(L, s) : launch_t<FMT_NV, 16, 8, true>(L, s))
                          : (m8 ? launch_t<FMT_MX, 8, 8, true>(L, s) : launch_t<FMT_MX, 16, 8, true>(L, s));
  if (launches) *launches = 2;
  return e;
}

cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t s, int* launches) {
  const int mt = decode_mt(L.M);
  cudaError_t e = cudaSuccess;
  if (L.resident) {  // one kernel: it converts the activations itself
    if (mt != 8 || L.w4a4) return cudaErrorInvalidValue;
    if (L.ks == 4)
      e = (L.fmt == FMT_NV) ? launch_t<FMT_NV, 8, 4, false, true>(L, s)
                            : launch_t<FMT_MX, 8, 4, false, true>(L, s);
    else if (L.epi)
      e = (L.fmt == FMT_NV) ? launch_t<FMT_NV, 8, 8, false, true, true>(L, s)
                            : launch_t<FMT_MX, 8, 8, false, true, true>(L, s);
    else
      e = (L.fmt == FMT_NV) ? launch_t<FMT_NV, 8, 8, false, true>(L, s)
                            : launch_t<FMT_MX, 8, 8, false, true>(L, s);
    if (launches) *launches = 1;
    return e;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)L.M, (unsigned)((L.KT + kPrepTiles - 1) / kPrepTiles));
    cfg.blockDim = dim3(kPrepThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const __nv_bfloat16* a = reinterpret_cast<const __nv_bfloat16*>(L.A);
    __half* ap = reinterpret_cast<__half*>(L.Ap);
    if (!L.w4a4)
      e = cudaLaunchKernelEx(&cfg, k_prep_a, a, L.lda, L.K, L.KT, L.M, ap, L.ascale, L.counters,
                             L.RT);
    else if (L.fmt == FMT_NV)
      e = cudaLaunchKernelEx(&cfg, k_prep_a4<FMT_NV>, a, L.lda, L.K, L.KT, L.M, ap, L.ascale,
                             L.alpha, 6.0f * L.alpha, L.counters, L.RT);
    else
      e = cudaLaunchKernelEx(&cfg, k_prep_a4<FMT_MX>, a, L.lda, L.K, L.KT, L.M, ap, L.ascale,
                             L.alpha, 6.0f * L.alpha, L.counters, L.RT);
    if (e != cudaSuccess) return e;
  }
  // stage width in k tiles (KS): 4, 8, or 16 (8-token tile only)
  if (L.ks == 16) {
    if (mt != 8) return cudaErrorInvalidValue;
    e = (L.fmt == FMT_NV) ? launch_t<FMT_NV, 8, 16>(L, s) : launch_t<FMT_MX, 8, 16>(L, s);
  } else if (L.ks == 4) {
    if (L.fmt == FMT_NV) e = (mt == 8) ? launch_t<FMT_NV, 8, 4>(L, s) : launch_t<FMT_NV, 16, 4>(L, s);
    else e = (mt == 8) ? launch_t<FMT_MX, 8, 4>(L, s) : launch_t<FMT_MX, 16, 4>(L, s);
  } else {
    if (mt == 8 && L.epi)
      e = (L.fmt == FMT_NV) ? launch_t<FMT_NV, 8, 8, false, false, true>(L, s)
                            : launch_t<FMT_MX, 8, 8, false, false, true>(L, s);
    else if (L.fmt == FMT_NV) e = (mt == 8) ? launch_t<FMT_NV, 8, 8>(L, s) : launch_t<FMT_NV, 16, 8>(L, s);
    else e = (mt == 8) ? launch_t<FMT_MX, 8, 8>(L, s) : launch_t<FMT_MX, 16, 8>(L, s);
  }
  if (launches) *launches = 2;
  return e;
}

}  // namespace vt
