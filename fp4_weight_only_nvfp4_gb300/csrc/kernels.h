// Host-side launchers implemented by the .cu files of libvtfp4 (internal header).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace vt {

cudaError_t launch_prepack(const uint8_t* const codes[2], const uint8_t* const scales[2],
                           int64_t split, float f0, float f1, int fmt, int64_t N, int64_t K,
                           int64_t RT, int64_t KT, uint32_t layout, void* dst, cudaStream_t s);
cudaError_t launch_unpack(const void* packed, int fmt, int64_t N, int64_t K, int64_t RT,
                          int64_t KT, int64_t split, uint32_t layout, uint8_t* codes,
                          uint8_t* scales, cudaStream_t s);
cudaError_t launch_dequant(const void* packed, int fmt, int64_t N, int64_t K, int64_t RT,
                           int64_t KT, int64_t split, uint32_t layout, float* out,
                           cudaStream_t s);

// Decode GEMM (M <= 16).
struct DecodeLaunch {
  const void* packed;     // header + tiles
  int fmt;
  int64_t N, K, RT, KT;
  int64_t seg_split;
  const void* A;          // bf16 [M][lda]
  int64_t lda;
  int M;
  void* C;                // bf16 [M][ldc]
  int64_t ldc;
  // workspace pieces
  int* status;
  int* counters;          // [RT]
  float* ascale;          // [KT][16] activation scale per (k tile, token)
  void* Ap;               // f16 [KT][M][64]
  float* partials;        // [grid*2][MT][128]
  // launch shape
  int grid, ks, stages;  // CTAs, k tiles per stage (4 or 8), ring depth
  uint64_t wait_ns;      // limit of every bounded wait
  int withhold;          // test hook: the producer issues no copies
  // greedy head (g_idx non-null): per-token argmax instead of the output
  int32_t* g_idx = nullptr;
  float* g_val = nullptr;
  unsigned long long* g_keys = nullptr;  // [16] in the workspace
  unsigned int* g_done = nullptr;
  uint32_t layout = 0;   // packed row order (kLayoutRows / kLayoutPaired)
  int silu = 0;          // paired gate_up: C[M][I] = silu(gate) * up
  // grouped (mixture-of-experts) mode: packed = expert 0's packed weight
  const int* gtab = nullptr;  // group table in the workspace
  int64_t expert_bytes = 0;   // bytes per expert's packed weight
  const int32_t* topk_ids = nullptr;  // the routing [npairs] (the kernel groups it again)
  int npairs = 0, E = 0;
  // W4A4: the pre-pass quantises the activations to the weight's block format (alpha:
  // NVFP4 activation global)
  int w4a4 = 0;
  float alpha = 1.0f;
  int resident = 0;  // resident-activation mode (decode_resident_ok; not with w4a4); grouped:
                    // the decode kernel groups the routing and converts A itself, no pre-pass
  int Mtok = 0, topk = 0;  // grouped resident mode: tokens of A, slots per token
  int epi = 0;  // 8 k tiles per stage, M <= 8: the per-group epilogue for complete tiles of
                // up to 2 tokens (decode_shape chooses it; the grouped one-launch mode takes
                // it at 8 and 16 k tiles per stage, for problems of up to 2 slots)
};
int decode_mt(int M);  // 8 or 16
// Resident-activation decode (small M * K): the decode kernel converts A into shared memory
// itself; no pre-pass.  The workspace keeps the split-K counters of weights with up to
// kFixedCounterTiles row tiles in a fixed 64 KB region that no other data overlaps.
constexpr int kResScaleStride = 8;               // floats per k tile of resident scales
constexpr int kResidentMaxM = 4;
constexpr size_t kResidentMaxBytes = 16 * 1024;  // of converted activations (M * K * 2)
constexpr int64_t kFixedCounterTiles = 16384;
__host__ __device__ inline size_t decode_resident_bytes(int M, int64_t KT) {
  return KT ? (size_t)M * (size_t)KT * 128 + (size_t)KT * kResScaleStride * 4 : 0;
}
bool decode_resident_ok(int M, int64_t KT, int64_t RT);
cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t s, int* launches);
// Grouped decode: a pre-pass groups the (token, slot) pairs of topk_ids [M][topk] by
// expert and converts their activations, then the decode kernel runs every problem.
cudaError_t launch_decode_grouped(const DecodeLaunch& L, const int32_t* topk_ids, int npairs,
                                  int topk, int E, cudaStream_t s, int* launches);
constexpr int kGroupTableInts = 1 + 3 * 128 + 128 * 16;  // see the decode kernel
// Grouped resident mode (M <= 8 tokens): the largest converted activation matrix a CTA keeps.
constexpr size_t kGroupedResidentMaxBytes = 64 * 1024;
size_t decode_smem_bytes(int fmt, int M, int ks, int stages, int64_t resident_kt = 0);

// Prefill tile GEMM (tensor cores), any M.
struct PrefillLaunch {
  const void* packed;
  int fmt;
  int64_t N, K, RT, KT;
  int64_t seg_split;
  const void* A;
  int64_t lda;
  int64_t M;
  void* C;
  int64_t ldc;
  int* status;
  float* rowscale;        // [Mp]
  void* Ap;               // f16 [Mp][Kp]
  int grid;
  uint64_t wait_ns;       // limit of every bounded wait
  int withhold;           // test hook: the producer issues no copies
  uint32_t layout = 0;    // packed row order (kLayoutRows / kLayoutPaired)
  int silu = 0;           // paired gate_up: C[M][I] = silu(gate) * up
  int w4a4 = 0;           // quantise the activations first (see DecodeLaunch)
  float alpha = 1.0f;
};
cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t s, int* launches, int* grid_out,
                           int64_t* tiles_out);

// Quantiser.
cudaError_t launch_quantize(const void* W, int64_t N, int64_t K, int fmt, uint8_t* codes,
                            uint8_t* scales, float* global_out, void* scratch, cudaStream_t s);
// W4A4 activation quantiser: bf16 A [M][lda] -> codes [M][K/2], scales [M][K/g].
cudaError_t launch_quantize_act(const void* A, int64_t M, int64_t lda, int64_t K, int fmt,
                                float alpha, uint8_t* codes, uint8_t* scales, cudaStream_t s);

constexpr int kMaxDecodeGrid = 512;

}  // namespace vt
