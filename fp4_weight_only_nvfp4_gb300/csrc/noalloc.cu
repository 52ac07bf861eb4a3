// vt_fp4_w4a16_gemm_noalloc: the decode GEMM for callers that cannot hand the library a
// device workspace.  Some callers cannot call cudaMalloc at all: a host program whose
// device memory is owned by someone else's allocator (a serving engine that reserves its
// HBM up front, a plugin inside a framework that forbids foreign allocations) or a call
// path that must not block on, or fail in, a runtime allocation.  This entry point uses a
// fixed scratch area that lives in this library's own device image instead of a caller
// workspace.  vt_fp4_noalloc_status reads the status word that area keeps, and
// vt_fp4_noalloc_test_hooks lets a test make its bounded waits run out.
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "handle.h"
#include "kernels.h"

namespace {

using namespace vt;

// 4 MiB of device memory, held by every GPU that loads this library until the process
// exits.  It holds the status word, the per-call split-K arrival counters, the activation
// scales, the converted activations and the split-K partial sums.
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Test hooks (vt_fp4_noalloc_test_hooks): the limit of the kernels' bounded waits and the
// weight-producer switch of vt_fp4_gemm_opts, for the calls that follow.
std::atomic<int> g_hook_wait_us{0}, g_hook_withhold{0};

inline size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// The device address of the scratch array for device `dev`, looked up once per device.
// In host code g_noalloc_scratch only names a host-side stand-in; the kernel needs the
// address the runtime reports for the current device.
cudaError_t scratch_address(int dev, void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

vt_status err(vt_status st, const char* msg) { return set_last_error(st, msg); }

vt_status cuda_err(cudaError_t e) { return err(VT_ERR_CUDA, cudaGetErrorString(e)); }

}  // namespace

extern "C" vt_status vt_fp4_w4a16_gemm_noalloc(const void* A, int64_t M, int64_t lda,
                                               vt_fp4_handle W, void* C, int64_t ldc,
                                               vt_stream_t s) {
  char msg[256];
  if (!W) return err(VT_ERR_INVALID_ARG, "weight handle is NULL");
  if (W->E > 1) return err(VT_ERR_INVALID_ARG, "a grouped weight serves vt_fp4_w4a16_gemm_moe");
  if (M < 0) return err(VT_ERR_INVALID_ARG, "M must be >= 0");
  if (M == 0) return VT_OK;
  if (M > 16) return err(VT_ERR_UNSUPPORTED, "the no-alloc GEMM serves M <= 16 only");
  if (!A || !C) return err(VT_ERR_INVALID_ARG, "A and C must be set");
  if (lda < W->K || ldc < W->N) return err(VT_ERR_INVALID_ARG, "lda must be >= K and ldc >= N");
  if (!aligned(A, 16) || lda % 8)
    return err(VT_ERR_MISALIGNED, "A must be 16-byte aligned with lda % 8 == 0");
  if (!aligned(C, 2)) return err(VT_ERR_MISALIGNED, "C must be 2-byte aligned");
  if (W->K > 110000) return err(VT_ERR_UNSUPPORTED, "K > 110000 is not supported");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_err(e);

  // launch shape: the same choice as vt_fp4_w4a16_gemm makes
  vt_fp4_gemm_opts hooks = {};
  hooks.wait_limit_us = g_hook_wait_us.load();
  hooks.withhold_weights = g_hook_withhold.load();
  DecodeShape sh;
  if (vt_status st = decode_shape(W, (int)M, nullptr, false, &sh)) return st;
  const int mt = decode_mt((int)M);

  // scratch layout: status | counters [RT] | activation scales [KT][16] | activations
  // [KT][M][64] f16 | split-K partials [grid][2][MT][128] fp32
  const size_t o_counters = 256;
  const size_t o_ascale = up256(o_counters + (size_t)W->RT * 4);
  const size_t o_ap = up256(o_ascale + (size_t)W->KT * 16 * 4);
  const size_t o_part = up256(o_ap + (size_t)W->KT * M * 128);
  const size_t need = up256(o_part + (size_t)sh.grid * 2 * mt * 128 * 4);
  if (need > kNoAllocScratchBytes) {
    snprintf(msg, sizeof(msg),
             "this weight and M need %zu bytes of scratch; the no-alloc scratch holds %zu",
             need, kNoAllocScratchBytes);
    return err(VT_ERR_UNSUPPORTED, msg);
  }
  void* base = nullptr;
  e = scratch_address(dev, &base);
  if (e != cudaSuccess) return cuda_err(e);
  uint8_t* ws = static_cast<uint8_t*>(base);
  // the arrival counters must start at zero (a call that gave up may have left counts); the
  // status word is left alone until vt_fp4_noalloc_status reads it
  e = cudaMemsetAsync(ws + o_counters, 0, o_ascale - o_counters, (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_err(e);

  DecodeLaunch D;
  D.packed = W->packed;
  D.fmt = W->fmt;
  D.N = W->N;
  D.K = W->K;
  D.RT = W->RT;
  D.KT = W->KT;
  D.seg_split = W->seg_split;
  D.A = A;
  D.lda = lda;
  D.M = (int)M;
  D.C = C;
  D.ldc = ldc;
  D.status = reinterpret_cast<int*>(ws);
  D.counters = reinterpret_cast<int*>(ws + o_counters);
  D.ascale = reinterpret_cast<float*>(ws + o_ascale);
  D.Ap = ws + o_ap;
  D.partials = reinterpret_cast<float*>(ws + o_part);
  D.grid = sh.grid;
  D.ks = sh.ks;
  D.stages = sh.stages;
  D.wait_ns = hooks.wait_limit_us > 0 ? (uint64_t)hooks.wait_limit_us * 1000ull : 0;
  D.withhold = hooks.withhold_weights;
  D.layout = (uint32_t)W->layout;
  D.resident = sh.resident;
  D.epi = sh.epi;
  int launches = 0;
  e = launch_decode(D, (cudaStream_t)s, &launches);
  if (e != cudaSuccess) return cuda_err(e);
  W->info.path = 1;
  W->info.tile_epilogue = sh.epi;
  W->info.stage_k_tiles = sh.ks;
  W->info.grid = D.grid;
  W->info.warps_per_cta = 18;
  W->info.m_tile = mt;
  W->info.items = W->RT * W->KT;
  W->info.launches = launches;
  W->info.calls += 1;
  return VT_OK;
}

extern "C" vt_status vt_fp4_noalloc_status(vt_stream_t s, int* status) {
  if (!status) return err(VT_ERR_INVALID_ARG, "status must be set");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  void* base = nullptr;
  if (e == cudaSuccess) e = scratch_address(dev, &base);
  int v = 0;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&v, base, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)s);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)s);
  if (e != cudaSuccess) return cuda_err(e);
  *status = v;
  if (v) {
    const int zero = 0;
    e = cudaMemcpyAsync(base, &zero, sizeof(int), cudaMemcpyHostToDevice, (cudaStream_t)s);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)s);
    if (e != cudaSuccess) return cuda_err(e);
  }
  return VT_OK;
}

extern "C" vt_status vt_fp4_noalloc_test_hooks(int wait_limit_us, int withhold_weights) {
  if (wait_limit_us < 0) return err(VT_ERR_INVALID_ARG, "wait_limit_us must be >= 0");
  g_hook_wait_us.store(wait_limit_us);
  g_hook_withhold.store(withhold_weights ? 1 : 0);
  return VT_OK;
}
