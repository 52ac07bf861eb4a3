// C ABI of libvtfp4 (declared in include/vt_fp4.h): argument checks, handle state, launch
// shape selection and kernel launches.  Every check that needs no GPU runs before any
// CUDA call, so bad arguments are rejected the same way on a host without a device.
#include <float.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <new>

#include "vt_fp4.h"
#include "common.cuh"
#include "handle.h"
#include "kernels.h"

using namespace vt;

namespace {

thread_local char g_err[512] = "";

vt_status fail(vt_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

vt_status cuda_fail(cudaError_t e, const char* where) {
  return fail(VT_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Greedy head state inside the workspace's first 256 bytes (after the status word): one
// 64-bit key per token and the finished-CTA counter; zero between calls.
constexpr size_t kGreedyKeysOff = 64;
constexpr size_t kGreedyDoneOff = 64 + 16 * 8;

inline int group_of(int fmt) { return fmt == VT_FP4_NVFP4 ? 16 : 32; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

vt_status check_shape(vt_fp4_format fmt, int64_t N, int64_t K) {
  if (fmt != VT_FP4_NVFP4 && fmt != VT_FP4_MXFP4)
    return fail(VT_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
  if (N <= 0 || K <= 0) return fail(VT_ERR_INVALID_ARG, "N and K must be > 0 (N=%lld K=%lld)",
                                    (long long)N, (long long)K);
  if (K % group_of(fmt))
    return fail(VT_ERR_INVALID_ARG, "K=%lld is not a multiple of the group size %d",
                (long long)K, group_of(fmt));
  if (N > (int64_t)1 << 31 || K > (int64_t)1 << 24)
    return fail(VT_ERR_UNSUPPORTED, "N or K too large (N=%lld K=%lld)", (long long)N,
                (long long)K);
  return VT_OK;
}

size_t packed_size(int fmt, int64_t N, int64_t K) {
  return (size_t)kHeaderBytes +
         (size_t)cdiv(N, kTileRows) * cdiv(K, kTileK) * tile_bytes(fmt);
}

// Workspace layout shared by vt_fp4_workspace_bytes and the GEMM.
struct WsLayout {
  size_t status, counters, rowscale, ap, partials, total;
};

WsLayout ws_layout(const vt_fp4_weight_s* W, int64_t M) {
  WsLayout L;
  const int64_t Kp = W->KT * kTileK;
  const int64_t mrows = M <= 16 ? 16 : cdiv(M, 128) * 128;
  L.status = 0;
  L.counters = 256;
  // the counters keep a fixed region (64 KB, or more for weights of more row tiles), so that
  // no data of another weight sharing the workspace lands on them
  const size_t nctr = (size_t)(W->RT > kFixedCounterTiles ? W->RT : kFixedCounterTiles);
  // activation scales: decode [KT][16] floats; prefill one per token row
  L.rowscale = up256(L.counters + nctr * 4);
  const size_t nscale = M <= 16 ? (size_t)W->KT * 16 : (size_t)mrows;
  L.ap = up256(L.rowscale + nscale * 4);
  L.partials = up256(L.ap + (size_t)mrows * Kp * 2);
  const size_t part = M <= 16 ? (size_t)kMaxDecodeGrid * 2 * 16 * 128 * 4 : 0;
  L.total = up256(L.partials + part);
  return L;
}

// Workspace of the grouped (mixture-of-experts) GEMM for `npairs` (token, slot) pairs.
// Every offset is independent of npairs (so calls of any size can share one workspace
// without one call's data landing on another's split-K counters): status word, split-K
// counters per (problem, row tile) for the largest possible problem count, split-K
// partials, the group table, the activation scales [problems][KT][16], and last the
// gathered f16 activations [npairs][KT*64], whose size alone depends on npairs.
struct MoeLayout {
  size_t status, counters, partials, table, ascale, ap, total;
};

MoeLayout moe_layout(const vt_fp4_weight_s* W, int64_t npairs) {
  MoeLayout L;
  const int64_t pcap = W->E < 128 ? W->E : 128;  // problems: distinct experts of <= 128 pairs
  L.status = 0;
  L.counters = 256;
  const size_t nctr = (size_t)pcap * W->RT;
  L.partials = up256(L.counters + (nctr > (size_t)kFixedCounterTiles ? nctr : kFixedCounterTiles) * 4);
  L.table = up256(L.partials + (size_t)kMaxDecodeGrid * 2 * 16 * 128 * 4);
  L.ascale = up256(L.table + (size_t)kGroupTableInts * 4);
  L.ap = up256(L.ascale + (size_t)pcap * W->KT * 16 * 4);
  L.total = up256(L.ap + (size_t)npairs * W->KT * kTileK * 2);
  return L;
}

vt_status do_prepack(const uint8_t* const codes[2], const uint8_t* const scales[2],
                     const float globals[2], int nsrc, vt_fp4_format fmt, int64_t I, int64_t K,
                     void* dst, size_t dst_bytes, vt_stream_t s, vt_fp4_handle* out,
                     uint32_t layout = kLayoutRows) {
  if (!out) return fail(VT_ERR_INVALID_ARG, "out handle pointer is NULL");
  *out = nullptr;
  const int64_t N = I * nsrc;
  vt_status st = check_shape(fmt, N, K);
  if (st) return st;
  for (int i = 0; i < nsrc; ++i) {
    if (!codes[i] || !scales[i]) return fail(VT_ERR_INVALID_ARG, "codes/scales pointer is NULL");
    if (fmt == VT_FP4_NVFP4) {
      if (!(isfinite(globals[i]) && globals[i] > 0.0f))
        return fail(VT_ERR_INVALID_ARG, "NVFP4 global scale must be finite and > 0 (got %g)",
                    (double)globals[i]);
    } else if (globals[i] != 1.0f) {
      return fail(VT_ERR_INVALID_ARG, "MXFP4 has no global scale: pass 1.0 (got %g)",
                  (double)globals[i]);
    }
  }
  if (!dst) return fail(VT_ERR_INVALID_ARG, "packed_dst is NULL");
  if (!aligned(dst, 16)) return fail(VT_ERR_MISALIGNED, "packed_dst must be 16-byte aligned");
  const size_t need = packed_size(fmt, N, K);
  if (dst_bytes < need)
    return fail(VT_ERR_INVALID_ARG, "packed_dst holds %zu bytes, %zu needed", dst_bytes, need);

  vt_fp4_weight_s* h = new (std::nothrow) vt_fp4_weight_s();
  if (!h) return fail(VT_ERR_INVALID_ARG, "out of host memory");
  h->fmt = fmt;
  h->N = N;
  h->K = K;
  h->RT = cdiv(N, kTileRows);
  h->KT = cdiv(K, kTileK);
  h->seg_split = nsrc == 2 ? I : N;
  h->layout = (int)layout;
  h->packed = dst;
  h->packed_bytes = need;
  memset(&h->info, 0, sizeof(h->info));
  const uint8_t* c2[2] = {codes[0], nsrc == 2 ? codes[1] : codes[0]};
  const uint8_t* s2[2] = {scales[0], nsrc == 2 ? scales[1] : scales[0]};
  const float f1 = nsrc == 2 ? globals[1] : globals[0];
  cudaError_t e = launch_prepack(c2, s2, h->seg_split, globals[0], f1, fmt, N, K, h->RT, h->KT,
                                 layout, dst, (cudaStream_t)s);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "prepack launch");
  }
  *out = h;
  return VT_OK;
}

// The W4A4 activation global: NVFP4 takes a positive normal float, MXFP4 has none (1.0).
vt_status check_input_scale(int fmt, float a) {
  if (fmt == VT_FP4_NVFP4 ? (isfinite(a) && a >= FLT_MIN) : a == 1.0f) return VT_OK;
  return fail(VT_ERR_INVALID_ARG,
              fmt == VT_FP4_NVFP4 ? "input_scale must be a positive normal float (got %g)"
                                  : "MXFP4 activations have no global scale: input_scale must be 1 (got %g)",
              (double)a);
}

vt_status check_handle(vt_fp4_handle W) {
  if (!W) return fail(VT_ERR_INVALID_ARG, "weight handle is NULL");
  return VT_OK;
}

}  // namespace

vt_status vt::set_last_error(vt_status st, const char* msg) { return fail(st, "%s", msg); }

int vt::sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

vt_status vt::decode_shape(const vt_fp4_weight_s* W, int M, const vt_fp4_gemm_opts* opts,
                           bool w4a4, DecodeShape* out) {
  const int64_t items = W->RT * W->KT;
  // k tiles per pipeline stage (8: up to 37 KB of weights per TMA copy) and ring depth
  int ks = (opts && opts->warps) ? opts->warps : 8;  // opts->warps selects the stage width
  if (ks != 4 && ks != 8) return fail(VT_ERR_INVALID_ARG, "stage width must be 4 or 8 k tiles");
  // A long call (at least three row tiles per CTA of the default grid; bound by the
  // consumers) of up to 8 tokens and more than 4096 activation elements streams stages of
  // 16 k tiles, with the activations from the pre-pass: half the per-stage work per weight
  // (lm_head K = 5120: M = 1 -4 %, M = 2 -6 %, M = 8 -4 %).  Smaller activations keep the
  // in-kernel conversion and 8-tile stages (K = 2560, M = 1: +1.3 % with 16), and so do the
  // shorter calls (two 16-tile stages hold fewer bytes in flight than six of 8: ~2 % slower).
  const int64_t g8 = sm_count() < cdiv(items, 16) ? sm_count() : cdiv(items, 16);
  const bool long16 = !(opts && (opts->warps || opts->grid || opts->stages)) && W->E <= 1 &&
                      M <= 8 && (int64_t)M * W->K > 4096 && items >= 3 * W->KT * g8 &&
                      decode_smem_bytes(W->fmt, M, 16, 2, 0) <= 226 * 1024;
  if (long16) ks = 16;
  // small M * K: the decode kernel converts the activations itself (no pre-pass)
  const bool resident = !w4a4 && !(opts && opts->force_path == 3) && !long16 &&
                        decode_resident_ok(M, W->KT, W->RT);
  const int64_t rkt = resident ? W->KT : 0;
  int stages = (opts && opts->stages) ? opts->stages : 0;
  if (!stages) {  // as deep as shared memory allows, at most 6
    stages = 6;
    while (stages > 2 && decode_smem_bytes(W->fmt, M, ks, stages, rkt) > 226 * 1024) --stages;
  }
  if (stages < 2 || stages > 16) return fail(VT_ERR_INVALID_ARG, "stages must be in [2, 16]");
  if (decode_smem_bytes(W->fmt, M, ks, stages, rkt) > 226 * 1024)
    return fail(VT_ERR_INVALID_ARG, "stage width x stages exceed shared memory");
  int64_t grid = (opts && opts->grid) ? opts->grid : sm_count();
  if (!(opts && opts->grid)) {
    const int64_t per_cta = 2 * ks;  // at least two stages of work per CTA
    grid = grid < cdiv(items, per_cta) ? grid : cdiv(items, per_cta);
  }
  if (grid > items) grid = items;
  if (grid > kMaxDecodeGrid) grid = kMaxDecodeGrid;
  if (grid < 1) grid = 1;
  out->ks = ks;
  out->stages = stages;
  out->grid = (int)grid;
  out->resident = resident ? 1 : 0;
  // up to 2 tokens and at least three row tiles per CTA (the long lm_head-like calls): the
  // per-group epilogue, so that most warps do not stop at every tile's end
  out->epi = (ks == 8 && M <= 2 && items >= 3 * W->KT * grid) ? 1 : 0;
  return VT_OK;
}

extern "C" {

const char* vt_fp4_last_error(void) { return g_err; }

vt_status vt_fp4_prepack_bytes(vt_fp4_format fmt, int64_t N, int64_t K, size_t* packed_bytes) {
  if (!packed_bytes) return fail(VT_ERR_INVALID_ARG, "packed_bytes is NULL");
  vt_status st = check_shape(fmt, N, K);
  if (st) return st;
  *packed_bytes = packed_size(fmt, N, K);
  return VT_OK;
}

vt_status vt_fp4_prepack(const uint8_t* codes, const uint8_t* scales, float global_scale,
                         vt_fp4_format fmt, int64_t N, int64_t K, void* packed_dst,
                         size_t dst_bytes, vt_stream_t s, vt_fp4_handle* out) {
  const uint8_t* c[2] = {codes, codes};
  const uint8_t* sc[2] = {scales, scales};
  const float g[2] = {global_scale, global_scale};
  return do_prepack(c, sc, g, 1, fmt, N, K, packed_dst, dst_bytes, s, out);
}

vt_status vt_fp4_prepack_gate_up(const uint8_t* gate_codes, const uint8_t* gate_scales,
                                 float gate_global, const uint8_t* up_codes,
                                 const uint8_t* up_scales, float up_global, vt_fp4_format fmt,
                                 int64_t I, int64_t K, void* packed_dst, size_t dst_bytes,
                                 vt_stream_t s, vt_fp4_handle* out) {
  const uint8_t* c[2] = {gate_codes, up_codes};
  const uint8_t* sc[2] = {gate_scales, up_scales};
  const float g[2] = {gate_global, up_global};
  return do_prepack(c, sc, g, 2, fmt, I, K, packed_dst, dst_bytes, s, out);
}

vt_status vt_fp4_prepack_gate_up_paired(const uint8_t* gate_codes, const uint8_t* gate_scales,
                                        float gate_global, const uint8_t* up_codes,
                                        const uint8_t* up_scales, float up_global,
                                        vt_fp4_format fmt, int64_t I, int64_t K, void* packed_dst,
                                        size_t dst_bytes, vt_stream_t s, vt_fp4_handle* out) {
  const uint8_t* c[2] = {gate_codes, up_codes};
  const uint8_t* sc[2] = {gate_scales, up_scales};
  const float g[2] = {gate_global, up_global};
  return do_prepack(c, sc, g, 2, fmt, I, K, packed_dst, dst_bytes, s, out, kLayoutPaired);
}

vt_status vt_fp4_prepack_grouped_bytes(vt_fp4_format fmt, int64_t E, int64_t N, int64_t K,
                                       size_t* packed_bytes) {
  if (!packed_bytes) return fail(VT_ERR_INVALID_ARG, "packed_bytes is NULL");
  if (E <= 0 || E > 65536) return fail(VT_ERR_INVALID_ARG, "E must be in [1, 65536]");
  vt_status st = check_shape(fmt, N, K);
  if (st) return st;
  *packed_bytes = (size_t)E * packed_size(fmt, N, K);
  return VT_OK;
}

vt_status vt_fp4_prepack_grouped(const uint8_t* codes, const uint8_t* scales,
                                 const float* globals, vt_fp4_format fmt, int64_t E, int64_t N,
                                 int64_t K, void* packed_dst, size_t dst_bytes, vt_stream_t s,
                                 vt_fp4_handle* out) {
  if (!out) return fail(VT_ERR_INVALID_ARG, "out handle pointer is NULL");
  *out = nullptr;
  size_t need = 0;
  if (vt_status st = vt_fp4_prepack_grouped_bytes(fmt, E, N, K, &need)) return st;
  if (!codes || !scales || !globals || !packed_dst)
    return fail(VT_ERR_INVALID_ARG, "codes, scales, globals and packed_dst must be set");
  if (dst_bytes < need)
    return fail(VT_ERR_INVALID_ARG, "packed_dst holds %zu bytes, %zu needed", dst_bytes, need);
  const size_t per = packed_size(fmt, N, K);
  const int64_t g = group_of(fmt);
  vt_fp4_handle first = nullptr;
  for (int64_t e = 0; e < E; ++e) {
    const uint8_t* c = codes + e * N * (K / 2);
    const uint8_t* sc = scales + e * N * (K / g);
    vt_fp4_handle h = nullptr;
    vt_status st = vt_fp4_prepack(c, sc, globals[e], fmt, N, K,
                                  static_cast<uint8_t*>(packed_dst) + e * per, per, s, &h);
    if (st) {
      delete first;
      return st;
    }
    if (e == 0) first = h;
    else delete h;
  }
  first->E = E;
  first->expert_bytes = (int64_t)per;
  first->packed_bytes = need;
  *out = first;
  return VT_OK;
}

vt_status vt_fp4_destroy(vt_fp4_handle W) {
  delete W;
  return VT_OK;
}

vt_status vt_fp4_shape(vt_fp4_handle W, vt_fp4_format* fmt, int64_t* N, int64_t* K) {
  if (vt_status st = check_handle(W)) return st;
  if (fmt) *fmt = (vt_fp4_format)W->fmt;
  if (N) *N = W->N;
  if (K) *K = W->K;
  return VT_OK;
}

vt_status vt_fp4_workspace_bytes(vt_fp4_handle W, int64_t M_max, size_t* bytes) {
  if (vt_status st = check_handle(W)) return st;
  if (!bytes) return fail(VT_ERR_INVALID_ARG, "bytes is NULL");
  if (M_max < 0) return fail(VT_ERR_INVALID_ARG, "M_max must be >= 0");
  WsLayout a = ws_layout(W, M_max < 1 ? 1 : M_max);
  size_t tot = a.total;
  if (M_max > 16) {  // a workspace sized for M_max also serves every smaller M
    WsLayout d = ws_layout(W, 16);
    if (d.total > tot) tot = d.total;
  }
  *bytes = tot;
  return VT_OK;
}

}  // extern "C"

namespace {

// The GEMM behind vt_fp4_w4a16_gemm_ex and vt_fp4_w4a16_gemm_greedy: with g_idx set, the
// decode kernel keeps the per-token greedy choice instead of writing C.
vt_status gemm_impl(const void* A, int64_t M, int64_t lda, vt_fp4_handle W, void* C,
                    int64_t ldc, void* workspace, size_t ws_bytes, vt_stream_t s,
                    const vt_fp4_gemm_opts* opts, int32_t* g_idx, float* g_val,
                    bool silu = false, bool w4a4 = false, float alpha = 1.0f) {
  if (vt_status st = check_handle(W)) return st;
  if (W->E > 1) return fail(VT_ERR_INVALID_ARG, "a grouped weight serves vt_fp4_w4a16_gemm_moe");
  if (M < 0) return fail(VT_ERR_INVALID_ARG, "M must be >= 0 (got %lld)", (long long)M);
  if (M == 0) return VT_OK;
  if (!A || !workspace || !(C || g_idx))
    return fail(VT_ERR_INVALID_ARG, "A, C and workspace must be set");
  const int64_t ncols = silu ? W->seg_split : W->N;  // output columns
  if (lda < W->K || (!g_idx && ldc < ncols))
    return fail(VT_ERR_INVALID_ARG, "lda (%lld) must be >= K and ldc (%lld) >= N",
                (long long)lda, (long long)ldc);
  if (!aligned(A, 16) || lda % 8)
    return fail(VT_ERR_MISALIGNED, "A must be 16-byte aligned with lda %% 8 == 0");
  if (!g_idx && !aligned(C, 2)) return fail(VT_ERR_MISALIGNED, "C must be 2-byte aligned");
  if (!aligned(workspace, 256)) return fail(VT_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  const int force = opts ? opts->force_path : 0;
  if (force < 0 || force > 3) return fail(VT_ERR_INVALID_ARG, "force_path must be 0..3");
  const bool decode = force ? force != 2 : M <= 16;
  if (decode && M > 16) return fail(VT_ERR_INVALID_ARG, "decode path needs M <= 16");
  if (W->K > 110000) return fail(VT_ERR_UNSUPPORTED, "K > 110000 is not supported");
  WsLayout L = ws_layout(W, decode ? (M < 16 ? M : 16) : M);
  if (ws_bytes < L.total)
    return fail(VT_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", ws_bytes, L.total);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);

  if (decode) {
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
    D.status = reinterpret_cast<int*>(ws + L.status);
    D.counters = reinterpret_cast<int*>(ws + L.counters);
    D.ascale = reinterpret_cast<float*>(ws + L.rowscale);
    D.Ap = ws + L.ap;
    D.partials = reinterpret_cast<float*>(ws + L.partials);
    const int64_t items = W->RT * W->KT;
    const int mt = decode_mt((int)M);
    DecodeShape sh;
    if (vt_status st = decode_shape(W, (int)M, opts, w4a4, &sh)) return st;
    D.grid = sh.grid;
    D.ks = sh.ks;
    D.stages = sh.stages;
    D.wait_ns = (opts && opts->wait_limit_us > 0) ? (uint64_t)opts->wait_limit_us * 1000ull : 0;
    D.withhold = opts ? opts->withhold_weights : 0;
    D.layout = (uint32_t)W->layout;
    D.silu = silu ? 1 : 0;
    D.w4a4 = w4a4 ? 1 : 0;
    D.alpha = alpha;
    D.resident = sh.resident;
    D.epi = sh.epi;
    if (g_idx) {
      D.g_idx = g_idx;
      D.g_val = g_val;
      D.g_keys = reinterpret_cast<unsigned long long*>(ws + kGreedyKeysOff);
      D.g_done = reinterpret_cast<unsigned int*>(ws + kGreedyDoneOff);
    }
    int launches = 0;
    cudaError_t e = launch_decode(D, (cudaStream_t)s, &launches);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    W->info.path = 1;
    W->info.tile_epilogue = sh.epi;
    W->info.stage_k_tiles = sh.ks;
    W->info.grid = D.grid;
    W->info.warps_per_cta = 18;  // 16 consumer warps, the TMA producer, the publisher
    W->info.m_tile = mt;
    W->info.items = items;
    W->info.launches = launches;
    W->info.calls += 1;
    return VT_OK;
  }
  PrefillLaunch P;
  P.packed = W->packed;
  P.fmt = W->fmt;
  P.N = W->N;
  P.K = W->K;
  P.RT = W->RT;
  P.KT = W->KT;
  P.seg_split = W->seg_split;
  P.A = A;
  P.lda = lda;
  P.M = M;
  P.C = C;
  P.ldc = ldc;
  P.status = reinterpret_cast<int*>(ws + L.status);
  P.rowscale = reinterpret_cast<float*>(ws + L.rowscale);
  P.Ap = ws + L.ap;
  P.grid = (opts && opts->grid) ? opts->grid : sm_count();
  P.wait_ns = (opts && opts->wait_limit_us > 0) ? (uint64_t)opts->wait_limit_us * 1000ull : 0;
  P.withhold = opts ? opts->withhold_weights : 0;
  P.layout = (uint32_t)W->layout;
  P.silu = silu ? 1 : 0;
  P.w4a4 = w4a4 ? 1 : 0;
  P.alpha = alpha;
  int launches = 0, grid = 0;
  int64_t tiles = 0;
  cudaError_t e = launch_prefill(P, (cudaStream_t)s, &launches, &grid, &tiles);
  if (e == cudaErrorNotSupported)
    return fail(VT_ERR_UNSUPPORTED, "the prefill tile path is not available in this build");
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  W->info.path = 2;
  W->info.tile_epilogue = 0;
  W->info.stage_k_tiles = 1;
  W->info.grid = grid;
  W->info.warps_per_cta = 14;  // TMA, MMA, 8 dequantiser and 4 epilogue warps
  W->info.m_tile = 128;
  W->info.items = tiles;
  W->info.launches = launches;
  W->info.calls += 1;
  return VT_OK;
}

}  // namespace

extern "C" {

vt_status vt_fp4_moe_workspace_bytes(vt_fp4_handle W, int64_t M_max, int64_t topk,
                                     size_t* bytes) {
  if (vt_status st = check_handle(W)) return st;
  if (!bytes) return fail(VT_ERR_INVALID_ARG, "bytes is NULL");
  if (M_max < 1 || M_max > 16 || topk < 1 || topk > 8)
    return fail(VT_ERR_INVALID_ARG, "M_max must be in [1, 16] and topk in [1, 8]");
  *bytes = moe_layout(W, M_max * topk).total;
  return VT_OK;
}

vt_status vt_fp4_w4a16_gemm_moe(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                                const int32_t* topk_ids, int64_t topk, void* C, int64_t ldc,
                                void* workspace, size_t ws_bytes, vt_stream_t s) {
  if (vt_status st = check_handle(W)) return st;
  if (M < 0 || M > 16) return fail(VT_ERR_UNSUPPORTED, "the grouped GEMM serves 0 <= M <= 16");
  if (topk < 1 || topk > 8) return fail(VT_ERR_INVALID_ARG, "topk must be in [1, 8]");
  if (M == 0) return VT_OK;
  if (!A || !C || !topk_ids || !workspace)
    return fail(VT_ERR_INVALID_ARG, "A, topk_ids, C and workspace must be set");
  if (W->layout != kLayoutRows || W->seg_split != W->N)
    return fail(VT_ERR_INVALID_ARG, "a grouped weight holds plain experts");
  if (lda < W->K || ldc < W->N)
    return fail(VT_ERR_INVALID_ARG, "lda must be >= K and ldc >= N");
  if (!aligned(A, 16) || lda % 8)
    return fail(VT_ERR_MISALIGNED, "A must be 16-byte aligned with lda %% 8 == 0");
  if (!aligned(C, 2)) return fail(VT_ERR_MISALIGNED, "C must be 2-byte aligned");
  if (!aligned(workspace, 256)) return fail(VT_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  if (!aligned(topk_ids, 4)) return fail(VT_ERR_MISALIGNED, "topk_ids must be 4-byte aligned");
  if (W->K > 110000) return fail(VT_ERR_UNSUPPORTED, "K > 110000 is not supported");
  const int npairs = (int)(M * topk);
  MoeLayout L = moe_layout(W, npairs);
  if (ws_bytes < L.total)
    return fail(VT_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", ws_bytes, L.total);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  int ks = 8;
  // token tile of the decode kernel: 8 rows when M <= 8 (an expert then has at most M pairs
  // unless a token names it twice; such extra pairs are left out), else 16
  const int mrows = decode_mt((int)M);
  // up to 8 tokens whose converted activations fit kGroupedResidentMaxBytes: the decode
  // kernel groups the routing and converts the activations itself (one kernel, no pre-pass)
  const bool resident = mrows == 8 && decode_resident_bytes(mrows, W->KT) <= kGroupedResidentMaxBytes;
  const int64_t rkt = resident ? W->KT : 0;
  // the routing names at most pmax experts (the grouping finds how many it does)
  const int64_t pmax = npairs < W->E ? npairs : W->E;
  // long calls (at least three row tiles per CTA for pmax experts): 16-k-tile stages halve
  // the consumers' per-stage waits and releases
  if (resident && pmax * W->RT >= 3 * (int64_t)sm_count() &&
      decode_smem_bytes(W->fmt, mrows, 16, 2, rkt) <= 222 * 1024)
    ks = 16;
  int stages = 6;  // the grouped kernel also holds ~3.5 KB of static shared memory (the grouping)
  while (stages > 2 && decode_smem_bytes(W->fmt, mrows, ks, stages, rkt) > 222 * 1024) --stages;
  if (decode_smem_bytes(W->fmt, mrows, ks, stages, rkt) > 222 * 1024)
    return fail(VT_ERR_UNSUPPORTED, "K too large for the grouped kernel's shared memory");
  const int64_t items = pmax * W->RT * W->KT;  // an upper bound
  int64_t grid = sm_count();
  if (grid > cdiv(items, 2 * ks)) grid = cdiv(items, 2 * ks);
  // one-launch mode whose row tiles (by the routing's upper bound) fit the SMs: one whole row
  // tile per CTA, no split-K reduction (128 experts of 1536 x 2048, one token, top-8: 96 CTAs,
  // 11.2 -> 10.0 us per call)
  if (resident && pmax * W->RT <= sm_count()) grid = pmax * W->RT;
  if (grid > kMaxDecodeGrid) grid = kMaxDecodeGrid;
  if (grid < 1) grid = 1;
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
  D.M = mrows;
  D.C = C;
  D.ldc = ldc;
  D.status = reinterpret_cast<int*>(ws + L.status);
  D.counters = reinterpret_cast<int*>(ws + L.counters);
  D.ascale = reinterpret_cast<float*>(ws + L.ascale);
  D.Ap = ws + L.ap;
  D.partials = reinterpret_cast<float*>(ws + L.partials);
  D.grid = (int)grid;
  D.ks = ks;
  D.stages = stages;
  D.wait_ns = 0;
  D.withhold = 0;
  D.gtab = reinterpret_cast<const int*>(ws + L.table);
  D.expert_bytes = W->expert_bytes ? W->expert_bytes : (int64_t)W->packed_bytes;
  D.resident = resident ? 1 : 0;
  int launches = 0;
  cudaError_t e = launch_decode_grouped(D, topk_ids, npairs, (int)topk, (int)W->E,
                                        (cudaStream_t)s, &launches);
  if (e != cudaSuccess) return cuda_fail(e, "grouped decode launch");
  W->info.path = 3;
  W->info.tile_epilogue = resident ? 1 : 0;  // one-launch mode: the per-group epilogue
  W->info.stage_k_tiles = D.ks;
  W->info.grid = D.grid;
  W->info.warps_per_cta = 18;
  W->info.m_tile = mrows;
  W->info.items = items;
  W->info.launches = launches;
  W->info.calls += 1;
  return VT_OK;
}

vt_status vt_fp4_w4a16_gemm_ex(const void* A, int64_t M, int64_t lda, vt_fp4_handle W, void* C,
                               int64_t ldc, void* workspace, size_t ws_bytes, vt_stream_t s,
                               const vt_fp4_gemm_opts* opts) {
  return gemm_impl(A, M, lda, W, C, ldc, workspace, ws_bytes, s, opts, nullptr, nullptr);
}

vt_status vt_fp4_w4a16_gemm_greedy(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                                   int32_t* token, float* value, void* workspace,
                                   size_t ws_bytes, vt_stream_t s) {
  if (!token) return fail(VT_ERR_INVALID_ARG, "token must be set");
  if (M > 16) return fail(VT_ERR_UNSUPPORTED, "the greedy head serves M <= 16");
  if (W && W->N > 2147483647LL) return fail(VT_ERR_UNSUPPORTED, "N must fit in int32");
  if (!aligned(token, 4) || (value && !aligned(value, 4)))
    return fail(VT_ERR_MISALIGNED, "token and value must be 4-byte aligned");
  vt_fp4_gemm_opts o = {};
  o.force_path = 1;
  return gemm_impl(A, M, lda, W, nullptr, 0, workspace, ws_bytes, s, &o, token, value);
}

vt_status vt_fp4_w4a16_gemm_silu_mul(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                                     void* C, int64_t ldc, void* workspace, size_t ws_bytes,
                                     vt_stream_t s) {
  if (vt_status st = check_handle(W)) return st;
  if (W->layout != kLayoutPaired)
    return fail(VT_ERR_INVALID_ARG,
                "the SiLU-and-multiply epilogue needs a weight from vt_fp4_prepack_gate_up_paired");
  return gemm_impl(A, M, lda, W, C, ldc, workspace, ws_bytes, s, nullptr, nullptr, nullptr, true);
}

vt_status vt_fp4_w4a4_gemm_ex(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                              float input_scale, void* C, int64_t ldc, void* workspace,
                              size_t ws_bytes, vt_stream_t s, const vt_fp4_gemm_opts* opts) {
  if (vt_status st = check_handle(W)) return st;
  if (vt_status st = check_input_scale(W->fmt, input_scale)) return st;
  return gemm_impl(A, M, lda, W, C, ldc, workspace, ws_bytes, s, opts, nullptr, nullptr, false,
                   true, input_scale);
}

vt_status vt_fp4_w4a4_gemm(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                           float input_scale, void* C, int64_t ldc, void* workspace,
                           size_t ws_bytes, vt_stream_t s) {
  return vt_fp4_w4a4_gemm_ex(A, M, lda, W, input_scale, C, ldc, workspace, ws_bytes, s, nullptr);
}

vt_status vt_fp4_quantize_act(const void* A, int64_t M, int64_t lda, int64_t K,
                              vt_fp4_format fmt, float input_scale, uint8_t* codes,
                              uint8_t* scales, vt_stream_t s) {
  if (vt_status st = check_shape(fmt, 1, K)) return st;
  if (vt_status st = check_input_scale(fmt, input_scale)) return st;
  if (M < 0) return fail(VT_ERR_INVALID_ARG, "M must be >= 0 (got %lld)", (long long)M);
  if (M == 0) return VT_OK;
  if (!A || !codes || !scales) return fail(VT_ERR_INVALID_ARG, "A, codes and scales must be set");
  if (lda < K) return fail(VT_ERR_INVALID_ARG, "lda (%lld) must be >= K", (long long)lda);
  if (!aligned(A, 16) || lda % 8 || !aligned(codes, 16))
    return fail(VT_ERR_MISALIGNED, "A and codes must be 16-byte aligned with lda %% 8 == 0");
  cudaError_t e = launch_quantize_act(A, M, lda, K, fmt, input_scale, codes, scales,
                                      (cudaStream_t)s);
  return e == cudaSuccess ? VT_OK : cuda_fail(e, "activation quantiser launch");
}

vt_status vt_fp4_w4a16_gemm(const void* A, int64_t M, int64_t lda, vt_fp4_handle W, void* C,
                            int64_t ldc, void* workspace, size_t ws_bytes, vt_stream_t s) {
  return vt_fp4_w4a16_gemm_ex(A, M, lda, W, C, ldc, workspace, ws_bytes, s, nullptr);
}

vt_status vt_fp4_workspace_status(void* workspace, vt_stream_t s, int* status) {
  if (!workspace || !status) return fail(VT_ERR_INVALID_ARG, "workspace and status must be set");
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)s);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace status");
  *status = v;
  if (v) {
    const int zero = 0;
    e = cudaMemcpyAsync(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice, (cudaStream_t)s);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace status");
  }
  return VT_OK;
}

vt_status vt_fp4_stats(vt_fp4_handle W, vt_fp4_launch_info* info) {
  if (vt_status st = check_handle(W)) return st;
  if (!info) return fail(VT_ERR_INVALID_ARG, "info is NULL");
  *info = W->info;
  return VT_OK;
}

vt_status vt_fp4_dequant(vt_fp4_handle W, float* out, vt_stream_t s) {
  if (vt_status st = check_handle(W)) return st;
  if (!out) return fail(VT_ERR_INVALID_ARG, "out is NULL");
  cudaError_t e = cudaSuccess;
  for (int64_t x = 0; x < W->E && e == cudaSuccess; ++x)  // grouped: experts one after another
    e = launch_dequant(static_cast<const uint8_t*>(W->packed) + x * W->expert_bytes, W->fmt, W->N,
                       W->K, W->RT, W->KT, W->seg_split, (uint32_t)W->layout,
                       out + x * W->N * W->K, (cudaStream_t)s);
  return e == cudaSuccess ? VT_OK : cuda_fail(e, "dequant launch");
}

vt_status vt_fp4_unpack(vt_fp4_handle W, uint8_t* codes, uint8_t* scales, vt_stream_t s) {
  if (vt_status st = check_handle(W)) return st;
  if (!codes || !scales) return fail(VT_ERR_INVALID_ARG, "codes and scales must be set");
  cudaError_t e = cudaSuccess;
  const int64_t g = group_of(W->fmt);
  for (int64_t x = 0; x < W->E && e == cudaSuccess; ++x)  // grouped: experts one after another
    e = launch_unpack(static_cast<const uint8_t*>(W->packed) + x * W->expert_bytes, W->fmt, W->N,
                      W->K, W->RT, W->KT, W->seg_split, (uint32_t)W->layout,
                      codes + x * W->N * (W->K / 2), scales + x * W->N * (W->K / g),
                      (cudaStream_t)s);
  return e == cudaSuccess ? VT_OK : cuda_fail(e, "unpack launch");
}

vt_status vt_fp4_quantize(const void* Wt, int64_t N, int64_t K, vt_fp4_format fmt,
                          uint8_t* codes, uint8_t* scales, float* global_out, void* scratch,
                          vt_stream_t s) {
  vt_status st = check_shape(fmt, N, K);
  if (st) return st;
  if (!Wt || !codes || !scales || !scratch)
    return fail(VT_ERR_INVALID_ARG, "W, codes, scales and scratch must be set");
  if (fmt == VT_FP4_NVFP4 && !global_out)
    return fail(VT_ERR_INVALID_ARG, "NVFP4 needs global_out");
  if (!aligned(Wt, 16) || !aligned(scratch, 16) || !aligned(codes, 16))
    return fail(VT_ERR_MISALIGNED, "W, codes and scratch must be 16-byte aligned");
  cudaError_t e = launch_quantize(Wt, N, K, fmt, codes, scales, global_out, scratch,
                                  (cudaStream_t)s);
  return e == cudaSuccess ? VT_OK : cuda_fail(e, "quantize launch");
}

}  // extern "C"
