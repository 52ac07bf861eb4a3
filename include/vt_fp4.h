/*
 * vt_fp4.h -- C ABI of libvtfp4: FP4 weight-only (W4A16) linear layers on GB300 (sm_103a).
 *
 * The layer:  C[m][n] = bf16( sum_k A[m][k] * w[n][k] ),  A bf16 [M][K], w dequantised
 * from FP4:
 *   NVFP4  w = e2m1(code) * e4m3(scale[n][k/16]) * global      (global: fp32 multiplier)
 *   MXFP4  w = e2m1(code) * 2^(e8m0(scale[n][k/32]) - 127)     (no global)
 * Sources (vllm.cpp pull-request pages):
 *   "keep the ModelOpt NVFP4 lm_head packed" (PR #263), "Why this row matters": the
 *     packed NVFP4 head is U8 codes (two per byte) + FP8 scales + FP32 second scale, and
 *     it runs as a W4A16 GEMM instead of being expanded to bf16;
 *   "re-verify 27B NVFP4 on the nvidia ModelOpt checkpoint" (PR #178), "Layer 3": the
 *     ModelOpt weight_scale_2 is a direct multiplier; "W4A16 is the default": activation
 *     scales (input_scale) are not consumed;
 *   "native MXFP4 keep-quant + Qwen e2e" (PR #38), commit "W2": MXFP4 is E2M1 with one
 *     E8M0 scale per 32 weights, U8 [N, K/32], and no global scale;
 *   "MXFP4 decode-graph + gate_up FUSION default-ON" (PR #54), "Step 2": gate and up are
 *     merged into one GEMM of N = 2*I.
 *
 * Conventions for every entry point:
 *   - Pointers marked (device) are CUDA device pointers owned by the caller; (host) are
 *     host pointers.  The library never allocates device memory and keeps no global
 *     cache keyed by address: all state of a prepacked weight lives in its handle and in
 *     the caller's packed buffer.  Source: "keep the ModelOpt NVFP4 lm_head packed"
 *     (PR #263), "Round-2 findings resolved", item 1 (residency is a property of the
 *     weight, not of the GEMM) and "Merge with origin/main" (#237 / #276: the weights own
 *     their resident device state, not a static address map, which reused stale pointers
 *     after teardown).
 *   - Work is enqueued on the caller's stream `s` and is asynchronous; no entry point
 *     synchronises the device except vt_fp4_workspace_status and vt_fp4_noalloc_status.
 *   - Every entry returns a vt_status and never aborts, and no entry falls back to another
 *     path when its own cannot run: a case it does not serve is an error.  On failure
 *     nothing is enqueued and vt_fp4_last_error() returns a message for the calling thread.
 *     Source: same page, "Round-2 findings resolved", the backend-asymmetric hard abort
 *     (an abort is recorded as a defect) and why it was preferred to a silent fall-through
 *     (a head that quietly lost its packed form costs throughput with no other symptom).
 *   - Built for sm_103a only; on another device the launches fail with VT_ERR_CUDA.
 */
#ifndef VT_FP4_H
#define VT_FP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* vt_stream_t; /* same object as cudaStream_t; NULL = default */

typedef enum { VT_FP4_NVFP4 = 0, VT_FP4_MXFP4 = 1 } vt_fp4_format;

typedef enum {
  VT_OK = 0,
  VT_ERR_INVALID_ARG = 1, /* bad size, null pointer, bad scale, format mismatch */
  VT_ERR_UNSUPPORTED = 2, /* a shape or option this build does not implement */
  VT_ERR_MISALIGNED = 3,  /* a pointer or leading dimension breaks the alignment rule */
  VT_ERR_CUDA = 4,        /* a CUDA runtime call failed (message has the CUDA error) */
  VT_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (see workspace status) */
} vt_status;

typedef struct vt_fp4_weight_s* vt_fp4_handle;

/* What the last GEMM call on a handle launched (host-side record). */
typedef struct {
  int path;           /* 0 none yet, 1 decode (M <= 16), 2 prefill tile path,
                         3 grouped mixture-of-experts decode */
  int grid;           /* CTAs of the main kernel */
  int warps_per_cta;  /* warps per CTA of the main kernel */
  int m_tile;         /* decode and grouped: tokens per MMA column block (8 or 16);
                         prefill: 128 */
  int64_t items;      /* decode: (row tile, k tile) work items; grouped: an upper bound on
                         them (the routing is read on the device); prefill: output tiles */
  int64_t launches;   /* kernels enqueued by that call */
  int64_t calls;      /* GEMM calls made on this handle so far */
  int tile_epilogue;  /* decode: 1 when complete row tiles were summed per row-block group
                         (up to 2 tokens, at least three row tiles per CTA), else 0; grouped:
                         1 in the one-launch mode, whose complete tiles of problems of up to
                         2 slots are summed that way */
  int stage_k_tiles;  /* decode and grouped: 64-wide k tiles per pipeline stage (4, 8, or 16
                         for up to 8 tokens and more than 4096 activation elements on a call
                         of at least three row tiles per CTA; grouped: 16 in the one-launch
                         mode when min(M * topk, E) experts give at least three row tiles
                         per CTA); prefill: 1 (one 64-wide k step per stage) */
} vt_fp4_launch_info;

/* Optional overrides for vt_fp4_w4a16_gemm_ex (0 = library choice). */
typedef struct {
  int grid;      /* decode: number of CTAs (clamped to [1, 512]); prefill: CTAs (>= 1) */
  int warps;     /* decode: k tiles (of 64) per pipeline stage, 4 or 8 (the library's own
                    choice is 8, or 16 for the long calls that stage_k_tiles describes;
                    setting grid, warps or stages keeps it from choosing 16) */
  int stages;    /* decode: depth of the CTA's TMA ring, 2..16 */
  int force_path;/* 1 decode (requires M <= 16), 2 prefill, 3 decode with the activations
                    always converted by the pre-pass kernel (small M * K otherwise converts
                    them inside the decode kernel) */
  int wait_limit_us;   /* limit of every bounded device-side wait, in microseconds
                        * (0 = 2 s); a wait that runs out sets VT_ERR_TIMEOUT in the
                        * workspace status word and the kernel finishes without waiting */
  int withhold_weights;/* test hook for the failure path: when nonzero the kernels' weight
                        * producer issues no copies, so the bounded waits run out; the call
                        * completes, the status word reads VT_ERR_TIMEOUT and the output is
                        * undefined.  The workspace stays reusable. */
} vt_fp4_gemm_opts;

/* ---------------------------------------------------------------------- sizes */

/* Exact size in bytes of the prepacked buffer for an N x K weight of format `fmt`:
 * a 256-byte header plus ceil(N/128)*ceil(K/64) tiles of 4608 (NVFP4) or 4352 (MXFP4)
 * bytes (the packed codes and scales plus padding of at most one tile in each direction).
 * Requires N > 0, K > 0, K % 16 == 0 (NVFP4) or K % 32 == 0 (MXFP4).  Source: "keep the
 * ModelOpt NVFP4 lm_head packed" (PR #263), "Round-2 findings resolved", item 5: the packed
 * head's operands had been built 4 bytes per element and are now exactly sized; the caller
 * allocates exactly this many bytes. */
vt_status vt_fp4_prepack_bytes(vt_fp4_format fmt, int64_t N, int64_t K, size_t* packed_bytes);

/* ------------------------------------------------------------------- prepack */

/* Reorders one weight into the kernels' tile layout (a bijection of the code and scale
 * bytes plus zero padding) and returns a handle.  Source: "keep the ModelOpt NVFP4
 * lm_head packed" (PR #263): the weight stays packed and its resident form is built once
 * at load, "paid once, instead of rebuilding ... every decode step".
 *   codes        (device) u8 [N][K/2], row-major; the low nibble holds the even k.
 *   scales       (device) u8 [N][K/g], row-major; g = 16 (E4M3) or 32 (E8M0).
 *   global_scale NVFP4: the fp32 multiplier (ModelOpt weight_scale_2), finite and > 0;
 *                MXFP4: must be 1.0f (the format has no global scale).
 *   packed_dst   (device) caller-owned, 16-byte aligned, >= vt_fp4_prepack_bytes bytes;
 *                it must outlive the handle and must not be written by the caller.
 * codes/scales are read by kernels enqueued on `s`; they may be freed once those have
 * run.  *out receives a new handle (free it with vt_fp4_destroy). */
vt_status vt_fp4_prepack(const uint8_t* codes, const uint8_t* scales, float global_scale,
                         vt_fp4_format fmt, int64_t N, int64_t K, void* packed_dst,
                         size_t dst_bytes, vt_stream_t s, vt_fp4_handle* out);

/* Fused gate_up: one handle holding gate (rows [0, I)) and up (rows [I, 2I)), each with
 * its own codes, scales and global, so that one GEMM call writes C[M][2I] with gate in
 * columns [0, I) and up in [I, 2I).  Source: "MXFP4 decode-graph + gate_up FUSION
 * default-ON" (PR #54), "Step 2".  Sizes as vt_fp4_prepack with N = 2*I. */
vt_status vt_fp4_prepack_gate_up(const uint8_t* gate_codes, const uint8_t* gate_scales,
                                 float gate_global, const uint8_t* up_codes,
                                 const uint8_t* up_scales, float up_global, vt_fp4_format fmt,
                                 int64_t I, int64_t K, void* packed_dst, size_t dst_bytes,
                                 vt_stream_t s, vt_fp4_handle* out);

/* Fused gate_up paired for the SiLU-and-multiply epilogue: the same two weights as
 * vt_fp4_prepack_gate_up, with each 128-row tile holding 64 gate rows and the same 64 up
 * rows, so that vt_fp4_w4a16_gemm_silu_mul can form silu(gate) * up inside one tile.
 * Source: "MXFP4 decode-graph + gate_up FUSION default-ON" (PR #54), "Step 2" (gate and up
 * as one GEMM) and "Attribution" (the glue between the MLP GEMMs is a measured cost).
 * Arguments and sizes as vt_fp4_prepack_gate_up.  The handle also serves
 * vt_fp4_w4a16_gemm (which then writes C[M][2I], gate in columns [0, I)), vt_fp4_unpack
 * and vt_fp4_dequant (both in gate-over-up row order). */
vt_status vt_fp4_prepack_gate_up_paired(const uint8_t* gate_codes, const uint8_t* gate_scales,
                                        float gate_global, const uint8_t* up_codes,
                                        const uint8_t* up_scales, float up_global,
                                        vt_fp4_format fmt, int64_t I, int64_t K, void* packed_dst,
                                        size_t dst_bytes, vt_stream_t s, vt_fp4_handle* out);

/* Frees the host-side handle (never device memory); the caller frees the packed buffer
 * afterwards.  NULL is a no-op.  Source: "keep the ModelOpt NVFP4 lm_head packed" (PR #263),
 * "Merge with origin/main" (#237 / #276): a weight's resident state is owned by the weight and
 * released with it, never kept in a cache keyed by address. */
vt_status vt_fp4_destroy(vt_fp4_handle W);

/* Shape and format of a handle. */
vt_status vt_fp4_shape(vt_fp4_handle W, vt_fp4_format* fmt, int64_t* N, int64_t* K);

/* ----------------------------------------------------------------- the GEMM */

/* Bytes of workspace a GEMM on W with M <= M_max needs.  The workspace holds the
 * activations converted for the tensor cores, split-K partial sums, per-tile arrival
 * counters and a status word.  The caller zeroes it ONCE after allocation.  Each call's
 * activation pre-pass zeroes the counters it will use, so one workspace, large enough for
 * each of them, may serve calls on weights of any shape and any M in stream order.  A
 * workspace must not be used by two calls that may run at the same time. */
vt_status vt_fp4_workspace_bytes(vt_fp4_handle W, int64_t M_max, size_t* bytes);

/* C = A . W^T in bf16 with fp32 accumulation.
 *   A  (device) bf16 [M][lda], 16-byte aligned, lda >= K, lda % 8 == 0.
 *   C  (device) bf16 [M][ldc], 2-byte aligned, ldc >= N.
 *   M  tokens; M == 0 is a no-op.  M <= 16 runs the decode kernel, larger M the
 *      tensor-core tile kernel.
 *   workspace (device) >= vt_fp4_workspace_bytes(W, M), 256-byte aligned, zeroed once.
 * Deterministic: the same inputs and launch configuration give the same bits.
 * Asynchronous on `s`, no host synchronisation, capturable in a CUDA graph.
 * Source: "keep the ModelOpt NVFP4 lm_head packed" (PR #263), "Why this row matters":
 * the logits GEMM runs on the packed weight (W4A16), never on a bf16 expansion. */
vt_status vt_fp4_w4a16_gemm(const void* A, int64_t M, int64_t lda, vt_fp4_handle W, void* C,
                            int64_t ldc, void* workspace, size_t ws_bytes, vt_stream_t s);

/* As vt_fp4_w4a16_gemm with tuning overrides (NULL opts = defaults). */
vt_status vt_fp4_w4a16_gemm_ex(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                               void* C, int64_t ldc, void* workspace, size_t ws_bytes,
                               vt_stream_t s, const vt_fp4_gemm_opts* opts);

/* The input of the down projection from a paired gate_up weight (from
 * vt_fp4_prepack_gate_up_paired): C[m][i] = bf16( silu(g) * u ), g and u the fp32 sums of
 * gate row i and up row i times their globals, silu(x) = x / (1 + e^-x) in fp32 -- the
 * gate_up GEMM and the SiLU-and-multiply step in one call, without writing the [M][2I]
 * intermediate.  Any M >= 0 (the decode path for M <= 16, the tile path above).
 *   C  (device) bf16 [M][ldc], ldc >= I, 2-byte aligned.
 * Other arguments as for vt_fp4_w4a16_gemm.  A weight not prepacked paired is rejected
 * with VT_ERR_INVALID_ARG. */
vt_status vt_fp4_w4a16_gemm_silu_mul(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                                     void* C, int64_t ldc, void* workspace, size_t ws_bytes,
                                     vt_stream_t s);

/* Mixture-of-experts (grouped) weights: E experts of the same N x K, prepacked one after
 * another as E independent packed weights (each with its own global scale, or MXFP4 scale
 * window).  Source: "keep the ModelOpt NVFP4 lm_head packed" (PR #263), "Why this row
 * matters" (the MoE shared experts are FP4 linear layers too) and "dense projections take
 * vLLM's own dense marlin" (the multi-expert route of the same W4A16 GEMM).
 *   codes   (device) u8 [E][N][K/2];  scales (device) u8 [E][N][K/g];
 *   globals (host)   fp32 [E]: NVFP4 multipliers (> 0), MXFP4 1.0f.
 * vt_fp4_prepack_grouped_bytes gives the buffer size (E x vt_fp4_prepack_bytes).  unpack
 * and dequant write [E][N][...] in expert order; the plain GEMM entry points reject a
 * grouped handle. */
vt_status vt_fp4_prepack_grouped_bytes(vt_fp4_format fmt, int64_t E, int64_t N, int64_t K,
                                       size_t* packed_bytes);
vt_status vt_fp4_prepack_grouped(const uint8_t* codes, const uint8_t* scales,
                                 const float* globals, vt_fp4_format fmt, int64_t E, int64_t N,
                                 int64_t K, void* packed_dst, size_t dst_bytes, vt_stream_t s,
                                 vt_fp4_handle* out);

/* Workspace bytes of vt_fp4_w4a16_gemm_moe for up to M_max (<= 16) tokens of topk (<= 8)
 * experts each; zeroed once by the caller, reusable afterwards. */
vt_status vt_fp4_moe_workspace_bytes(vt_fp4_handle W, int64_t M_max, int64_t topk,
                                     size_t* bytes);

/* Mixture-of-experts decode GEMM (M <= 16): for every token m and slot j,
 *   C[m * topk + j][n] = sum_k A[m][k] * W_e[n][k],  e = topk_ids[m * topk + j],
 * in one call.  The (m, j) pairs are grouped by expert on the device (each expert in use is
 * streamed once, however many tokens chose it), in increasing expert order with pairs in
 * increasing order, so results do not depend on the routing's order; one decode kernel runs
 * every expert's problem.  Up to 8 tokens whose converted activations fit 64 KB (8 rows x K
 * f16 plus their scales: K <= 3968) take one launch, the decode kernel grouping the pairs
 * and converting A itself; otherwise a pre-pass on the stream does both first.
 *   topk_ids (device) int32 [M][topk], 1 <= topk <= 8; C (device) bf16 [M*topk][ldc].
 * A pair whose expert id is outside [0, E) is skipped (its C row is not written) and the
 * workspace status word reads 6.  Each token's ids should be distinct: an expert serves at
 * most 8 pairs when M <= 8 (16 when M > 8), so pairs beyond that -- possible only when a
 * token names an expert more than once -- are skipped the same way (status 6). */
vt_status vt_fp4_w4a16_gemm_moe(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                                const int32_t* topk_ids, int64_t topk, void* C, int64_t ldc,
                                void* workspace, size_t ws_bytes, vt_stream_t s);

/* Greedy head: the decode GEMM (M <= 16) that keeps, per token m, only the index of the
 * largest output, instead of writing the M x N outputs.  Source: "re-verify 27B NVFP4 on
 * the nvidia ModelOpt checkpoint" (PR #178), "Correctness -- resolved, not fixed": greedy
 * sampling takes the argmax with ties broken by the lowest index; "Speed -- warp-shuffle
 * MoE router top-k": under that total order every reduction order gives the same
 * (value, index).
 *   A, M, lda, W, workspace, ws_bytes, s  as for vt_fp4_w4a16_gemm (1 <= M <= 16).
 *   token  (device) int32 [M]: argmax over n of the bf16 output y[m][n] that
 *          vt_fp4_w4a16_gemm would write with the same workspace; equal values -> the
 *          lowest n; -0 equals +0; a NaN output counts as larger than every number.
 *   value  (device, optional, may be NULL) fp32 [M]: that bf16 output value.
 * N must fit in int32.  The workspace's first 256 bytes hold the per-token keys between
 * the kernel's CTAs; they are back to zero when the call completes. */
vt_status vt_fp4_w4a16_gemm_greedy(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                                   int32_t* token, float* value, void* workspace,
                                   size_t ws_bytes, vt_stream_t s);

/* The decode GEMM (M <= 16) without a caller workspace, for callers that cannot allocate
 * device memory: a host program whose HBM belongs to another allocator (a serving engine
 * that reserves memory up front, a plugin whose host forbids foreign allocations) or a
 * call path that must not depend on a runtime allocation.  The pages have no counterpart
 * of this entry point; it exists for such callers only.
 *   A, M, lda, W, C, ldc, s  as for vt_fp4_w4a16_gemm (M <= 16; M == 0 is a no-op); the
 *   launch shape is the one vt_fp4_w4a16_gemm chooses.  A grouped weight is rejected with
 *   VT_ERR_INVALID_ARG, K > 110000 with VT_ERR_UNSUPPORTED.
 * It uses one scratch area of 4 MiB inside the library's device image instead of a
 * workspace; every GPU that loads the library holds that area until the process exits.
 * A weight and M whose scratch needs exceed it are rejected with VT_ERR_UNSUPPORTED.
 * It allocates nothing: no cudaMalloc, no cudaFree.  The first call on a device looks up
 * the scratch area's device address (with that device current), so make that first call
 * before any stream capture.  Every call shares the same area and clears its split-K
 * counters on the stream first: calls that may overlap on the GPU (other streams, other
 * threads) race and must not be issued.  A bounded device-side wait that gives up records
 * VT_ERR_TIMEOUT in the area's status word, which stays set until vt_fp4_noalloc_status
 * reads it. */
vt_status vt_fp4_w4a16_gemm_noalloc(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                                    void* C, int64_t ldc, vt_stream_t s);

/* The status word of the no-alloc scratch area on the current device (synchronises `s`):
 * *status = VT_OK, or VT_ERR_TIMEOUT if a bounded wait of an earlier
 * vt_fp4_w4a16_gemm_noalloc call gave up (that call's output is then undefined); the word
 * is then cleared.  No counterpart on the pages (see vt_fp4_w4a16_gemm_noalloc). */
vt_status vt_fp4_noalloc_status(vt_stream_t s, int* status);

/* Test hook of vt_fp4_w4a16_gemm_noalloc, whose signature has no options: for the calls
 * made after it, every bounded device-side wait gives up after wait_limit_us microseconds
 * (0 = the 2 s default), and a nonzero withhold_weights stops the weight producer from
 * issuing copies, as vt_fp4_gemm_opts does for the workspace entry points.  Process-wide;
 * (0, 0) restores the defaults.  No counterpart on the pages. */
vt_status vt_fp4_noalloc_test_hooks(int wait_limit_us, int withhold_weights);

/* Reads the workspace status word (synchronises `s`): *status = VT_OK, VT_ERR_TIMEOUT if
 * a bounded device-side wait gave up during an earlier call, or 6 if a grouped call
 * skipped pairs (vt_fp4_w4a16_gemm_moe); the word is then cleared.
 * After VT_ERR_TIMEOUT zero the whole workspace again before reusing it: a call that gave up
 * may leave split-K arrival counts behind. */
vt_status vt_fp4_workspace_status(void* workspace, vt_stream_t s, int* status);

/* Host-side record of the last GEMM launched on W. */
vt_status vt_fp4_stats(vt_fp4_handle W, vt_fp4_launch_info* info);

/* -------------------------------------------------------------------- W4A4 */

/* The W4A4 arm: C = Q(A) . W^T with Q the activation quantiser below (activations in the
 * weight's block format), fp32 accumulation, bf16 output.  NVFP4: input_scale is the
 * per-tensor activation global (the checkpoint's input_scale, a multiplier like the
 * weight's global), a positive normal float; MXFP4: input_scale must be 1.0f.  Source:
 * "re-verify 27B NVFP4 on the nvidia ModelOpt checkpoint" (PR #178), section "W4A16 is
 * the default for ModelOpt" (consuming input_scale makes the layer true W4A4 and routes
 * it to the fp4-activation GEMM; the W4A16 arm stays the default); "native MXFP4
 * keep-quant + Qwen e2e" (PR #38), commit "W0" (MXFP4 activations, group 32).  The
 * quantised activations are held as their exact dequantised values in f16 and multiplied
 * on the same tensor-core paths as vt_fp4_w4a16_gemm (decode M <= 16, tile kernel above).
 * A group of activations holding an inf or NaN yields NaN outputs for its tokens.
 * Arguments, workspace, determinism and errors as vt_fp4_w4a16_gemm; a bad input_scale
 * is VT_ERR_INVALID_ARG. */
vt_status vt_fp4_w4a4_gemm(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                           float input_scale, void* C, int64_t ldc, void* workspace,
                           size_t ws_bytes, vt_stream_t s);

/* As vt_fp4_w4a4_gemm with tuning overrides (NULL opts = defaults). */
vt_status vt_fp4_w4a4_gemm_ex(const void* A, int64_t M, int64_t lda, vt_fp4_handle W,
                              float input_scale, void* C, int64_t ldc, void* workspace,
                              size_t ws_bytes, vt_stream_t s, const vt_fp4_gemm_opts* opts);

/* The W4A4 activation quantiser on its own: A (device) bf16 [M][lda] (16-byte aligned,
 * lda % 8 == 0, lda >= K, K % g == 0) -> codes (device, 16-byte aligned) u8 [M][K/2]
 * (low nibble = even k) and scales (device) u8 [M][K/g].  Decisions in fp32, round to
 * nearest even, saturating:
 *   NVFP4: s = E4M3(amax_g / fl32(6 input_scale)); code = E2M1(x / fl32(s input_scale))
 *          (all codes 0 when s = 0)
 *   MXFP4: e = min{e : 6 2^e >= amax_g} in [-127, 127], byte e + 127; code = E2M1(x 2^-e)
 * A group holding an inf or NaN gets the NaN scale byte (0x7F E4M3, 0xFF E8M0) and zero
 * codes.  Asynchronous on `s`. */
vt_status vt_fp4_quantize_act(const void* A, int64_t M, int64_t lda, int64_t K,
                              vt_fp4_format fmt, float input_scale, uint8_t* codes,
                              uint8_t* scales, vt_stream_t s);

/* ------------------------------------------------------------ debug / tests */

/* out (device) fp32 [N][K]: the dequantised weight as the kernels see it,
 * NVFP4 fl32(e2m1*e4m3*global) (e2m1*e4m3 is exact), MXFP4 fl32(e2m1*2^(e-127)) (exact for
 * every scale byte 0x00..0xFE, inf where 6 * 2^127 exceeds fp32; 0xFF gives NaN).  A weight
 * whose finite MXFP4 scale bytes span at most 30 exponents keeps them in the tiles as f16
 * powers of two relative to the largest; a wider span keeps the raw bytes and the kernels
 * apply each group's scale in fp32 (the decode kernel) or as exact bf16 tiles (the
 * tensor-core path); both hold every weight exactly. */
vt_status vt_fp4_dequant(vt_fp4_handle W, float* out, vt_stream_t s);

/* Inverse of the prepack: codes (device) u8 [N][K/2] and scales (device) u8 [N][K/g] in
 * the input layout, recovered from the packed buffer. */
vt_status vt_fp4_unpack(vt_fp4_handle W, uint8_t* codes, uint8_t* scales, vt_stream_t s);

/* ------------------------------------------------------------- quantiser */

/* Quantises a bf16 weight [N][K] (device, row-major, 16-byte aligned, K % g == 0) into
 * codes [N][K/2] and scales [N][K/g] (device) with the synthetic-weight recipe:
 *   NVFP4: G = fl32(amax/(6*448)); s = E4M3_RNE_sat(amax_g/(6G)); code = E2M1_RNE(w/(s G))
 *   MXFP4: e = min{e : 2^e >= amax_g/6}; code = E2M1_RNE(w / 2^e)
 * (quotients in fp64, ties to even, saturating).  NVFP4 writes G to *global_out
 * (device, 4 bytes; MXFP4 ignores it).  `scratch` (device, >= 16 bytes, 16-aligned) is
 * overwritten. */
vt_status vt_fp4_quantize(const void* W, int64_t N, int64_t K, vt_fp4_format fmt,
                          uint8_t* codes, uint8_t* scales, float* global_out, void* scratch,
                          vt_stream_t s);

/* Message for the last failing call on this thread ("" if none). */
const char* vt_fp4_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* VT_FP4_H */
