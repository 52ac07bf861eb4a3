// Internal: the host-side state behind a vt_fp4_handle, shared by the C ABI files.
#pragma once
#include <stddef.h>
#include <stdint.h>

#include "vt_fp4.h"

struct vt_fp4_weight_s {
  int fmt;
  int64_t N, K, RT, KT;
  int64_t seg_split;
  int layout;  // kLayoutRows or kLayoutPaired
  int64_t E = 1;             // experts (grouped weight); 1 otherwise
  int64_t expert_bytes = 0;  // grouped: bytes of one expert's packed weight
  const void* packed;
  size_t packed_bytes;
  vt_fp4_launch_info info;
};

namespace vt {
// Records the message returned by vt_fp4_last_error() for this thread; returns st.
vt_status set_last_error(vt_status st, const char* msg);

// Multiprocessors of the current device (cached per device).
int sm_count();

// Launch shape of the decode GEMM (M <= 16) on W: k tiles per pipeline stage, ring depth, CTAs
// and whether the kernel converts the activations itself (resident mode).  `opts` may be NULL
// (library choice); w4a4 calls always take the activation pre-pass.  Shared by every decode
// entry point so that they launch the same shapes.
struct DecodeShape {
  int ks, stages, grid, resident, epi;
};
vt_status decode_shape(const vt_fp4_weight_s* W, int M, const vt_fp4_gemm_opts* opts, bool w4a4,
                       DecodeShape* out);
}  // namespace vt
