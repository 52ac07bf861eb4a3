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
}  // namespace vt
