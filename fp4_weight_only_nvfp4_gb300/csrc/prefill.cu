// Prefill tile GEMM (M > 16): placeholder until the tensor-core tile kernel lands.
#include "common.cuh"
#include "kernels.h"

namespace vt {

cudaError_t launch_prefill(const PrefillLaunch&, cudaStream_t, int* launches, int* grid_out,
                           int64_t* tiles_out) {
  if (launches) *launches = 0;
  if (grid_out) *grid_out = 0;
  if (tiles_out) *tiles_out = 0;
  return cudaErrorNotSupported;
}

}  // namespace vt
