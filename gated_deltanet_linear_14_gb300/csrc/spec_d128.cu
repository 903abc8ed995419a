// Closed-form speculative kernels for head dimension 128 (see spec.cuh).
#include "kernels.h"
#include "spec.cuh"

namespace gdn {

cudaError_t launch_spec_d128(int mode, const Geom& G, const Batch& B, const Params& P,
                           const SlotGeom& SG, int io_bf16, int state_bf16, int out_f32,
                           const void* rows, const void* conv_w, const void* a, const void* b,
                           void* o, void* pages, int32_t* status, int splits,
                           cudaStream_t stream) {
  return launch_spec_dk<128>(mode, G, B, P, SG, io_bf16, state_bf16, out_f32, rows, conv_w, a, b,
                           o, pages, status, splits, stream);
}

}  // namespace gdn
