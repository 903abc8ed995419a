// Token-by-token rule kernels for head dimension 128 (see rule.cuh).
#include "kernels.h"
#include "rule.cuh"

namespace gdn {

cudaError_t launch_rule_d128(const Geom& G, const Batch& B, const Params& P, int io_bf16,
                           int state_bf16, int out_f32, const void* qkv, const void* a,
                           const void* b, void* o, void* pages, int32_t* status,
                           cudaStream_t stream) {
  return launch_rule_dk<128>(G, B, P, io_bf16, state_bf16, out_f32, qkv, a, b, o, pages, status,
                           stream);
}

}  // namespace gdn
