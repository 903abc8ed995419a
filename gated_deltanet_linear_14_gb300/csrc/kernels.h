// Launchers implemented by the kernel translation units (internal).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace gdn {

// SMs of the current device.
int device_sms();

cudaError_t launch_conv(const Geom& G, const Batch& B, const Params& P, int io_bf16, int y_f32,
                        const void* x, const void* w, void* y, void* pages, int32_t* status,
                        cudaStream_t stream);

cudaError_t launch_conv_slots(const Geom& G, const Batch& B, const Params& P, const SlotGeom& SG,
                              int io_bf16, const void* x, const void* w, void* y, void* slots,
                              int32_t* status, cudaStream_t stream);


// Chunked prefill on the tensor cores; tmap points to the CUtensorMap of
// the packed qkv rows ([num_rows][C] bf16, box 64 x 64, 128B swizzle).
cudaError_t launch_chunk(const void* tmap, const Geom& G, const Batch& B, const Params& P,
                         int state_bf16, int out_f32, const void* a, const void* b, void* o,
                         void* pages, int32_t* status, cudaStream_t stream);

// The two-pass form (chunk2.cu): a pre-pass per (request, value head, chunk)
// writes one workspace item each, then the chain per (request, value head)
// reads them. Item (r, h, c) sits at ((r * Hv + h) * ws_chunks + c) *
// kChunkItemBytes; ws_chunks >= ceil(max_rows / 64). Item layout (bytes):
//   CW_WT   W^T hi | Q^T | W^T lo: [128][64] bf16 each, 128B-swizzled
//           operand tiles (Q^T is exact in bf16), one 48 KiB block
//   CW_P    P hi | lo, [64][64] bf16 each, the same layout
//   CW_UT   U^T fp32 [128][64]: 4-float piece q of row j's half h at
//           ((h * 8 + q) * 128 + j) * 16
//   CW_VEC  e^{gamma_L-gamma}/|k| [64] | e^gamma/|q| [64] | e^{gamma_L} (768 B)
constexpr uint32_t CW_WT = 0, CW_P = 49152, CW_UT = 65536, CW_VEC = 98304;
constexpr size_t kChunkItemBytes = 99328;
cudaError_t launch_chunk2(const void* tmap, const Geom& G, const Batch& B, const Params& P,
                          int state_bf16, int out_f32, const void* a, const void* b, void* o,
                          void* pages, void* ws, int ws_chunks, int32_t* status,
                          cudaStream_t stream);

// Fused conv + rule for one token per request (plain requests).
cudaError_t launch_decode(const Geom& G, const Batch& B, const Params& P, int io_bf16,
                          int state_bf16, int out_f32, const void* x, const void* w, const void* a,
                          const void* b, void* o, void* pages, int32_t* status,
                          cudaStream_t stream);

// Page <-> slot pool hand-over (handover.cu). dir 0: page -> slot 0,
// dir 1: slot slot[i] -> page.
cudaError_t launch_handover(const Geom& G, const SlotGeom& SG, int dir, int n, const int32_t* page,
                            const int32_t* pool, const int32_t* slot, int num_pages,
                            int num_pools, void* pages, void* slots, size_t state_bytes,
                            size_t window_bytes, int32_t* status, cudaStream_t stream);

// Speculative decode in closed form (spec.cuh). mode: 0 = one-page verify
// (rows = conv'd qkv), 1 = the same with the conv fused in (rows = raw x),
// 2 = slot-per-candidate layout (rows = conv'd qkv, pages = slot pools).
// Mode 0 launches two kernels (run coefficients, then items); modes 1 and 2
// one. splits: CTAs per (request, q/k head) of mode 2.
cudaError_t launch_spec_d32(int mode, const Geom&, const Batch&, const Params&, const SlotGeom&,
                            int, int, int, const void*, const void*, const void*, const void*,
                            void*, void*, int32_t*, int, cudaStream_t);
cudaError_t launch_spec_d64(int mode, const Geom&, const Batch&, const Params&, const SlotGeom&,
                            int, int, int, const void*, const void*, const void*, const void*,
                            void*, void*, int32_t*, int, cudaStream_t);
cudaError_t launch_spec_d128(int mode, const Geom&, const Batch&, const Params&, const SlotGeom&,
                             int, int, int, const void*, const void*, const void*, const void*,
                             void*, void*, int32_t*, int, cudaStream_t);

// Token-by-token rule (rule.cuh) for the plain requests of a batch, per head
// dimension (one translation unit each).
cudaError_t launch_rule_d32(const Geom&, const Batch&, const Params&, int io_bf16, int state_bf16,
                            int out_f32, const void* qkv, const void* a, const void* b, void* o,
                            void* pages, int32_t* status, cudaStream_t);
cudaError_t launch_rule_d64(const Geom&, const Batch&, const Params&, int io_bf16, int state_bf16,
                            int out_f32, const void* qkv, const void* a, const void* b, void* o,
                            void* pages, int32_t* status, cudaStream_t);
cudaError_t launch_rule_d128(const Geom&, const Batch&, const Params&, int io_bf16, int state_bf16,
                             int out_f32, const void* qkv, const void* a, const void* b, void* o,
                             void* pages, int32_t* status, cudaStream_t);

}  // namespace gdn
