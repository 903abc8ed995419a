// C ABI of the GDN layer core: host-side validation, layouts and launches.
// Every entry point checks its arguments completely before launching, so a
// negative return means nothing was launched and nothing was written.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "gdn.h"
#include "kernels.h"
#include "spec.cuh"
#include "umma.cuh"

namespace gdn {

// One thread waits on an mbarrier that nothing arrives at; the bounded wait
// gives up after limit_ns and the kernel reports GDN_DEV_TIMEOUT, the path
// every kernel takes when one of its own copies or MMAs does not complete.
__global__ void wait_check_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = umma::smem_u32(&bar);
    umma::mbar_init(b, 1);
    umma::mbar_fence_init();
    if (!umma::mbar_wait(b, 0, limit_ns)) report(status, GDN_DEV_TIMEOUT);
  }
}

// SMs of the current device (looked up once per device; declared in kernels.h).
int device_sms() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev < 0 || dev >= 64) return 152;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    sms[dev] = n;
  }
  return sms[dev];
}

}  // namespace gdn

namespace {

using namespace gdn;

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline size_t dsize(int32_t dt) { return dt == GDN_BF16 ? 2 : 4; }
inline bool valid_dtype(int32_t dt) { return dt == GDN_F32 || dt == GDN_BF16; }

gdn_status check_dims(const gdn_dims* d) {
  if (!d) return GDN_ERR_INVALID_ARG;
  if (d->num_k_heads <= 0 || d->num_v_heads <= 0 || d->head_k_dim <= 0 || d->head_v_dim <= 0 ||
      d->conv_width <= 0 || d->max_candidates < 0)
    return GDN_ERR_INVALID_ARG;
  if (!valid_dtype(d->io_dtype) || !valid_dtype(d->state_dtype) || !valid_dtype(d->out_dtype))
    return GDN_ERR_INVALID_ARG;
  if (d->num_v_heads % d->num_k_heads != 0) return GDN_ERR_UNSUPPORTED;
  if (d->head_k_dim != d->head_v_dim) return GDN_ERR_UNSUPPORTED;
  if (d->head_k_dim != 32 && d->head_k_dim != 64 && d->head_k_dim != 128) return GDN_ERR_UNSUPPORTED;
  if (d->conv_width != 4) return GDN_ERR_UNSUPPORTED;
  if (d->max_candidates > 8) return GDN_ERR_UNSUPPORTED;
  if (d->num_v_heads > 4096 || d->num_k_heads > 4096) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

void layout(const gdn_dims* d, gdn_page_layout_t* L, int* rec_row_elems) {
  const size_t C = 2 * (size_t)d->num_k_heads * d->head_k_dim + (size_t)d->num_v_heads * d->head_v_dim;
  const size_t io = dsize(d->io_dtype), st = dsize(d->state_dtype);
  const size_t rec_row = align_up((C + 2 * (size_t)d->num_v_heads) * io, 16) / io;
  std::memset(L, 0, sizeof(*L));
  L->state_offset = 0;
  L->state_bytes = (size_t)d->num_v_heads * d->head_v_dim * d->head_k_dim * st;
  L->window_offset = align_up(L->state_offset + L->state_bytes, kAlign);
  L->window_bytes = (size_t)(d->conv_width - 1 + d->max_candidates) * C * io;
  L->record_offset = align_up(L->window_offset + L->window_bytes, kAlign);
  // both slots' rows, then both slots' run coefficients (fp32, one block of
  // kRunCoefBytes per value head and slot), then the live slot's u (fp32, per
  // value head, candidate and value column; a step reads it before it
  // writes its candidates' u there)
  L->record_bytes = 2 * (size_t)d->max_candidates * rec_row * io +
                    (d->max_candidates > 0 ? 2 * (size_t)d->num_v_heads * kRunCoefBytes : 0) +
                    (size_t)d->num_v_heads * d->max_candidates * d->head_v_dim * 4;
  L->flag_offset = align_up(L->record_offset + L->record_bytes, kAlign);
  L->page_bytes = align_up(L->flag_offset + sizeof(uint32_t), kAlign);
  if (rec_row_elems) *rec_row_elems = (int)rec_row;
}

void slot_layout(const gdn_dims* d, gdn_slot_layout_t* S) {
  const size_t C = 2 * (size_t)d->num_k_heads * d->head_k_dim + (size_t)d->num_v_heads * d->head_v_dim;
  const size_t state_bytes =
      (size_t)d->num_v_heads * d->head_v_dim * d->head_k_dim * dsize(d->state_dtype);
  const size_t window_bytes = (size_t)(d->conv_width - 1) * C * dsize(d->io_dtype);
  S->state_offset = 0;
  S->window_offset = align_up(state_bytes, kAlign);
  S->slot_bytes = align_up(S->window_offset + window_bytes, kAlign);
  S->pool_bytes = S->slot_bytes * (size_t)(d->max_candidates > 0 ? d->max_candidates : 1);
}

Geom make_geom(const gdn_dims* d) {
  gdn_page_layout_t L;
  int rec_row = 0;
  layout(d, &L, &rec_row);
  Geom G;
  G.Hk = d->num_k_heads;
  G.Hv = d->num_v_heads;
  G.Dk = d->head_k_dim;
  G.Dv = d->head_v_dim;
  G.W = d->conv_width;
  G.Kc = d->max_candidates;
  G.C = 2 * G.Hk * G.Dk + G.Hv * G.Dv;
  G.rec_row = rec_row;
  G.page_bytes = L.page_bytes;
  G.window_off = L.window_offset;
  G.state_off = L.state_offset;
  G.record_off = L.record_offset;
  G.rcoef_off = L.record_offset + 2 * (size_t)d->max_candidates * rec_row * dsize(d->io_dtype);
  G.ru_off = G.rcoef_off + (d->max_candidates > 0 ? 2 * (size_t)d->num_v_heads * kRunCoefBytes : 0);
  G.flag_off = L.flag_offset;
  return G;
}

gdn_status check_batch(const gdn_batch* b, bool accepted_may_be_null) {
  if (!b) return GDN_ERR_INVALID_ARG;
  if (b->num_requests < 0 || b->num_rows < 0 || b->max_rows < 0 || b->num_pages < 0)
    return GDN_ERR_INVALID_ARG;
  if (b->num_requests > 65535) return GDN_ERR_UNSUPPORTED;
  if (b->num_requests > 0 && (!b->row_start || !b->row_len || !b->page || !b->flags))
    return GDN_ERR_INVALID_ARG;
  if (!accepted_may_be_null && b->num_requests > 0 && !b->n_accepted) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

gdn_status check_params(const gdn_params* p, bool need_gates) {
  if (!p) return GDN_ERR_INVALID_ARG;
  if (need_gates && (!p->A_log || !p->dt_bias)) return GDN_ERR_INVALID_ARG;
  if (p->gate_mode != 0 && p->gate_mode != 1) return GDN_ERR_INVALID_ARG;
  if (!(p->norm_eps >= 0.0f) || !std::isfinite(p->norm_eps)) return GDN_ERR_INVALID_ARG;
  if (std::isnan(p->scale)) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

Batch make_batch(const gdn_batch* b) {
  Batch B;
  B.R = b->num_requests;
  B.num_rows = b->num_rows;
  B.max_rows = b->max_rows;
  B.num_pages = b->num_pages;
  B.row_start = b->row_start;
  B.row_len = b->row_len;
  B.page = b->page;
  B.flags = b->flags;
  B.n_accepted = b->n_accepted;
  B.order = b->order;
  B.min_len = 0;
  B.max_len = 0x7fffffff;
  return B;
}

Params make_params(const gdn_params* p, const gdn_dims* d) {
  Params P;
  P.A_log = p->A_log;
  P.dt_bias = p->dt_bias;
  P.conv_bias = p->conv_bias;
  P.scale = (p->scale > 0.0f) ? p->scale : 1.0f / std::sqrt((float)d->head_k_dim);
  P.eps = p->norm_eps;
  P.gate_mode = p->gate_mode;
  return P;
}

cudaError_t rule(const Geom& G, const Batch& B, const Params& P, const gdn_dims* d,
                 const void* qkv, const void* a, const void* b, void* o, void* pages,
                 int32_t* status, cudaStream_t s) {
  const int io = d->io_dtype == GDN_BF16, st = d->state_dtype == GDN_BF16,
            of = d->out_dtype == GDN_F32;
  switch (d->head_k_dim) {
    case 32: return launch_rule_d32(G, B, P, io, st, of, qkv, a, b, o, pages, status, s);
    case 64: return launch_rule_d64(G, B, P, io, st, of, qkv, a, b, o, pages, status, s);
    default: return launch_rule_d128(G, B, P, io, st, of, qkv, a, b, o, pages, status, s);
  }
}

// CTAs per (request, q/k head) for the slot-layout kernel: one unless the
// batch would leave SMs idle; then the group's items are split in halves (as
// long as they divide evenly) until there are three CTAs per SM. (The
// one-page step's item kernel always runs one CTA per item.)
int spec_splits(const gdn_dims* d, int R, int mode) {
  if (mode != SPEC_SLOTS) return 1;
  const int Gh = d->num_v_heads / d->num_k_heads;
  const int bvi = d->head_v_dim < kSpecBV ? d->head_v_dim : kSpecBV;
  const int items = Gh * (d->head_v_dim / bvi);
  const long long ctas = (long long)d->num_k_heads * R;
  const long long want = 3LL * device_sms();
  int s = 1;
  while (ctas * s < want && items % (2 * s) == 0) s *= 2;
  return s;
}

// The shared memory the entry point's spec kernels need fits (else the
// shape is not supported: a very wide group of value heads).
bool spec_fits(const gdn_dims* d, int mode) {
  const int Gh = d->num_v_heads / d->num_k_heads;
  return (int)spec_smem_need(mode, d->head_k_dim, Gh, (int)dsize(d->io_dtype),
                             (int)dsize(d->state_dtype)) <= kSpecSmemMax;
}

cudaError_t spec(int mode, const Geom& G, const Batch& B, const Params& P, const SlotGeom& SG,
                 const gdn_dims* d, const void* rows, const void* conv_w, const void* a,
                 const void* b, void* o, void* pages, int32_t* status, cudaStream_t s) {
  const int io = d->io_dtype == GDN_BF16, st = d->state_dtype == GDN_BF16,
            of = d->out_dtype == GDN_F32;
  const int splits = spec_splits(d, B.R, mode);
  switch (d->head_k_dim) {
    case 32:
      return launch_spec_d32(mode, G, B, P, SG, io, st, of, rows, conv_w, a, b, o, pages, status,
                             splits, s);
    case 64:
      return launch_spec_d64(mode, G, B, P, SG, io, st, of, rows, conv_w, a, b, o, pages, status,
                             splits, s);
    default:
      return launch_spec_d128(mode, G, B, P, SG, io, st, of, rows, conv_w, a, b, o, pages, status,
                              splits, s);
  }
}

gdn_status seq_entry(const gdn_dims* dims, const gdn_batch* batch, const gdn_params* params,
                     const void* qkv, const void* a, const void* b, void* o, void* pages,
                     int32_t* status, gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if ((e = check_batch(batch, true)) != GDN_OK) return e;
  if ((e = check_params(params, true)) != GDN_OK) return e;
  if (batch->num_requests == 0) return GDN_OK;
  if (!status || !pages) return GDN_ERR_INVALID_ARG;
  if (batch->num_rows > 0 && (!qkv || !a || !b || !o)) return GDN_ERR_INVALID_ARG;
  const Geom G = make_geom(dims);
  const Batch B = make_batch(batch);
  const Params P = make_params(params, dims);
  if (rule(G, B, P, dims, qkv, a, b, o, pages, status, (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no link-time
// dependency on libcuda). The only process-wide value the library keeps.
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// TMA descriptor of the packed rows [num_rows][C] bf16: boxes of 64 rows x
// 64 channels (128 bytes), 128-byte swizzle, zero fill past the last row.
gdn_status encode_rows_tmap(CUtensorMap* tm, const void* rows, int num_rows, const gdn_dims* d) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return GDN_ERR_NO_DEVICE;
  const cuuint64_t C = 2 * (cuuint64_t)d->num_k_heads * d->head_k_dim +
                       (cuuint64_t)d->num_v_heads * d->head_v_dim;
  cuuint64_t gdim[2] = {C, (cuuint64_t)num_rows};
  cuuint64_t gstride[1] = {C * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estride[2] = {1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(rows), gdim,
                         gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GDN_OK : GDN_ERR_UNSUPPORTED;
}

gdn_status handover_entry(int dir, const gdn_dims* dims, int32_t n, const int32_t* page,
                          const int32_t* pool, const int32_t* slot, int32_t num_pages,
                          int32_t num_pools, void* pages, void* slots, int32_t* status,
                          gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if (dims->max_candidates == 0) return GDN_ERR_UNSUPPORTED;
  if (n < 0 || num_pages < 0 || num_pools < 0) return GDN_ERR_INVALID_ARG;
  if (n > 65535) return GDN_ERR_UNSUPPORTED;
  if (n == 0) return GDN_OK;
  if (!page || !pool || (dir == 1 && !slot) || !pages || !slots || !status)
    return GDN_ERR_INVALID_ARG;
  const Geom G = make_geom(dims);
  gdn_slot_layout_t SL;
  slot_layout(dims, &SL);
  const SlotGeom SG{SL.pool_bytes, SL.slot_bytes, SL.state_offset, SL.window_offset};
  const size_t C = (size_t)G.C;
  const size_t state_bytes = (size_t)G.Hv * G.Dv * G.Dk * dsize(dims->state_dtype);
  const size_t window_bytes = (size_t)(G.W - 1) * C * dsize(dims->io_dtype);
  if (launch_handover(G, SG, dir, n, page, pool, slot, num_pages, num_pools, pages, slots,
                      state_bytes, window_bytes, status, (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

}  // namespace

// Scratch of gdn_chunk_prefill_noalloc: one array per device, part of the
// library's device image (every device that loads this module holds it until
// the process exits). Its size bounds the batches that entry point takes.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_chunk_scratch[kNoAllocScratchBytes];

namespace {

// The array's device address, looked up once per device (with that device
// current) and kept; nullptr and the runtime's error if the lookup fails.
cudaError_t chunk_scratch_address(void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_chunk_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

int32_t gdn_abi_version(void) { return (2 << 16) | 1; }

gdn_status gdn_page_layout(const gdn_dims* dims, gdn_page_layout_t* out) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if (!out) return GDN_ERR_INVALID_ARG;
  layout(dims, out, nullptr);
  return GDN_OK;
}

gdn_status gdn_slot_layout(const gdn_dims* dims, gdn_slot_layout_t* out) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if (!out) return GDN_ERR_INVALID_ARG;
  slot_layout(dims, out);
  return GDN_OK;
}

gdn_status gdn_conv(const gdn_dims* dims, const gdn_batch* batch, const gdn_params* params,
                    const void* x, const void* conv_w, void* y, int32_t y_dtype, void* pages,
                    int32_t* status, gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if ((e = check_batch(batch, true)) != GDN_OK) return e;
  if ((e = check_params(params, false)) != GDN_OK) return e;
  if (!valid_dtype(y_dtype)) return GDN_ERR_INVALID_ARG;
  if (y_dtype != GDN_F32 && y_dtype != dims->io_dtype) return GDN_ERR_UNSUPPORTED;
  if (batch->num_requests == 0) return GDN_OK;
  if (!status || !pages || !conv_w) return GDN_ERR_INVALID_ARG;
  if (batch->num_rows > 0 && (!x || !y)) return GDN_ERR_INVALID_ARG;
  const Geom G = make_geom(dims);
  const Batch B = make_batch(batch);
  const Params P = make_params(params, dims);
  if (launch_conv(G, B, P, dims->io_dtype == GDN_BF16, y_dtype == GDN_F32, x, conv_w, y, pages,
                  status, (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

gdn_status gdn_seq(const gdn_dims* dims, const gdn_batch* batch, const gdn_params* params,
                   const void* qkv, const void* a, const void* b, void* o, void* pages,
                   int32_t* status, gdn_stream_t stream) {
  return seq_entry(dims, batch, params, qkv, a, b, o, pages, status, stream);
}

gdn_status gdn_spec_verify(const gdn_dims* dims, const gdn_batch* batch, const gdn_params* params,
                           const void* qkv, const void* a, const void* b, void* o, void* pages,
                           int32_t* status, gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if ((e = check_batch(batch, false)) != GDN_OK) return e;
  if ((e = check_params(params, true)) != GDN_OK) return e;
  if (dims->max_candidates == 0) return GDN_ERR_UNSUPPORTED;
  if (!spec_fits(dims, SPEC_VERIFY)) return GDN_ERR_UNSUPPORTED;
  if (batch->num_requests == 0) return GDN_OK;
  if (!status || !pages) return GDN_ERR_INVALID_ARG;
  if (batch->num_rows > 0 && (!qkv || !a || !b || !o)) return GDN_ERR_INVALID_ARG;
  const Geom G = make_geom(dims);
  const Batch B = make_batch(batch);
  const Params P = make_params(params, dims);
  SlotGeom SG{};
  if (spec(SPEC_VERIFY, G, B, P, SG, dims, qkv, nullptr, a, b, o, pages, status,
           (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

gdn_status gdn_spec_step(const gdn_dims* dims, const gdn_batch* batch, const gdn_params* params,
                         const void* x, const void* conv_w, const void* a, const void* b, void* o,
                         void* pages, int32_t* status, gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if ((e = check_batch(batch, false)) != GDN_OK) return e;
  if ((e = check_params(params, true)) != GDN_OK) return e;
  if (dims->max_candidates == 0) return GDN_ERR_UNSUPPORTED;
  if (!spec_fits(dims, SPEC_FUSED)) return GDN_ERR_UNSUPPORTED;
  if (batch->num_requests == 0) return GDN_OK;
  if (!status || !pages || !conv_w) return GDN_ERR_INVALID_ARG;
  if (batch->num_rows > 0 && (!x || !a || !b || !o)) return GDN_ERR_INVALID_ARG;
  const Geom G = make_geom(dims);
  const Batch B = make_batch(batch);
  const Params P = make_params(params, dims);
  SlotGeom SG{};
  if (spec(SPEC_FUSED, G, B, P, SG, dims, x, conv_w, a, b, o, pages, status,
           (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

gdn_status gdn_spec_slots(const gdn_dims* dims, const gdn_batch* batch, const gdn_params* params,
                          const void* x, const void* conv_w, void* y, const void* a, const void* b,
                          void* o, void* slots, int32_t* status, gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if ((e = check_batch(batch, false)) != GDN_OK) return e;
  if ((e = check_params(params, true)) != GDN_OK) return e;
  if (dims->max_candidates == 0) return GDN_ERR_UNSUPPORTED;
  if (!spec_fits(dims, SPEC_SLOTS)) return GDN_ERR_UNSUPPORTED;
  if (batch->num_requests == 0) return GDN_OK;
  if (!status || !slots || !conv_w) return GDN_ERR_INVALID_ARG;
  if (batch->num_rows > 0 && (!x || !y || !a || !b || !o)) return GDN_ERR_INVALID_ARG;
  const Geom G = make_geom(dims);
  const Batch B = make_batch(batch);
  const Params P = make_params(params, dims);
  gdn_slot_layout_t SL;
  slot_layout(dims, &SL);
  SlotGeom SG{SL.pool_bytes, SL.slot_bytes, SL.state_offset, SL.window_offset};
  const cudaStream_t s = (cudaStream_t)stream;
  const int io = dims->io_dtype == GDN_BF16;
  if (launch_conv_slots(G, B, P, SG, io, x, conv_w, y, slots, status, s) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  if (spec(SPEC_SLOTS, G, B, P, SG, dims, y, nullptr, a, b, o, slots, status, s) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

gdn_status gdn_page_to_slots(const gdn_dims* dims, int32_t n, const int32_t* page,
                             const int32_t* pool, int32_t num_pages, int32_t num_pools,
                             const void* pages, void* slots, int32_t* status,
                             gdn_stream_t stream) {
  return handover_entry(0, dims, n, page, pool, nullptr, num_pages, num_pools,
                        const_cast<void*>(pages), slots, status, stream);
}

gdn_status gdn_slots_to_page(const gdn_dims* dims, int32_t n, const int32_t* pool,
                             const int32_t* slot, const int32_t* page, int32_t num_pools,
                             int32_t num_pages, const void* slots, void* pages, int32_t* status,
                             gdn_stream_t stream) {
  return handover_entry(1, dims, n, page, pool, slot, num_pages, num_pools, pages,
                        const_cast<void*>(slots), status, stream);
}

gdn_status gdn_decode(const gdn_dims* dims, const gdn_batch* batch, const gdn_params* params,
                      const void* x, const void* conv_w, const void* a, const void* b, void* o,
                      void* pages, int32_t* status, gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if ((e = check_batch(batch, true)) != GDN_OK) return e;
  if ((e = check_params(params, true)) != GDN_OK) return e;
  const int items = (dims->num_v_heads / dims->num_k_heads) * (dims->head_v_dim / 32);
  if (items > 16) return GDN_ERR_UNSUPPORTED;
  if (batch->max_rows > 1) return GDN_ERR_INVALID_ARG;
  if (batch->num_requests == 0) return GDN_OK;
  if (!status || !pages || !conv_w) return GDN_ERR_INVALID_ARG;
  if (batch->num_rows > 0 && (!x || !a || !b || !o)) return GDN_ERR_INVALID_ARG;
  const Geom G = make_geom(dims);
  const Batch B = make_batch(batch);
  const Params P = make_params(params, dims);
  if (launch_decode(G, B, P, dims->io_dtype == GDN_BF16, dims->state_dtype == GDN_BF16,
                    dims->out_dtype == GDN_F32, x, conv_w, a, b, o, pages, status,
                    (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

gdn_status gdn_prefill(const gdn_dims* dims, const gdn_batch* batch, const gdn_params* params,
                       const void* qkv, const void* a, const void* b, void* o, void* pages,
                       int32_t chunk_min_rows, void* workspace, size_t workspace_bytes,
                       int32_t* status, gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if ((e = check_batch(batch, true)) != GDN_OK) return e;
  if ((e = check_params(params, true)) != GDN_OK) return e;
  if (batch->num_requests == 0) return GDN_OK;
  if (!status || !pages) return GDN_ERR_INVALID_ARG;
  if (batch->num_rows > 0 && (!qkv || !a || !b || !o)) return GDN_ERR_INVALID_ARG;
  const int threshold = chunk_min_rows > 0 ? chunk_min_rows : GDN_PREFILL_CHUNK_MIN_ROWS;
  const bool chunk_ok = dims->io_dtype == GDN_BF16 && dims->head_k_dim == 128 &&
                        dims->head_v_dim == 128 && ((uintptr_t)qkv & 15) == 0;
  const bool any_long = chunk_ok && batch->max_rows >= threshold && batch->num_rows > 0;
  const Geom G = make_geom(dims);
  const Params P = make_params(params, dims);
  const cudaStream_t s = (cudaStream_t)stream;
  // the chunked launch's row map is encoded before anything is launched, so
  // that a failure to encode it still leaves nothing launched or written
  CUtensorMap tmap;
  std::memset(&tmap, 0, sizeof(tmap));
  size_t need = 0;
  if (any_long) {
    const gdn_status te = encode_rows_tmap(&tmap, qkv, batch->num_rows, dims);
    if (te != GDN_OK) return te;
    need = gdn_chunk_prefill_workspace_bytes(dims, batch);
    if (workspace && workspace_bytes < need) return GDN_ERR_WORKSPACE;
    if (workspace && ((uintptr_t)workspace & 15) != 0) return GDN_ERR_INVALID_ARG;
  }
  Batch Bs = make_batch(batch);
  if (any_long) Bs.max_len = threshold - 1;
  if (rule(G, Bs, P, dims, qkv, a, b, o, pages, status, s) != cudaSuccess) return GDN_ERR_LAUNCH;
  if (!any_long) return GDN_OK;
  Batch Bc = make_batch(batch);
  Bc.min_len = threshold;
  if (workspace && need > 0) {
    const int ws_chunks = (batch->max_rows + 63) / 64;
    if (launch_chunk2(&tmap, G, Bc, P, dims->state_dtype == GDN_BF16, dims->out_dtype == GDN_F32,
                      a, b, o, pages, workspace, ws_chunks, status, s) != cudaSuccess)
      return GDN_ERR_LAUNCH;
    return GDN_OK;
  }
  if (launch_chunk(&tmap, G, Bc, P, dims->state_dtype == GDN_BF16, dims->out_dtype == GDN_F32, a,
                   b, o, pages, status, s) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

size_t gdn_chunk_prefill_workspace_bytes(const gdn_dims* dims, const gdn_batch* batch) {
  if (check_dims(dims) != GDN_OK || check_batch(batch, true) != GDN_OK) return 0;
  if (dims->io_dtype != GDN_BF16 || dims->head_k_dim != 128 || dims->head_v_dim != 128) return 0;
  const size_t chunks = ((size_t)batch->max_rows + 63) / 64;
  return (size_t)batch->num_requests * (size_t)dims->num_v_heads * chunks * gdn::kChunkItemBytes;
}

gdn_status gdn_chunk_prefill(const gdn_dims* dims, const gdn_batch* batch, const gdn_params* params,
                             const void* qkv, const void* a, const void* b, void* o, void* pages,
                             void* workspace, size_t workspace_bytes, int32_t* status,
                             gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if ((e = check_batch(batch, true)) != GDN_OK) return e;
  if ((e = check_params(params, true)) != GDN_OK) return e;
  if (dims->io_dtype != GDN_BF16 || dims->head_k_dim != 128 || dims->head_v_dim != 128)
    return GDN_ERR_UNSUPPORTED;
  if (batch->num_requests == 0) return GDN_OK;
  if (!status || !pages) return GDN_ERR_INVALID_ARG;
  CUtensorMap tmap;
  std::memset(&tmap, 0, sizeof(tmap));
  if (batch->num_rows > 0) {
    // with no rows every request has length 0 and the map is never read
    if (!qkv || !a || !b || !o) return GDN_ERR_INVALID_ARG;
    if (((uintptr_t)qkv & 15) != 0) return GDN_ERR_UNSUPPORTED;
    const gdn_status te = encode_rows_tmap(&tmap, qkv, batch->num_rows, dims);
    if (te != GDN_OK) return te;
  }
  const Geom G = make_geom(dims);
  const Batch B = make_batch(batch);
  const Params P = make_params(params, dims);
  const size_t need = gdn_chunk_prefill_workspace_bytes(dims, batch);
  if (workspace && need > 0) {
    if (workspace_bytes < need) return GDN_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 15) != 0) return GDN_ERR_INVALID_ARG;
    const int ws_chunks = (batch->max_rows + 63) / 64;
    if (launch_chunk2(&tmap, G, B, P, dims->state_dtype == GDN_BF16, dims->out_dtype == GDN_F32,
                      a, b, o, pages, workspace, ws_chunks, status,
                      (cudaStream_t)stream) != cudaSuccess)
      return GDN_ERR_LAUNCH;
    return GDN_OK;
  }
  if (launch_chunk(&tmap, G, B, P, dims->state_dtype == GDN_BF16, dims->out_dtype == GDN_F32, a, b,
                   o, pages, status, (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

gdn_status gdn_chunk_prefill_noalloc(const gdn_dims* dims, const gdn_batch* batch,
                                     const gdn_params* params, const void* qkv, const void* a,
                                     const void* b, void* o, void* pages, int32_t* status,
                                     gdn_stream_t stream) {
  gdn_status e = check_dims(dims);
  if (e != GDN_OK) return e;
  if ((e = check_batch(batch, true)) != GDN_OK) return e;
  if ((e = check_params(params, true)) != GDN_OK) return e;
  if (dims->io_dtype != GDN_BF16 || dims->head_k_dim != 128 || dims->head_v_dim != 128)
    return GDN_ERR_UNSUPPORTED;
  if (batch->num_requests == 0) return GDN_OK;
  if (!status || !pages) return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_chunk_prefill_workspace_bytes(dims, batch);
  if (need > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;
  CUtensorMap tmap;
  std::memset(&tmap, 0, sizeof(tmap));
  if (batch->num_rows > 0) {
    if (!qkv || !a || !b || !o) return GDN_ERR_INVALID_ARG;
    if (((uintptr_t)qkv & 15) != 0) return GDN_ERR_UNSUPPORTED;
    const gdn_status te = encode_rows_tmap(&tmap, qkv, batch->num_rows, dims);
    if (te != GDN_OK) return te;
  }
  void* scratch = nullptr;
  if (chunk_scratch_address(&scratch) != cudaSuccess) return GDN_ERR_LAUNCH;
  // every item the chain reads is written by the pre-pass of the same call,
  // so nothing in the scratch has to start at zero
  const Geom G = make_geom(dims);
  const Batch B = make_batch(batch);
  const Params P = make_params(params, dims);
  const int ws_chunks = (batch->max_rows + 63) / 64;
  if (launch_chunk2(&tmap, G, B, P, dims->state_dtype == GDN_BF16, dims->out_dtype == GDN_F32, a,
                    b, o, pages, scratch, ws_chunks, status, (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  return GDN_OK;
}

gdn_status gdn_check_bounded_wait(int64_t limit_ns, int32_t* status, gdn_stream_t stream) {
  if (!status || limit_ns <= 0 || limit_ns > 10000000000LL) return GDN_ERR_INVALID_ARG;
  gdn::wait_check_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_ns, status);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

const char* gdn_strerror(int32_t s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument (null pointer, negative count or bad enum)";
    case GDN_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case GDN_ERR_LAUNCH: return "kernel launch failed";
    case GDN_ERR_WORKSPACE: return "workspace too small";
    case GDN_ERR_NO_DEVICE: return "no usable device";
    case GDN_DEV_BAD_PAGE: return "device: page index out of range";
    case GDN_DEV_BAD_ROWS: return "device: row range out of bounds";
    case GDN_DEV_BAD_ACCEPTED: return "device: accepted count outside the record width";
    case GDN_DEV_STALE_STEP: return "device: page step parity does not match the request";
    case GDN_DEV_TOO_MANY_CANDIDATES: return "device: more candidate rows than max_candidates";
    case GDN_DEV_RECORD_OPEN: return "device: plain rows on a page whose spec record is open";
    case GDN_DEV_BAD_FLAG: return "device: corrupt page flag word (or FRESH with SPEC)";
    case GDN_DEV_TIMEOUT: return "device: a bounded on-chip wait gave up";
    default: return "unknown status";
  }
}

}  // extern "C"
