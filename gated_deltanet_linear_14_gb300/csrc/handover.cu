// Hand-over between the one-page layout and the slot-per-candidate layout
// (sm_103a).
//
// r9700-stack v0.2.4, "What it does": with prefix caching on, the stock
// design's per-candidate pages are kept; a request can therefore move from
// its one state page to a slot pool (and back) between steps. What moves is
// what the next step starts from: the state and the W-1 history columns of
// the conv window. A page hands over only with its record closed (after a
// commit), so nothing of an unverified step is carried; a page received
// from a slot starts with an empty record.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

constexpr int kHandThreads = 256;

// One CTA-row per request; the blocks of a row copy 16-byte pieces of the
// state, then of the window history. dir 0: page -> slot 0 of the pool;
// dir 1: slot slot[i] of the pool -> page (and the page's record closed).
__global__ void __launch_bounds__(kHandThreads)
handover_kernel(Geom G, SlotGeom SG, int dir, int n, const int32_t* __restrict__ page,
                const int32_t* __restrict__ pool, const int32_t* __restrict__ slot,
                int num_pages, int num_pools, char* pages, char* slots, size_t state_bytes,
                size_t window_bytes, int32_t* status) {
  pdl_begin();
  const int i = blockIdx.y;
  if (i >= n) return;
  const bool reporter = (blockIdx.x == 0 && threadIdx.x == 0);
  const int p = page[i], q = pool[i];
  const int s = (dir == 1) ? slot[i] : 0;
  int err = 0;
  if (p < 0 || p >= num_pages || q < 0 || q >= num_pools) err = GDN_DEV_BAD_PAGE;
  else if (dir == 1 && (s < 0 || s >= G.Kc)) err = GDN_DEV_BAD_ACCEPTED;
  char* pg = pages + (size_t)(err ? 0 : p) * G.page_bytes;
  char* sl = slots + (size_t)(err ? 0 : q) * SG.pool_bytes + (size_t)(err ? 0 : s) * SG.slot_bytes;
  uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
  if (!err && dir == 0 && flag_width(*flagp) != 0) err = GDN_DEV_RECORD_OPEN;
  if (err) {
    if (reporter) report(status, err);
    return;
  }
  const size_t ns = state_bytes / 16, nw = window_bytes / 16;
  for (size_t k = (size_t)blockIdx.x * kHandThreads + threadIdx.x; k < ns + nw;
       k += (size_t)gridDim.x * kHandThreads) {
    const size_t po = (k < ns) ? G.state_off + 16 * k : G.window_off + 16 * (k - ns);
    const size_t so = (k < ns) ? SG.state_off + 16 * k : SG.window_off + 16 * (k - ns);
    uint4* dst = reinterpret_cast<uint4*>(dir == 0 ? sl + so : pg + po);
    const uint4* src = reinterpret_cast<const uint4*>(dir == 0 ? pg + po : sl + so);
    *dst = *src;
  }
  if (dir == 1 && reporter) *flagp = 0u;   // an empty record, step parity 0
}

cudaError_t launch_handover(const Geom& G, const SlotGeom& SG, int dir, int n, const int32_t* page,
                            const int32_t* pool, const int32_t* slot, int num_pages,
                            int num_pools, void* pages, void* slots, size_t state_bytes,
                            size_t window_bytes, int32_t* status, cudaStream_t stream) {
  const size_t pieces = (state_bytes + window_bytes) / 16;
  int bx = (int)((pieces + kHandThreads * 8 - 1) / (kHandThreads * 8));
  if (bx < 1) bx = 1;
  if (bx > 64) bx = 64;
  return launch_pdl(handover_kernel, dim3(bx, n), dim3(kHandThreads), 0, stream, G, SG, dir, n,
                    page, pool, slot, num_pages, num_pools, static_cast<char*>(pages),
                    static_cast<char*>(slots), state_bytes, window_bytes, status);
}

}  // namespace gdn
