// Causal depthwise conv + SiLU over the step's packed rows (sm_103a).
//
// r9700-stack v0.2.3, section 1 (r9k_gdn_conv: one launch over the batch's
// own rows); v0.2.4, "A defect found and fixed before the tag" (the window
// rolls by the candidate count read from the record); vllm.cpp PR #155,
// "What changed" (the width-4 specialisation, one channel group per thread).
//
// Design (HBM-bound streaming):
//   * a thread owns one 8-byte vector of channels (4 bf16 or 2 fp32) and a
//     tile of TR consecutive rows of one request; the W-1 previous columns
//     live in registers and slide down the tile, so every input element is
//     read once (plus W-1 halo rows per tile);
//   * grid = (channel tiles, row tiles, requests); empty row tiles exit;
//   * the conv window of a page is read ONLY by row tile 0 of the request,
//     and that same thread also writes the new window (from its registers
//     and the read-only input rows). No other block touches the window, so a
//     long request split over many blocks cannot race on it (the hazard
//     vllm.cpp's exact-chunk conv has, where one block reads the initial
//     window and another writes the final one).
//   * accumulation is fp32 in a fixed order: bias (or 0), then taps
//     j = 0..W-1 oldest first, each a fused multiply-add; SiLU uses the
//     library's own exp and the correctly rounded quotient t / (1 + t)
//     (common.cuh). The CPU fp32 conv reproduces this bit for bit.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

// The exact SiLU (own exp and quotient per element) keeps the conv's
// floating-point pipe busier than its HBM traffic, so the kernel is built to
// keep that pipe fed: channel pairs in packed f32x2 form, 8-byte vectors, 4
// CTAs of 256 threads per SM (32 warps), and the input rows staged into
// shared memory by each thread's own cp.async two batches ahead, so the
// arithmetic of a batch never waits for its loads.
constexpr int kConvThreads = 256;
constexpr int kConvVecBytes = 8;
// Rows per tile (TILE): 64 where the launch has rows for several waves of
// CTAs (fewer tiles: less per-tile setup, fewer halo rows, and rows in ring
// stages of 8), else 32 (more CTAs for batches of short requests, stages of
// 4: the 24 KB ring of the short tile leaves the shared memory the kernels
// after it in a mixed step want).
constexpr int kConvRowsLong = 64;
constexpr int kConvRowsShort = 32;
constexpr int kConvStages = 3;  // ring stages: the batch in use and two in flight

__device__ __forceinline__ void conv_cp8(void* smem, const void* gmem) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void conv_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most kConvStages - 1 groups of this thread are pending
__device__ __forceinline__ void conv_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kConvStages - 1) : "memory");
}

template <class IO, class YT, int W, bool SLOTS, int TILE>
__global__ void __launch_bounds__(kConvThreads, 4)
conv_kernel(Geom G, Batch B, Params P, SlotGeom SG, const IO* __restrict__ x,
            const IO* __restrict__ w, YT* __restrict__ y, void* pages, int32_t* status) {
  pdl_begin();
  constexpr int V = kConvVecBytes / (int)sizeof(IO);  // channels per thread
  constexpr int H = W - 1;
  constexpr int kConvBatch = TILE / 8;   // rows per ring stage
  const bool reporter = (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0);

  Batch Bi = B;
  Bi.order = nullptr;  // the conv has no scheduling order
  const Req q = load_req(Bi, blockIdx.z);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  const int t0 = blockIdx.y * TILE;
  if (t0 > 0 && t0 >= q.len) return;

  char* pg = nullptr;
  const IO* hist_src = nullptr;  // history column 0 (oldest), or null for zeros
  IO* win = nullptr;
  IO* rec_out = nullptr;         // record slot receiving conv'd candidate rows
  char* pool = nullptr;
  if constexpr (!SLOTS) {
    pg = page_ptr(G, pages, q.page);
    win = reinterpret_cast<IO*>(pg + G.window_off);
    const uint32_t flag = *reinterpret_cast<const uint32_t*>(pg + G.flag_off);
    if (q.spec) {
      SpecState ss = spec_state(G, B, q, flag);
      if (q.fresh) ss.err = GDN_DEV_BAD_FLAG;
      if (ss.err) {
        if (reporter) report(status, ss.err);
        return;
      }
      const int base = (ss.width > 0) ? ss.accepted + 1 : 0;
      hist_src = win + (size_t)base * G.C;
      rec_out = reinterpret_cast<IO*>(pg + G.record_off) + (size_t)(1 - ss.live) * G.Kc * G.rec_row;
    } else if (!q.fresh) {
      if (flag_width(flag) != 0) {
        if (reporter) report(status, GDN_DEV_RECORD_OPEN);
        return;
      }
      hist_src = win;
    }
  } else {
    const int src = B.n_accepted ? B.n_accepted[q.r] : -1;
    if (src < 0 || src >= G.Kc) {
      if (reporter) report(status, GDN_DEV_BAD_ACCEPTED);
      return;
    }
    if (q.len > G.Kc) {
      if (reporter) report(status, GDN_DEV_TOO_MANY_CANDIDATES);
      return;
    }
    pool = reinterpret_cast<char*>(pages) + (size_t)q.page * SG.pool_bytes;
    hist_src = reinterpret_cast<const IO*>(pool + (size_t)src * SG.slot_bytes + SG.window_off);
  }

  const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * V;
  if (c0 >= G.C) return;

  // Each thread copies its own 8-byte vector of every row into its own
  // column of the ring and reads back only that, so its cp.async waits are
  // the only ordering needed (no block-wide barrier). Every copy is issued
  // here, after the last early return, and waited for before the end.
  __shared__ uint2 ring[kConvStages][kConvBatch][kConvThreads];
  const int t_end = min(q.len, t0 + TILE);
  const int nb = (t_end - t0 + kConvBatch - 1) / kConvBatch;
  const IO* xr = x + (size_t)q.start * G.C + c0;  // row t at xr + t C
  auto issue = [&](int b) {
    if (b < nb) {
#pragma unroll
      for (int i = 0; i < kConvBatch; ++i) {
        const int t = t0 + b * kConvBatch + i;
        if (t < t_end) conv_cp8(&ring[b % kConvStages][i][threadIdx.x], xr + (size_t)t * G.C);
      }
    }
    conv_commit();
  };
#pragma unroll
  for (int b = 0; b < kConvStages - 1; ++b) issue(b);

  // taps and bias
  float wt[W][V];
  {
    float tmp[W * V];
#pragma unroll
    for (int i = 0; i < W * V; i += 16 / (int)sizeof(IO)) load_f<IO, 16 / sizeof(IO)>(w + (size_t)c0 * W + i, tmp + i);
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
      for (int j = 0; j < W; ++j) wt[j][v] = tmp[v * W + j];
  }
  float bias[V];
#pragma unroll
  for (int v = 0; v < V; ++v) bias[v] = P.conv_bias ? P.conv_bias[c0 + v] : 0.0f;

  // history for the tile's first row: sequence positions t0-H .. t0-1
  float h[H][V];
#pragma unroll
  for (int j = 0; j < H; ++j) {
    const int pos = t0 - H + j;
    if (pos >= 0) {
      load_f<IO, V>(xr + (size_t)pos * G.C, h[j]);
    } else if (hist_src) {
      load_f<IO, V>(hist_src + (size_t)(H + pos) * G.C + c0, h[j]);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) h[j][v] = 0.0f;
    }
  }

  // The new window. The window channels [c0, c0+V) are read and written
  // only by this thread of row tile 0, which has already taken its history
  // into registers; the history is read again here where the new window
  // keeps some of it. Writing it before the rows keeps its pointers out of
  // the main loop.
  if (!SLOTS && blockIdx.y == 0) {
    if (q.spec) {
      // columns 0..H-1 keep the history this step started from; the raw
      // candidates follow, so the next step can roll by its accepted count
      float hw[H][V];
#pragma unroll
      for (int j = 0; j < H; ++j) load_f<IO, V>(hist_src + (size_t)j * G.C + c0, hw[j]);
#pragma unroll
      for (int j = 0; j < H; ++j) store_f<IO, V>(win + (size_t)j * G.C + c0, hw[j]);
      for (int t = 0; t < q.len; ++t) {
        float xv[V];
        load_f<IO, V>(x + (size_t)(q.start + t) * G.C + c0, xv);
        store_f<IO, V>(win + (size_t)(H + t) * G.C + c0, xv);
      }
    } else {
      // last H columns of [history; rows], oldest first. Column j comes from
      // sequence position len-H+j, which is a history column when negative;
      // for j < H those history columns sit at index >= j, so reading them
      // in increasing j before overwriting column j is safe.
#pragma unroll
      for (int j = 0; j < H; ++j) {
        const int pos = q.len - H + j;
        float col[V];
        if (pos >= 0) {
          load_f<IO, V>(x + (size_t)(q.start + pos) * G.C + c0, col);
        } else if (hist_src) {
          load_f<IO, V>(hist_src + (size_t)(H + pos) * G.C + c0, col);
        } else {
#pragma unroll
          for (int v = 0; v < V; ++v) col[v] = 0.0f;
        }
        store_f<IO, V>(win + (size_t)j * G.C + c0, col);
      }
    }
  }

  // one row: taps, SiLU, stores, then the window slides by one. rec is a
  // constant at each call, so the full-batch path below has no branch
  // between its rows and their arithmetic interleaves. The output row moves
  // by one row stride per row (an address add, not a 64-bit product).
  YT* yrow = y + ((size_t)q.start + t0) * G.C + c0;
  const size_t ystride = (size_t)G.C;
  auto row = [&](const uint2 raw, int t, bool rec) {
    float xv[V];
    {
      const IO* e = reinterpret_cast<const IO*>(&raw);
#pragma unroll
      for (int v = 0; v < V; ++v) xv[v] = to_f(e[v]);
    }
    // channel pairs in packed f32x2 form: each channel sees the same fused
    // multiply-adds, in the same order, as a scalar loop would
    float yv[V];
#pragma unroll
    for (int v = 0; v < V; v += 2) {
      float2 acc = make_float2(bias[v], bias[v + 1]);
#pragma unroll
      for (int j = 0; j < H; ++j)
        acc = __ffma2_rn(make_float2(wt[j][v], wt[j][v + 1]), make_float2(h[j][v], h[j][v + 1]), acc);
      acc = __ffma2_rn(make_float2(wt[H][v], wt[H][v + 1]), make_float2(xv[v], xv[v + 1]), acc);
      const float2 y2 = own_silu2(acc);
      yv[v] = y2.x;
      yv[v + 1] = y2.y;
    }
    store_f<YT, V>(yrow, yv);
    yrow += ystride;
#pragma unroll
    for (int j = 0; j < H - 1; ++j)
#pragma unroll
      for (int v = 0; v < V; ++v) h[j][v] = h[j + 1][v];
#pragma unroll
    for (int v = 0; v < V; ++v) h[H - 1][v] = xv[v];
    if constexpr (!SLOTS) {
      if (rec) store_f<IO, V>(rec_out + (size_t)t * G.rec_row + c0, yv);
    } else {
      // window after candidate t goes to slot t
      IO* wdst = reinterpret_cast<IO*>(pool + (size_t)t * SG.slot_bytes + SG.window_off);
#pragma unroll
      for (int j = 0; j < H; ++j) store_f<IO, V>(wdst + (size_t)j * G.C + c0, h[j]);
    }
  };

  for (int b = 0; b < nb; ++b) {
    issue(b + kConvStages - 1);
    conv_wait();  // batch b has landed
    const int tb = t0 + b * kConvBatch;
    const int s = b % kConvStages;
    if (tb + kConvBatch <= t_end && rec_out == nullptr) {
      // a full batch of plain rows
#pragma unroll
      for (int i = 0; i < kConvBatch; ++i) row(ring[s][i][threadIdx.x], tb + i, false);
    } else {
      // the ragged end of a tile, or candidate rows that also go to the record
#pragma unroll
      for (int i = 0; i < kConvBatch; ++i)
        if (tb + i < t_end) row(ring[s][i][threadIdx.x], tb + i, rec_out != nullptr);
    }
  }

}

template <class IO, class YT, bool SLOTS>
static cudaError_t launch_conv_t(const Geom& G, const Batch& B, const Params& P, const SlotGeom& SG,
                                 const void* x, const void* w, void* y, void* pages,
                                 int32_t* status, cudaStream_t stream) {
  constexpr int V = kConvVecBytes / (int)sizeof(IO);
  const int ctiles = (G.C + kConvThreads * V - 1) / (kConvThreads * V);
  // several waves (4 CTAs per SM) of long tiles, counting the rows present
  const long long long_ctas = (long long)ctiles * (B.num_rows / kConvRowsLong);
  const int tile = (long_ctas >= 4LL * 4 * device_sms()) ? kConvRowsLong : kConvRowsShort;
  const int rtiles = B.max_rows > 0 ? (B.max_rows + tile - 1) / tile : 1;
  auto kern = (tile == kConvRowsLong) ? conv_kernel<IO, YT, 4, SLOTS, kConvRowsLong>
                                      : conv_kernel<IO, YT, 4, SLOTS, kConvRowsShort>;
  return launch_pdl(kern, dim3(ctiles, rtiles, B.R), dim3(kConvThreads), 0, stream, G, B, P, SG,
                    static_cast<const IO*>(x), static_cast<const IO*>(w), static_cast<YT*>(y),
                    pages, status);
}

cudaError_t launch_conv(const Geom& G, const Batch& B, const Params& P, int io_bf16, int y_f32,
                        const void* x, const void* w, void* y, void* pages, int32_t* status,
                        cudaStream_t stream) {
  SlotGeom SG{};
  if (io_bf16) {
    if (y_f32) return launch_conv_t<bf16, float, false>(G, B, P, SG, x, w, y, pages, status, stream);
    return launch_conv_t<bf16, bf16, false>(G, B, P, SG, x, w, y, pages, status, stream);
  }
  return launch_conv_t<float, float, false>(G, B, P, SG, x, w, y, pages, status, stream);
}

cudaError_t launch_conv_slots(const Geom& G, const Batch& B, const Params& P, const SlotGeom& SG,
                              int io_bf16, const void* x, const void* w, void* y, void* slots,
                              int32_t* status, cudaStream_t stream) {
  if (io_bf16) return launch_conv_t<bf16, bf16, true>(G, B, P, SG, x, w, y, slots, status, stream);
  return launch_conv_t<float, float, true>(G, B, P, SG, x, w, y, slots, status, stream);
}

}  // namespace gdn
