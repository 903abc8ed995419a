// Fused decode step: causal conv + SiLU, q/k L2 norm and gates, and the gated
// delta rule for requests with one token each, in one launch (sm_103a).
//
// It computes exactly what gdn_conv (io-dtype output) followed by gdn_seq
// computes for such a batch, bit for bit: the conv uses the same fp32
// fused-multiply-add order and the library's own SiLU, its outputs are
// rounded to the io dtype before the rule reads them, and the rule uses the
// same staging (fetch/publish) and token step as the token-by-token kernel.
// The r9700-stack v0.2.3 notes (section 1) describe the cost this removes: a
// prefill or decode step that runs several small launches per layer is bound
// by launches rather than by the work.
//
// Design. One CTA per (request, q/k head kh): the group of Hv/Hk value heads
// that read q/k head kh, times the Dv/32 column blocks of each, is the CTA's
// list of items. The conv'd q, k and the group's v channels are computed once
// into shared memory, and this CTA is the only writer of those channels'
// conv windows (nothing else reads them in this launch). The items' state
// tiles (32 columns x Dk, contiguous in the page) stream through a 3-stage
// shared-memory ring filled by bulk asynchronous copies (cp.async.bulk with
// an mbarrier per stage), so several tiles per CTA are in flight while the
// current one is updated; new state goes back to HBM straight from registers.
#include "common.cuh"
#include "kernels.h"
#include "rule.cuh"
#include "umma.cuh"

namespace gdn {

using namespace umma;

// 3 stages (about 53 KB of shared memory) leave room for 4 CTAs per SM; with
// 4 stages (70 KB, 3 CTAs per SM) the 64-request batch ran 8 % slower and
// with 2 stages (6 CTAs per SM) no faster.
constexpr int kDecStages = 3;
// Item i's stage is refilled (with item i + kDecStages) at the barrier of
// item i + 1, after its own wait: one stage would wait on a copy never issued.
static_assert(kDecStages >= 2, "the ring needs at least two stages");
constexpr int kDecMaxRow = 2 * 128 + 512;  // q | k | the group's v (items <= kTC)

// What the items of one CTA share: one token's q^ and k^, and per item the
// value block and (alpha, beta, q^.k^).
template <int DK>
struct DecStage {
  float q[DK];
  float k[DK];
  float v[kTC][kBV];
  float4 sc[kTC];
  float kq;
};

template <class IO, class ST, int DK>
struct DecLayout {
  static constexpr uint32_t TILE = kBV * DK;                       // state elements per item
  static constexpr uint32_t TILE_BYTES = TILE * sizeof(ST);
  static constexpr uint32_t OFF_STAGE = kDecStages * TILE_BYTES;   // DecStage<DK>
  static constexpr uint32_t OFF_ROW = OFF_STAGE + ((sizeof(DecStage<DK>) + 127) / 128) * 128;
  static constexpr uint32_t BYTES = OFF_ROW + kDecMaxRow * sizeof(IO);
};

template <class IO, class ST, int DK>
__global__ void __launch_bounds__(kRuleThreads)
decode_kernel(Geom G, Batch B, Params P, const IO* __restrict__ x, const IO* __restrict__ w,
              const IO* __restrict__ a_in, const IO* __restrict__ b_in, void* o, int out_f32,
              void* pages, int32_t* status) {
  using Lay = DecLayout<IO, ST, DK>;
  constexpr int PE = DK / 8;
  extern __shared__ __align__(128) uint8_t dsm[];
  ST* tiles = reinterpret_cast<ST*>(dsm);
  DecStage<DK>& st = *reinterpret_cast<DecStage<DK>*>(dsm + Lay::OFF_STAGE);
  IO* mrow = reinterpret_cast<IO*>(dsm + Lay::OFF_ROW);
  __shared__ __align__(8) uint64_t full[kDecStages];

  pdl_begin();
  const int kh = blockIdx.x;
  const int tid = threadIdx.x;
  const bool reporter = (kh == 0 && tid == 0);
  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  if (q.spec) return;
  if (q.len > 1) {
    if (reporter) report(status, GDN_DEV_BAD_ROWS);
    return;
  }
  char* pg = page_ptr(G, pages, q.page);
  uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
  if (!q.fresh && flag_width(*flagp) != 0) {
    if (reporter) report(status, GDN_DEV_RECORD_OPEN);
    return;
  }
  if (!q.fresh && q.len == 0) return;

  const int Gh = G.Hv / G.Hk, nCB = G.Dv / kBV, n_items = Gh * nCB;
  const int h0 = kh * Gh;
  ST* Sbase = reinterpret_cast<ST*>(pg + G.state_off);
  IO* win = reinterpret_cast<IO*>(pg + G.window_off);
  const bool stream_state = !q.fresh;   // a fresh request starts from zero

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    mbar_fence_init();
  }
  __syncthreads();
  auto issue = [&](int i) {
    const int s = i % kDecStages;
    const int h = h0 + i / nCB, cb = i % nCB;
    const ST* src = Sbase + ((size_t)h * G.Dv + (size_t)cb * kBV) * DK;
    mbar_expect_tx(smem_u32(&full[s]), Lay::TILE_BYTES);
    bulk_load(smem_u32(tiles + (size_t)s * Lay::TILE), src, Lay::TILE_BYTES, smem_u32(&full[s]));
  };
  int issued = 0;  // items whose copy has been started (thread 0's count)
  if (tid == 0 && stream_state)
    for (; issued < n_items && issued < kDecStages; ++issued) issue(issued);

  // conv of the group's channels (q, k of head kh; v of heads h0..h0+Gh-1),
  // four channels per thread, and the new conv window of those channels
  const int nch = 2 * DK + Gh * G.Dv;
  for (int c4 = 4 * tid; c4 < nch; c4 += 4 * kRuleThreads) {
    const int c = (c4 < DK) ? kh * DK + c4
                : (c4 < 2 * DK) ? G.Hk * DK + kh * DK + (c4 - DK)
                                : 2 * G.Hk * DK + h0 * G.Dv + (c4 - 2 * DK);
    float wt[4][4];
    {
      float tmp[16];
      load_f<IO, 16>(w + (size_t)c * 4, tmp);
#pragma unroll
      for (int v = 0; v < 4; ++v)
#pragma unroll
        for (int j = 0; j < 4; ++j) wt[j][v] = tmp[v * 4 + j];
    }
    float hcol[3][4];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      if (q.fresh) {
#pragma unroll
        for (int v = 0; v < 4; ++v) hcol[j][v] = 0.0f;
      } else {
        load_f<IO, 4>(win + (size_t)j * G.C + c, hcol[j]);
      }
    }
    float xv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (q.len == 1) load_f<IO, 4>(x + (size_t)q.start * G.C + c, xv);
    float yv[4];
#pragma unroll
    for (int v = 0; v < 4; v += 2) {   // channel pairs, as the conv kernel
      float2 acc = P.conv_bias ? make_float2(P.conv_bias[c + v], P.conv_bias[c + v + 1])
                               : make_float2(0.0f, 0.0f);
#pragma unroll
      for (int j = 0; j < 3; ++j)
        acc = __ffma2_rn(make_float2(wt[j][v], wt[j][v + 1]),
                         make_float2(hcol[j][v], hcol[j][v + 1]), acc);
      acc = __ffma2_rn(make_float2(wt[3][v], wt[3][v + 1]), make_float2(xv[v], xv[v + 1]), acc);
      const float2 y2 = own_silu2(acc);
      yv[v] = y2.x;
      yv[v + 1] = y2.y;
    }
    store_f<IO, 4>(mrow + c4, yv);
    // new window: the last three columns of [history; this row]
    if (q.len == 1) {
      store_f<IO, 4>(win + c, hcol[1]);
      store_f<IO, 4>(win + (size_t)G.C + c, hcol[2]);
      store_f<IO, 4>(win + 2 * (size_t)G.C + c, xv);
    } else {
#pragma unroll
      for (int j = 0; j < 3; ++j) store_f<IO, 4>(win + (size_t)j * G.C + c, hcol[j]);
    }
  }
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31, cg = lane >> 3, r8 = lane & 7;
  const int vcol = warp * 8 + cg * 2;
  int col[kColsPerLane];
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m) col[m] = vcol + m;   // column inside the 32-wide block

  if (q.len == 0) {
    // a fresh request with no token: a zero state
    LaneState<DK / 8> Z;
    zero_state<DK / 8>(Z);
    for (int i = 0; i < n_items; ++i) {
      const int h = h0 + i / nCB, cb = i % nCB;
      store_state<DK, ST>(Sbase + ((size_t)h * G.Dv + (size_t)cb * kBV) * DK, Z, col, r8);
    }
    if (kh == 0 && tid == 0) *flagp = 0u;
    return;
  }

  // Stage q^, k^ (through the token-by-token kernel's own normalisation, so
  // the token step sees bit-identical inputs), each item's value block and
  // gates.
  {
    const int t = tid >> 3, p = tid & 7;
    if (t == 0) {
      RawVec<IO, PE> rq, rk;
      rq.load(mrow + PE * p);
      rk.load(mrow + DK + PE * p);
      const float kq = publish_qk<DK, IO, ST>(st.q, st.k, PE * p, rq, rk, P);
      if (p == 0) st.kq = kq;
    }
    float alpha = 0.0f, beta = 0.0f;
    if (t < n_items) {
      const int g = t / nCB, cb = t % nCB;
      RawVec<IO, 4> rv;
      rv.load(mrow + 2 * DK + g * G.Dv + cb * kBV + 4 * p);
#pragma unroll
      for (int e = 0; e < 4; ++e) st.v[t][4 * p + e] = rv.get(e);
      if (p == 0)
        gates(P, h0 + g, to_f(a_in[(size_t)q.start * G.Hv + h0 + g]),
              to_f(b_in[(size_t)q.start * G.Hv + h0 + g]), alpha, beta);
    }
    __syncthreads();
    if (t < n_items && p == 0) st.sc[t] = make_float4(alpha, beta, st.kq, 0.0f);
  }
  __syncthreads();

  bool failed = false;
  int consumed = 0;
  for (int i = 0; i < n_items; ++i, consumed = i) {
    const int s = i % kDecStages;
    const int h = h0 + i / nCB, cb = i % nCB;
    LaneState<DK / 8> S;
    if (stream_state) {
      const bool ok = mbar_wait(smem_u32(&full[s]), (uint32_t)((i / kDecStages) & 1));
      // one barrier per item: past it every thread has also finished reading
      // the previous item's stage, which can then be refilled
      if (__syncthreads_or(!ok)) {
        failed = true;
        break;
      }
      if (tid == 0 && i > 0 && issued < n_items) issue(issued++);
      load_state<DK, ST>(S, tiles + (size_t)s * Lay::TILE, col, r8);
    } else {
      zero_state<DK / 8>(S);
    }
    const float ov = token_step_rows<DK, ST>(S, st.q, st.k, st.v[i], st.sc[i], r8, vcol, P.scale,
                                             true);
    if ((r8 & 3) == 0) {
      const size_t off = ((size_t)q.start * G.Hv + h) * G.Dv + (size_t)cb * kBV + vcol + (r8 >> 2);
      store_out(o, out_f32, off, ov);
    }
    int gcol[kColsPerLane];
#pragma unroll
    for (int m = 0; m < kColsPerLane; ++m) gcol[m] = cb * kBV + col[m];
    store_state<DK, ST>(Sbase + (size_t)h * G.Dv * DK, S, gcol, r8);
  }
  if (failed) {
    if (tid == 0) report(status, GDN_DEV_TIMEOUT);
    // let copies still in flight land before the CTA's shared memory goes away
    if (tid == 0)
      for (int j = consumed; j < issued; ++j)
        mbar_wait(smem_u32(&full[j % kDecStages]), (uint32_t)((j / kDecStages) & 1));
    return;
  }
  if (q.fresh && kh == 0 && tid == 0) *flagp = 0u;  // empty record
}

template <class IO, class ST, int DK>
static cudaError_t launch_decode_t(const Geom& G, const Batch& B, const Params& P, int out_f32,
                                   const void* x, const void* w, const void* a, const void* b,
                                   void* o, void* pages, int32_t* status, cudaStream_t stream) {
  using Lay = DecLayout<IO, ST, DK>;
  cudaError_t e = ensure_smem_limit<decode_kernel<IO, ST, DK>>((int)Lay::BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_kernel<IO, ST, DK>, dim3(G.Hk, B.R), dim3(kRuleThreads), Lay::BYTES,
                    stream, G, B, P, static_cast<const IO*>(x), static_cast<const IO*>(w),
                    static_cast<const IO*>(a), static_cast<const IO*>(b), o, out_f32, pages,
                    status);
}

template <class IO, class ST>
static cudaError_t launch_decode_io_st(const Geom& G, const Batch& B, const Params& P, int out_f32,
                                       const void* x, const void* w, const void* a, const void* b,
                                       void* o, void* pages, int32_t* status, cudaStream_t s) {
  switch (G.Dk) {
    case 32: return launch_decode_t<IO, ST, 32>(G, B, P, out_f32, x, w, a, b, o, pages, status, s);
    case 64: return launch_decode_t<IO, ST, 64>(G, B, P, out_f32, x, w, a, b, o, pages, status, s);
    default: return launch_decode_t<IO, ST, 128>(G, B, P, out_f32, x, w, a, b, o, pages, status, s);
  }
}

cudaError_t launch_decode(const Geom& G, const Batch& B, const Params& P, int io_bf16,
                          int state_bf16, int out_f32, const void* x, const void* w, const void* a,
                          const void* b, void* o, void* pages, int32_t* status,
                          cudaStream_t stream) {
  if (io_bf16) {
    if (state_bf16)
      return launch_decode_io_st<bf16, bf16>(G, B, P, out_f32, x, w, a, b, o, pages, status, stream);
    return launch_decode_io_st<bf16, float>(G, B, P, out_f32, x, w, a, b, o, pages, status, stream);
  }
  if (state_bf16)
    return launch_decode_io_st<float, bf16>(G, B, P, out_f32, x, w, a, b, o, pages, status, stream);
  return launch_decode_io_st<float, float>(G, B, P, out_f32, x, w, a, b, o, pages, status, stream);
}

}  // namespace gdn
