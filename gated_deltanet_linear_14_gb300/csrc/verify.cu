// One-page speculative verify, pipelined over state tiles (sm_103a).
//
// r9700-stack v0.2.4, "What it does": one state page per request; a step
// replays the previous step's accepted rows from the page's record into the
// state, stores that as the checkpoint, then runs this step's candidates
// from it. The arithmetic is the token-by-token kernel's (rule.cuh): the
// same q/k normalisation, the same token step, and a replay step that leaves
// a bit-identical state without the output half, so results are
// bit-identical to the slot-per-candidate layout.
//
// Design. The work is cut into units (request, q/k head kh, part); a part is
// a run of `ipu` consecutive items, an item being one value head of the group
// that reads kh times one block of 32 value columns. A persistent CTA of two
// warpgroups walks its units; warpgroup w takes items w, w+2, ... of each.
// Every warpgroup has its own two-stage ring of state tiles (32 columns x Dk,
// contiguous in the page) in shared memory, filled by bulk asynchronous
// copies that run ahead across unit boundaries, so the HBM read of the next
// tile overlaps the token work on the current one; the checkpoint goes back
// to HBM straight from registers. Per unit the CTA stages once, for all rows
// (replayed rows, then candidates): q^ and k^, the unit's value columns, and
// the gates of the heads its items belong to.
#include "common.cuh"
#include "kernels.h"
#include "rule.cuh"
#include "umma.cuh"

namespace gdn {

using namespace umma;

constexpr int kVerThreads = 256;                 // two warpgroups
constexpr int kVerStagesPerWG = 2;
constexpr int kVerStages = 2 * kVerStagesPerWG;
constexpr int kVerMaxItems = 4;                  // items per unit
constexpr long long kVerWaitLimit = 1LL << 26;

template <class ST, int DK>
struct VerLayout {
  static constexpr uint32_t TILE = kBV * DK;     // state elements per item
  static constexpr uint32_t TILE_BYTES = TILE * sizeof(ST);
  static constexpr uint32_t OFF_Q = kVerStages * TILE_BYTES;
  static constexpr uint32_t OFF_K = OFF_Q + kTC * DK * 4;
  static constexpr uint32_t OFF_V = OFF_K + kTC * DK * 4;
  // then v [kTC][ipu*kBV] floats, q^.k^ [kTC] floats, and (alpha, beta)
  // [kTC][kVerMaxItems] for the (at most ipu) heads the unit's items touch
  __host__ __device__ static uint32_t off_kq(int ipu) { return OFF_V + kTC * ipu * kBV * 4; }
  __host__ __device__ static uint32_t off_ab(int ipu) { return off_kq(ipu) + kTC * 4; }
  __host__ __device__ static uint32_t bytes(int ipu) { return off_ab(ipu) + kTC * kVerMaxItems * 8; }
};

template <class IO, class ST, int DK>
__global__ void __launch_bounds__(kVerThreads, 2)
verify_kernel(Geom G, Batch B, Params P, int ipu, const IO* __restrict__ y,
              const IO* __restrict__ a_in, const IO* __restrict__ b_in, void* o, int out_f32,
              void* pages, int32_t* status) {
  using Lay = VerLayout<ST, DK>;
  constexpr int PE = DK / 8;
  extern __shared__ __align__(128) uint8_t vsm[];
  ST* tiles = reinterpret_cast<ST*>(vsm);
  float* sq = reinterpret_cast<float*>(vsm + Lay::OFF_Q);
  float* sk = reinterpret_cast<float*>(vsm + Lay::OFF_K);
  float* sv = reinterpret_cast<float*>(vsm + Lay::OFF_V);
  float* skq = reinterpret_cast<float*>(vsm + Lay::off_kq(ipu));
  float2* sab = reinterpret_cast<float2*>(vsm + Lay::off_ab(ipu));
  __shared__ __align__(8) uint64_t full[kVerStages];
  __shared__ int s_fail;

  const int tid = threadIdx.x;
  const int w = tid >> 7, wtid = tid & 127;
  const int warp = wtid >> 5, lane = tid & 31, cg = lane >> 3, r8 = lane & 7;
  const int vcol = warp * 8 + cg * 2;
  int col[kColsPerLane];
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m) col[m] = vcol + m;

  const int Gh = G.Hv / G.Hk, nCB = G.Dv / kBV;
  const int nparts = (Gh * nCB) / ipu;
  const int per_req = G.Hk * nparts;
  const int n_units = B.R * per_req;
  const int ncols = ipu * kBV;

  if (tid == 0) {
    for (int s = 0; s < kVerStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    mbar_fence_init();
    s_fail = 0;
  }
  __syncthreads();

  // ---- producer: thread 0 of each warpgroup issues that warpgroup's tiles
  // in the order the warpgroup consumes them (units with items: valid spec
  // requests, judged from the batch alone, exactly as the consumer does).
  int pu = blockIdx.x, pi = w - 2;   // cursor: unit, item (of this warpgroup's parity)
  int issued = 0;                    // tiles this warpgroup has started
  auto advance = [&]() -> bool {
    pi += 2;
    while (pu < n_units) {
      if (pi < ipu) {
        const Req q = load_req(B, pu / per_req);
        if (!q.err && q.spec) return true;
      }
      pu += gridDim.x;
      pi = w;
    }
    return false;
  };
  auto issue = [&]() {
    const Req q = load_req(B, pu / per_req);
    const int rem = pu % per_req, kh = rem / nparts, part = rem % nparts;
    const int ig = part * ipu + pi;
    const int h = kh * Gh + ig / nCB, cb = ig % nCB;
    const ST* src = reinterpret_cast<const ST*>(page_ptr(G, pages, q.page) + G.state_off) +
                    ((size_t)h * G.Dv + (size_t)cb * kBV) * DK;
    const int s = w * kVerStagesPerWG + (issued % kVerStagesPerWG);
    mbar_expect_tx(smem_u32(&full[s]), Lay::TILE_BYTES);
    bulk_load(smem_u32(tiles + (size_t)s * Lay::TILE), src, Lay::TILE_BYTES, smem_u32(&full[s]));
    ++issued;
  };
  bool more = false;
  if (wtid == 0) {
    more = advance();
    for (int k = 0; k < kVerStagesPerWG && more; ++k) {
      issue();
      more = advance();
    }
  }

  int jw = 0;  // tiles this warpgroup has consumed
  bool failed = false;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int slot = u / per_req, rem = u % per_req, kh = rem / nparts, part = rem % nparts;
    const bool reporter = (rem == 0 && tid == 0);
    const Req q = load_req(B, slot);
    if (q.err) {
      if (reporter) report(status, q.err);
      continue;
    }
    if (!q.spec) continue;
    char* pg = page_ptr(G, pages, q.page);
    uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
    const uint32_t flag = *reinterpret_cast<volatile uint32_t*>(flagp);
    SpecState ss = spec_state(G, B, q, flag);
    if (q.fresh) ss.err = GDN_DEV_BAD_FLAG;
    const bool skip = ss.err != 0;   // the unit's tiles are still consumed
    if (skip && reporter) report(status, ss.err);
    const int n_rep = (!skip && ss.width > 0) ? ss.accepted + 1 : 0;
    const int n_all = skip ? 0 : n_rep + q.len;
    IO* rec = reinterpret_cast<IO*>(pg + G.record_off);
    const int g_lo = (part * ipu) / nCB, g_hi = (part * ipu + ipu - 1) / nCB;  // heads touched
    ST* Sbase = reinterpret_cast<ST*>(pg + G.state_off);

    // ---- stage the unit's rows: row t < n_rep is record row t of the live
    // slot, the rest are this step's candidates
    {
      const int t = wtid >> 3, p = tid & 7;
      if (t < n_all) {
        const IO* row = (t < n_rep) ? rec + ((size_t)ss.live * G.Kc + t) * G.rec_row
                                    : y + (size_t)(q.start + t - n_rep) * G.C;
        if (w == 0) {
          RawVec<IO, PE> rq, rk;
          rq.load(row + (size_t)kh * DK + PE * p);
          rk.load(row + (size_t)G.Hk * DK + (size_t)kh * DK + PE * p);
          const float kq = publish_qk<DK, IO>(sq + t * DK + PE * p, sk + t * DK + PE * p, rq, rk, P);
          if (p == 0) skq[t] = kq;
        } else {
          const IO* vsrc = row + 2 * (size_t)G.Hk * DK + (size_t)kh * Gh * G.Dv + (size_t)part * ncols;
          for (int c = 4 * p; c < ncols; c += 32) {
            RawVec<IO, 4> rv;
            rv.load(vsrc + c);
            *reinterpret_cast<float4*>(sv + t * ncols + c) =
                make_float4(rv.get(0), rv.get(1), rv.get(2), rv.get(3));
          }
          if (p == 0) {
            const IO* ar = (t < n_rep) ? row + G.C : a_in + (size_t)(q.start + t - n_rep) * G.Hv;
            const IO* br = (t < n_rep) ? row + G.C + G.Hv : b_in + (size_t)(q.start + t - n_rep) * G.Hv;
            for (int g = g_lo; g <= g_hi; ++g) {
              const int h = kh * Gh + g;
              float alpha, beta;
              gates(P, h, to_f(ar[h]), to_f(br[h]), alpha, beta);
              sab[t * kVerMaxItems + (g - g_lo)] = make_float2(alpha, beta);
            }
          }
        }
      }
      // the candidates' gates go next to their conv'd rows in the other slot
      if (!skip && part == 0) {
        for (int idx = tid; idx < q.len * Gh; idx += kVerThreads) {
          const int tc = idx / Gh, h = kh * Gh + idx % Gh;
          IO* rrow = rec + ((size_t)(1 - ss.live) * G.Kc + tc) * G.rec_row;
          const size_t rn = (size_t)q.start + tc;
          rrow[G.C + h] = a_in[rn * G.Hv + h];
          rrow[G.C + G.Hv + h] = b_in[rn * G.Hv + h];
        }
      }
    }
    __syncthreads();

    // ---- this warpgroup's items
    for (int i = w; i < ipu; i += 2, ++jw) {
      const int s = w * kVerStagesPerWG + (jw % kVerStagesPerWG);
      const bool ok = mbar_wait(smem_u32(&full[s]), (uint32_t)((jw / kVerStagesPerWG) & 1),
                                kVerWaitLimit);
      LaneState<DK / 8> S;
      if (!skip) load_state<DK, ST>(S, tiles + (size_t)s * Lay::TILE, col, r8);
      // past this barrier the whole warpgroup has read the tile
      if (w == 0 ? bar_any<1, 128>(!ok) : bar_any<2, 128>(!ok)) {
        failed = true;
        break;
      }
      if (wtid == 0 && more) {
        issue();
        more = advance();
      }
      if (skip) continue;
      const int ig = part * ipu + i;
      const int g = ig / nCB, cb = ig % nCB, h = kh * Gh + g;
      const float* vb = sv + i * kBV;
      for (int t = 0; t < n_rep; ++t) {
        const float2 ab = sab[t * kVerMaxItems + (g - g_lo)];
        token_update_rows<DK, ST>(S, sk + t * DK, vb + t * ncols, ab.x, ab.y, r8, vcol);
      }
      if (n_rep > 0) {
        int gcol[kColsPerLane];
#pragma unroll
        for (int m = 0; m < kColsPerLane; ++m) gcol[m] = cb * kBV + col[m];
        store_state<DK, ST>(Sbase + (size_t)h * G.Dv * DK, S, gcol, r8);
        // continue from exactly what was stored (a bf16 page rounds here)
#pragma unroll
        for (int m = 0; m < kColsPerLane; ++m)
#pragma unroll
          for (int j = 0; j < DK / 16; ++j)
            S.s[m][j] = make_float2(through<ST>(S.s[m][j].x), through<ST>(S.s[m][j].y));
      }
      for (int t = 0; t < q.len; ++t) {
        const int tt = n_rep + t;
        const float2 ab = sab[tt * kVerMaxItems + (g - g_lo)];
        const float ov = token_step_rows<DK, ST>(S, sq + tt * DK, sk + tt * DK, vb + tt * ncols,
                                                 make_float4(ab.x, ab.y, skq[tt], 0.0f), r8,
                                                 vcol, P.scale, t + 1 < q.len);
        if ((r8 & 3) == 0) {
          const size_t off =
              (((size_t)q.start + t) * G.Hv + h) * G.Dv + cb * kBV + vcol + (r8 >> 2);
          store_out(o, out_f32, off, ov);
        }
      }
    }
    if (failed) s_fail = 1;
    __syncthreads();
    if (s_fail) break;
    // the last unit of this request to finish publishes the new flag word
    if (!skip && tid == 0) {
      __threadfence();
      const uint32_t old = atomicAdd(flagp, 256u);
      if ((old >> 8) == (uint32_t)per_req - 1) {
        __threadfence();
        const int live = (q.len > 0) ? 1 - ss.live : ss.live;
        atomicExch(flagp, make_flag(live, 1 - ss.parity, q.len));
      }
    }
  }
  if (s_fail) {
    if (tid == 0) report(status, GDN_DEV_TIMEOUT);
    // let this warpgroup's copies still in flight land before the CTA's
    // shared memory goes away
    if (wtid == 0)
      for (int j = jw; j < issued; ++j)
        mbar_wait(smem_u32(&full[w * kVerStagesPerWG + (j % kVerStagesPerWG)]),
                  (uint32_t)((j / kVerStagesPerWG) & 1), kVerWaitLimit);
  }
}

// Items per unit: 4, 2 or 1, whichever divides the group's item count.
static int verify_ipu(const Geom& G) {
  const int n_items = (G.Hv / G.Hk) * (G.Dv / kBV);
  return (n_items % 4 == 0) ? 4 : (n_items % 2 == 0) ? 2 : 1;
}

static int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev] = n;
  return n;
}

template <class IO, class ST, int DK>
static cudaError_t launch_verify_t(const Geom& G, const Batch& B, const Params& P, int out_f32,
                                   const void* y, const void* a, const void* b, void* o,
                                   void* pages, int32_t* status, cudaStream_t stream) {
  using Lay = VerLayout<ST, DK>;
  const int ipu = verify_ipu(G);
  const int Gh = G.Hv / G.Hk;
  // the attribute is raised once to the largest size any shape can ask for
  cudaError_t e = ensure_smem_limit<verify_kernel<IO, ST, DK>>((int)Lay::bytes(kVerMaxItems));
  if (e != cudaSuccess) return e;
  const long long units = (long long)B.R * G.Hk * ((Gh * (G.Dv / kBV)) / ipu);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = (int)((units < 2LL * sms) ? units : 2LL * sms);
  if (grid == 0) return cudaSuccess;
  verify_kernel<IO, ST, DK><<<grid, kVerThreads, Lay::bytes(ipu), stream>>>(
      G, B, P, ipu, static_cast<const IO*>(y), static_cast<const IO*>(a),
      static_cast<const IO*>(b), o, out_f32, pages, status);
  return cudaGetLastError();
}

template <class IO, class ST>
static cudaError_t launch_verify_io_st(const Geom& G, const Batch& B, const Params& P, int out_f32,
                                       const void* y, const void* a, const void* b, void* o,
                                       void* pages, int32_t* status, cudaStream_t s) {
  switch (G.Dk) {
    case 32: return launch_verify_t<IO, ST, 32>(G, B, P, out_f32, y, a, b, o, pages, status, s);
    case 64: return launch_verify_t<IO, ST, 64>(G, B, P, out_f32, y, a, b, o, pages, status, s);
    default: return launch_verify_t<IO, ST, 128>(G, B, P, out_f32, y, a, b, o, pages, status, s);
  }
}

cudaError_t launch_verify(const Geom& G, const Batch& B, const Params& P, int io_bf16,
                          int state_bf16, int out_f32, const void* y, const void* a, const void* b,
                          void* o, void* pages, int32_t* status, cudaStream_t stream) {
  if (io_bf16) {
    if (state_bf16)
      return launch_verify_io_st<bf16, bf16>(G, B, P, out_f32, y, a, b, o, pages, status, stream);
    return launch_verify_io_st<bf16, float>(G, B, P, out_f32, y, a, b, o, pages, status, stream);
  }
  if (state_bf16)
    return launch_verify_io_st<float, bf16>(G, B, P, out_f32, y, a, b, o, pages, status, stream);
  return launch_verify_io_st<float, float>(G, B, P, out_f32, y, a, b, o, pages, status, stream);
}

}  // namespace gdn
