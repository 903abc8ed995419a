// Speculative decode in closed form per run of rows (sm_103a): the one-page
// verify (gdn_spec_verify), the same step with the conv fused in
// (gdn_spec_step), and the slot-per-candidate layout (gdn_spec_slots).
//
// r9700-stack v0.2.4, "What it does": one state page per request holds the
// state, a two-slot record of the previous step's candidate rows and a flag
// word; a step replays the accepted rows from the record into the state,
// stores the checkpoint, then runs the new candidates, and its results equal
// those of the stock design that keeps a state page per candidate.
//
// The rule, per value head with state S (Dk x Dv) and L2-normalised k^, q^:
//   S <- alpha_t S; u_t = beta_t (v_t - S^T k^_t); S <- S + k^_t u_t^T;
//   o_t = scale S^T q^_t.
// Over a run of rows t = 0..n-1 that starts from a state S, with the decay
// products R[t][s] = alpha_{s+1} ... alpha_t (R[t][t] = 1) and
// G_t = alpha_0 ... alpha_t, it unrolls to
//   u_t = beta_t (v_t - G_t S^T k^_t - sum_{s<t} R[t][s] (k^_s.k^_t) u_s)
//   o_t = scale (G_t S^T q^_t + sum_{s<=t} R[t][s] (k^_s.q^_t) u_s)
//   S_t = G_t S + sum_{s<=t} R[t][s] k^_s u_s^T           (state after row t)
// so a run costs one read of S for all its dot products, a short scalar
// recurrence per value column, and (only where a state is kept) one rank-n
// update. The verify runs two such runs: the replayed rows (state only: the
// checkpoint is S_a) and the candidates (outputs only). The slot layout runs
// the candidates and stores every S_t. Both compute each quantity with the
// same code and in the same order from the same inputs (a replayed row and
// the candidate row it was are the same bits, its dot products come from the
// same stored state), so the one-page checkpoint equals the slot that was
// kept for it, bit for bit, and so do all outputs.
//
// Work decomposition. One CTA per (request, q/k head kh, split): the Hv/Hk
// value heads that read q/k head kh, in items of 64 value columns; a
// request's items may be split over several CTAs when the batch alone would
// not fill the GPU (not with the conv fused in: every CTA of a group reads
// the q/k window columns that the group's writer rolls, so the fused step
// runs one CTA per group). A CTA normalises the group's q/k rows, forms their Gram
// products and the gates once, and derives the run coefficients per head in
// shared memory. Items then run with no block-wide barrier: 4 warps x 16
// columns; inside a warp, 8 column pairs x 4 lanes, a lane holding 2 columns
// x Dk/4 entries of S in registers (16-byte chunks at Dk index
// VEC (4 i + r4), so a warp's accesses are contiguous per column). The next
// item's state is loaded into registers while the current one is computed.
#pragma once

#include "common.cuh"

namespace gdn {

enum SpecMode { SPEC_VERIFY = 0, SPEC_FUSED = 1, SPEC_SLOTS = 2 };

constexpr int kSpecThreads = 128;
constexpr int kSpecBV = 64;   // value columns per item
constexpr int kSpecK = 8;     // rows in a run at most (max_candidates)

template <int DK, class ST>
struct SpecMap {
  static constexpr int E = DK / 4;                      // entries per column per lane
  static constexpr int VEC0 = 16 / (int)sizeof(ST);
  static constexpr int VEC = (E < VEC0) ? E : VEC0;     // contiguous entries per chunk
  static constexpr int NI = E / VEC;                    // chunks per column
  static constexpr int P = E / 2;                       // float2 pairs per column
  __device__ static int idx(int r4, int i) { return VEC * (4 * i + r4); }
};

// A lane's part of S: 2 columns x E entries, as float2 pairs.
template <int DK>
struct SpecS {
  float2 s[2][DK / 8];
};

// Coefficients of one run (one value head): see the header comment.
struct RunCoef {
  float gk[kSpecK];            // G_t / |k_t|
  float gq[kSpecK];            // G_t / |q_t|
  float gam[kSpecK];           // G_t
  float beta[kSpecK];          // beta_t
  float aneg[kSpecK][kSpecK];  // -R[t][s] k^_s.k^_t   (s < t)
  float bco[kSpecK][kSpecK];   //  R[t][s] k^_s.q^_t   (s <= t)
  float rk[kSpecK][kSpecK];    //  R[t][s] / |k_s|     (s <= t)
};

// Raw dot products of a CTA's rows (k_s.k_t with s <= t, k_s.q_t, q_t.q_t).
struct RunDots {
  float kkr[kSpecK][kSpecK];   // replayed rows: [t][s]
  float kkc[kSpecK][kSpecK];   // candidates: [t][s]
  float kqc[kSpecK][kSpecK];   // candidates: k_s.q_t at [t][s]
  float qqc[kSpecK];
};

// Dynamic shared memory of the spec kernel (byte offsets, 16-byte aligned).
struct SpecSmem {
  uint32_t raw;     // [2 Kc][RW] io dtype: rows q | k | v of the group
  uint32_t ab;      // [2 Kc][2 Gh] float: a then b per head of the group
  uint32_t kx;      // [2 Kc][DKP] float: k rows (replayed, then candidates)
  uint32_t qx;      // [Kc][DKP] float: candidate q rows
  uint32_t dots;    // RunDots
  uint32_t gates;   // [Gh][2 runs][2][Kc] float: alpha, beta
  uint32_t coef;    // RunCoef [Gh][2 runs]
  uint32_t stage;   // [NC][threads] 16-byte chunks: one item's state per thread
  uint32_t total;
  int RW, DKP;
};

__host__ __device__ inline uint32_t spec_al16(uint32_t x) { return (x + 15u) & ~15u; }

__host__ __device__ inline SpecSmem spec_smem(int DK, int DV, int Gh, int io_bytes,
                                               int st_bytes) {
  SpecSmem L;
  L.RW = (2 * DK + Gh * DV + 7) / 8 * 8;
  L.DKP = DK + 4;
  uint32_t off = 0;
  L.raw = off;   off = spec_al16(off + (uint32_t)(2 * kSpecK * L.RW * io_bytes));
  L.ab = off;    off = spec_al16(off + (uint32_t)(2 * kSpecK * 2 * Gh * 4));
  L.kx = off;    off = spec_al16(off + (uint32_t)(2 * kSpecK * L.DKP * 4));
  L.qx = off;    off = spec_al16(off + (uint32_t)(kSpecK * L.DKP * 4));
  L.dots = off;  off = spec_al16(off + (uint32_t)sizeof(RunDots));
  L.gates = off; off = spec_al16(off + (uint32_t)(Gh * 2 * 2 * kSpecK * 4));
  L.coef = off;  off = spec_al16(off + (uint32_t)(Gh * 2 * sizeof(RunCoef)));
  L.stage = off; off = spec_al16(off + (uint32_t)(2 * DK * st_bytes / 4 * kSpecThreads));
  L.total = off;
  return L;
}

// A lane's state chunks are 16 bytes each: (column m, chunk i) is chunk
// c = m NI + i. They are staged in shared memory thread-major (chunk c of
// thread t at (c threads + t) 16 bytes), so a warp's 16-byte accesses are
// contiguous, and each thread reads back only what it copied itself: its own
// cp.async wait is the only synchronisation.
template <int DK, class ST>
__device__ __forceinline__ void spec_stage_async(uint8_t* stage, const ST* col0, int r4, int tid) {
  using M = SpecMap<DK, ST>;
  static_assert(M::VEC * sizeof(ST) == 16, "state chunks are 16 bytes");
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int i = 0; i < M::NI; ++i) {
      const uint32_t dst = (uint32_t)__cvta_generic_to_shared(
          stage + ((size_t)(m * M::NI + i) * kSpecThreads + tid) * 16);
      const ST* src = col0 + (size_t)m * DK + M::idx(r4, i);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
    }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void spec_stage_wait() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <int DK, class ST>
__device__ __forceinline__ void spec_unstage(SpecS<DK>& S, const uint8_t* stage, int tid) {
  using M = SpecMap<DK, ST>;
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int i = 0; i < M::NI; ++i)
      load_f<ST, M::VEC>(reinterpret_cast<const ST*>(
                             stage + ((size_t)(m * M::NI + i) * kSpecThreads + tid) * 16),
                         reinterpret_cast<float*>(&S.s[m][0]) + i * M::VEC);
}

template <int DK, class ST>
__device__ __forceinline__ void spec_store(ST* col0, const SpecS<DK>& S, int r4) {
  using M = SpecMap<DK, ST>;
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int i = 0; i < M::NI; ++i)
      store_f<ST, M::VEC>(col0 + (size_t)m * DK + M::idx(r4, i),
                          reinterpret_cast<const float*>(&S.s[m][0]) + i * M::VEC);
}

// The complete dot products of the lane's column (column b1 of its pair)
// with NG rows of X (fp32, rows at x[g]): per-lane partial sums over its
// entries, then across the 4 lanes of the pair: lane bit 1 first (which also
// hands each lane its column), then lane bit 0. Every dot product, whichever
// rows it is grouped with, is summed in this one order.
template <int DK, class ST, int NG>
__device__ __forceinline__ void spec_dots(const SpecS<DK>& S, const float* const (&x)[NG], int r4,
                                          bool b1, float (&out)[NG]) {
  using M = SpecMap<DK, ST>;
  float2 acc[2][NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) acc[0][g] = acc[1][g] = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < M::NI; ++i)
#pragma unroll
    for (int e = 0; e < M::VEC; e += 4) {
      const int p = (i * M::VEC + e) / 2;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const float4 v = *reinterpret_cast<const float4*>(x[g] + M::idx(r4, i) + e);
        const float2 lo = make_float2(v.x, v.y), hi = make_float2(v.z, v.w);
        acc[0][g] = __ffma2_rn(S.s[0][p], lo, acc[0][g]);
        acc[1][g] = __ffma2_rn(S.s[1][p], lo, acc[1][g]);
        acc[0][g] = __ffma2_rn(S.s[0][p + 1], hi, acc[0][g]);
        acc[1][g] = __ffma2_rn(S.s[1][p + 1], hi, acc[1][g]);
      }
    }
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const float p0 = __fadd_rn(acc[0][g].x, acc[0][g].y);
    const float p1 = __fadd_rn(acc[1][g].x, acc[1][g].y);
    const float keep = b1 ? p1 : p0, send = b1 ? p0 : p1;
    float v = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
    out[g] = v;
  }
}

// u_t of a run for one value column: v holds v_t, dk the raw S^T k_t.
__device__ __forceinline__ void spec_u(const RunCoef& C, int n, const float (&v)[kSpecK],
                                       const float (&dk)[kSpecK], float (&u)[kSpecK]) {
#pragma unroll
  for (int t = 0; t < kSpecK; ++t) {
    u[t] = 0.0f;
    if (t < n) {
      float acc = __fmaf_rn(-C.gk[t], dk[t], v[t]);
#pragma unroll
      for (int s = 0; s < t; ++s) acc = __fmaf_rn(C.aneg[t][s], u[s], acc);
      u[t] = __fmul_rn(C.beta[t], acc);
    }
  }
}

// S <- the state after row a of a run that started from S:
//   G_a S + sum_{s<=a} k_s (R[a][s] / |k_s|) u_s^T,
// k rows (raw, fp32) at kx + s * kstride; u0/u1 hold u_s of the lane's two
// columns.
template <int DK, class ST>
__device__ __forceinline__ void spec_advance(SpecS<DK>& S, const RunCoef& C, int a,
                                             const float* kx, int kstride,
                                             const float (&u0)[kSpecK],
                                             const float (&u1)[kSpecK], int r4) {
  using M = SpecMap<DK, ST>;
  const float g = C.gam[a];
  const float2 g2 = make_float2(g, g);
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int p = 0; p < M::P; ++p) S.s[m][p] = __fmul2_rn(g2, S.s[m][p]);
#pragma unroll
  for (int s = 0; s < kSpecK; ++s) {
    if (s <= a) {
      const float c = C.rk[a][s];
      const float w0 = __fmul_rn(c, u0[s]), w1 = __fmul_rn(c, u1[s]);
      const float2 w02 = make_float2(w0, w0), w12 = make_float2(w1, w1);
      const float* xr = kx + s * kstride;
#pragma unroll
      for (int i = 0; i < M::NI; ++i)
#pragma unroll
        for (int e = 0; e < M::VEC; e += 4) {
          const int p = (i * M::VEC + e) / 2;
          const float4 v = *reinterpret_cast<const float4*>(xr + M::idx(r4, i) + e);
          const float2 lo = make_float2(v.x, v.y), hi = make_float2(v.z, v.w);
          S.s[0][p] = __ffma2_rn(lo, w02, S.s[0][p]);
          S.s[1][p] = __ffma2_rn(lo, w12, S.s[1][p]);
          S.s[0][p + 1] = __ffma2_rn(hi, w02, S.s[0][p + 1]);
          S.s[1][p + 1] = __ffma2_rn(hi, w12, S.s[1][p + 1]);
        }
    }
  }
}

// Plain dot product of two fp32 rows in shared memory, in a fixed order.
template <int DK>
__device__ __forceinline__ float spec_rowdot(const float* a, const float* b) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int d = 0; d < DK; d += 4) {
    const float4 x = *reinterpret_cast<const float4*>(a + d);
    const float4 y = *reinterpret_cast<const float4*>(b + d);
    acc.x = __fmaf_rn(x.x, y.x, acc.x);
    acc.y = __fmaf_rn(x.y, y.y, acc.y);
    acc.z = __fmaf_rn(x.z, y.z, acc.z);
    acc.w = __fmaf_rn(x.w, y.w, acc.w);
  }
  return __fadd_rn(__fadd_rn(acc.x, acc.y), __fadd_rn(acc.z, acc.w));
}

// (s, t) with s <= t of triangular task index k (row t holds t + 1 tasks).
__device__ __forceinline__ void spec_tri(int k, int& s, int& t) {
  t = 0;
  while (k > t) {
    k -= t + 1;
    ++t;
  }
  s = k;
}

template <class IO, class ST, int DK, int MODE>
__global__ void __launch_bounds__(kSpecThreads, 2)
spec_kernel(Geom G, Batch B, Params P, SlotGeom SG, const IO* __restrict__ rows_in,
            const IO* __restrict__ conv_w, const IO* __restrict__ a_in,
            const IO* __restrict__ b_in, void* o, int out_f32, void* pages, int32_t* status,
            int splits) {
  using M = SpecMap<DK, ST>;
  constexpr int DV = DK;
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_begin();

  const int Gh = G.Hv / G.Hk;
  const int kh = blockIdx.x / splits, split = blockIdx.x % splits;
  const int BVI = DV < kSpecBV ? DV : kSpecBV;     // columns per item
  const int nCB = DV / BVI;
  const int n_items = Gh * nCB;
  const int per = (n_items + splits - 1) / splits;
  const int it0 = split * per, it1 = min(n_items, it0 + per);
  const int h0 = kh * Gh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r4 = lane & 3, cg = lane >> 2;
  const bool b1 = (r4 & 2) != 0, b0 = (r4 & 1) != 0;
  const int colw = 16 * warp + 2 * cg;             // the lane's first column in an item
  const bool active = colw < BVI;
  const bool reporter = (blockIdx.x == 0 && tid == 0);

  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  if (MODE != SPEC_SLOTS && !q.spec) return;

  // where the starting state lives: the page (one-page modes) or the slot
  // the request resumes from
  char* pg = page_ptr(G, pages, q.page);
  ST* Sbase;
  int n_r = 0, live = 0, parity = 0;
  uint32_t* flagp = nullptr;
  if constexpr (MODE == SPEC_SLOTS) {
    const int src = B.n_accepted ? B.n_accepted[q.r] : -1;
    if (src < 0 || src >= G.Kc) {
      if (reporter) report(status, GDN_DEV_BAD_ACCEPTED);
      return;
    }
    if (q.len > G.Kc) {
      if (reporter) report(status, GDN_DEV_TOO_MANY_CANDIDATES);
      return;
    }
    pg = reinterpret_cast<char*>(pages) + (size_t)q.page * SG.pool_bytes;
    Sbase = reinterpret_cast<ST*>(pg + (size_t)src * SG.slot_bytes + SG.state_off);
  } else {
    Sbase = reinterpret_cast<ST*>(pg + G.state_off);
  }
  auto item_col0 = [&](int it) -> ST* {
    const int h = h0 + it / nCB, cb = it % nCB;
    return Sbase + ((size_t)h * DV + (size_t)cb * BVI + colw) * DK;
  };
  const SpecSmem L = spec_smem(DK, DV, Gh, (int)sizeof(IO), (int)sizeof(ST));
  uint8_t* stage = smem + L.stage;
  // the first item's state is requested before the flag is checked (one
  // round trip, not two); a refused request only lets the copy land
  if (active && it0 < it1) spec_stage_async<DK, ST>(stage, item_col0(it0), r4, tid);

  if constexpr (MODE != SPEC_SLOTS) {
    flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
    const uint32_t flag = *reinterpret_cast<volatile uint32_t*>(flagp);
    SpecState ss = spec_state(G, B, q, flag);
    if (q.fresh) ss.err = GDN_DEV_BAD_FLAG;
    if (ss.err) {
      if (reporter) report(status, ss.err);
      spec_stage_wait();   // the copy lands before the CTA's shared memory goes away
      return;
    }
    n_r = (ss.width > 0) ? ss.accepted + 1 : 0;
    live = ss.live;
    parity = ss.parity;
  }
  const int n_c = q.len;
  const int n_all = n_r + n_c;
  IO* raw = reinterpret_cast<IO*>(smem + L.raw);
  float* abs_ = reinterpret_cast<float*>(smem + L.ab);
  float* kx = reinterpret_cast<float*>(smem + L.kx);
  float* qx = reinterpret_cast<float*>(smem + L.qx);
  RunDots& D = *reinterpret_cast<RunDots*>(smem + L.dots);
  float* gts = reinterpret_cast<float*>(smem + L.gates);
  RunCoef* coef = reinterpret_cast<RunCoef*>(smem + L.coef);
  const int RW = L.RW, DKP = L.DKP;
  IO* rec = reinterpret_cast<IO*>(pg + G.record_off);   // one-page modes only
  const int g_lo = it0 / nCB, g_hi = (it1 > it0) ? (it1 - 1) / nCB + 1 : g_lo;  // own heads
  const int q_off = kh * DK, k_off = G.Hk * DK + kh * DK, v_off = 2 * G.Hk * DK + h0 * DV;
  // head g's record gates and conv channels are written by the CTA holding
  // its first item; the q/k channels by split 0
  auto owns_head = [&](int g) { return (g * nCB) / per == split; };

  // ---- 1. the group's rows into shared memory (raw, io dtype) ----------
  {
    constexpr int VE = 16 / (int)sizeof(IO);          // elements per 16-byte piece
    const int pieces = RW / VE;
    // replayed rows: k and v from the live record slot (their q is not used)
    for (int idx = tid; idx < n_r * pieces; idx += kSpecThreads) {
      const int t = idx / pieces, c = (idx % pieces) * VE;
      if (c < DK) continue;
      const int ch = (c < 2 * DK) ? k_off + (c - DK) : v_off + (c - 2 * DK);
      if (c >= 2 * DK + Gh * DV) continue;
      const IO* src = rec + ((size_t)live * G.Kc + t) * G.rec_row + ch;
      *reinterpret_cast<uint4*>(raw + (size_t)t * RW + c) = *reinterpret_cast<const uint4*>(src);
    }
    if constexpr (MODE != SPEC_FUSED) {
      for (int idx = tid; idx < n_c * pieces; idx += kSpecThreads) {
        const int t = idx / pieces, c = (idx % pieces) * VE;
        if (c >= 2 * DK + Gh * DV) continue;
        const int ch = (c < DK) ? q_off + c : (c < 2 * DK) ? k_off + (c - DK) : v_off + (c - 2 * DK);
        const IO* src = rows_in + (size_t)(q.start + t) * G.C + ch;
        *reinterpret_cast<uint4*>(raw + (size_t)(n_r + t) * RW + c) =
            *reinterpret_cast<const uint4*>(src);
      }
    } else {
      // the conv of the group's channels for this step's candidates, exactly
      // as gdn_conv computes it for a spec request: history = window
      // columns n_r .. n_r+W-2 (the record's accepted rows rolled out),
      // taps oldest first, own SiLU, rounded to the io dtype
      const int nvec = (2 * DK + Gh * DV) / 4;
      IO* win = reinterpret_cast<IO*>(pg + G.window_off);
      IO* rec_out = rec + (size_t)(1 - live) * G.Kc * G.rec_row;
      for (int vi = tid; vi < nvec; vi += kSpecThreads) {
        const int c4 = 4 * vi;
        const int gg = (c4 < 2 * DK) ? -1 : (c4 - 2 * DK) / DV;
        if (gg >= 0 && (gg < g_lo || gg >= g_hi)) continue;   // another split's head
        const bool owner = (gg < 0) ? (split == 0) : owns_head(gg);
        const int ch = (c4 < DK) ? q_off + c4 : (c4 < 2 * DK) ? k_off + (c4 - DK) : v_off + (c4 - 2 * DK);
        float wt[4][4];
        {
          float tmp[16];
          load_f<IO, 16>(conv_w + (size_t)ch * 4, tmp);
#pragma unroll
          for (int v = 0; v < 4; ++v)
#pragma unroll
            for (int j = 0; j < 4; ++j) wt[j][v] = tmp[v * 4 + j];
        }
        float hcol[3][4], h0c[3][4];
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          load_f<IO, 4>(win + (size_t)(n_r + j) * G.C + ch, hcol[j]);
#pragma unroll
          for (int v = 0; v < 4; ++v) h0c[j][v] = hcol[j][v];
        }
        for (int t = 0; t < n_c; ++t) {
          float xv[4];
          load_f<IO, 4>(rows_in + (size_t)(q.start + t) * G.C + ch, xv);
          float yv[4];
#pragma unroll
          for (int v = 0; v < 4; v += 2) {
            float2 acc = P.conv_bias ? make_float2(P.conv_bias[ch + v], P.conv_bias[ch + v + 1])
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
          store_f<IO, 4>(raw + (size_t)(n_r + t) * RW + c4, yv);
          if (owner) {
            store_f<IO, 4>(rec_out + (size_t)t * G.rec_row + ch, yv);
            store_f<IO, 4>(win + (size_t)(3 + t) * G.C + ch, xv);
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            hcol[0][v] = hcol[1][v];
            hcol[1][v] = hcol[2][v];
            hcol[2][v] = xv[v];
          }
        }
        if (owner) {
          // window columns 0..2: the history this step started from
#pragma unroll
          for (int j = 0; j < 3; ++j) store_f<IO, 4>(win + (size_t)j * G.C + ch, h0c[j]);
        }
      }
    }
    // gate inputs per row and own head: record rows, then this step's rows
    for (int idx = tid; idx < n_all * (g_hi - g_lo); idx += kSpecThreads) {
      const int t = idx / (g_hi - g_lo), g = g_lo + idx % (g_hi - g_lo), h = h0 + g;
      float av, bv;
      if (t < n_r) {
        const IO* row = rec + ((size_t)live * G.Kc + t) * G.rec_row;
        av = to_f(row[G.C + h]);
        bv = to_f(row[G.C + G.Hv + h]);
      } else {
        const size_t rn = (size_t)q.start + (t - n_r);
        av = to_f(a_in[rn * G.Hv + h]);
        bv = to_f(b_in[rn * G.Hv + h]);
        if (MODE != SPEC_SLOTS && owns_head(g)) {
          // the candidates' gates go next to their conv'd rows in the other slot
          IO* row = rec + ((size_t)(1 - live) * G.Kc + (t - n_r)) * G.rec_row;
          row[G.C + h] = a_in[rn * G.Hv + h];
          row[G.C + G.Hv + h] = b_in[rn * G.Hv + h];
        }
      }
      abs_[t * 2 * Gh + g] = av;
      abs_[t * 2 * Gh + Gh + g] = bv;
    }
  }
  __syncthreads();

  // ---- 2. fp32 copies of the k rows (all) and q rows (candidates) -------
  for (int idx = tid; idx < (n_all + n_c) * (DK / 4); idx += kSpecThreads) {
    const int r = idx / (DK / 4), d = (idx % (DK / 4)) * 4;
    float f[4];
    if (r < n_all) {
      load_f<IO, 4>(raw + (size_t)r * RW + DK + d, f);
      *reinterpret_cast<float4*>(kx + r * DKP + d) = make_float4(f[0], f[1], f[2], f[3]);
    } else {
      const int t = r - n_all;
      load_f<IO, 4>(raw + (size_t)(n_r + t) * RW + d, f);
      *reinterpret_cast<float4*>(qx + t * DKP + d) = make_float4(f[0], f[1], f[2], f[3]);
    }
  }
  __syncthreads();

  // ---- 3. Gram products and norms (one per thread), gates ---------------
  {
    const int A = n_r * (n_r + 1) / 2, Bc = n_c * (n_c + 1) / 2;
    int k = tid;
    if (k < A) {
      int s, t;
      spec_tri(k, s, t);
      D.kkr[t][s] = spec_rowdot<DK>(kx + s * DKP, kx + t * DKP);
    } else if ((k -= A) < Bc) {
      int s, t;
      spec_tri(k, s, t);
      D.kkc[t][s] = spec_rowdot<DK>(kx + (n_r + s) * DKP, kx + (n_r + t) * DKP);
    } else if ((k -= Bc) < Bc) {
      int s, t;
      spec_tri(k, s, t);
      D.kqc[t][s] = spec_rowdot<DK>(kx + (n_r + s) * DKP, qx + t * DKP);
    } else if ((k -= Bc) < n_c) {
      D.qqc[k] = spec_rowdot<DK>(qx + k * DKP, qx + k * DKP);
    }
    // gates of own heads: thread -> (head, row)
    const int ng = g_hi - g_lo;
    for (int idx = tid; idx < ng * n_all; idx += kSpecThreads) {
      const int g = g_lo + idx / n_all, t = idx % n_all;
      float alpha, beta;
      gates(P, h0 + g, abs_[t * 2 * Gh + g], abs_[t * 2 * Gh + Gh + g], alpha, beta);
      const int run = (t < n_r) ? 0 : 1, tr = (t < n_r) ? t : t - n_r;
      gts[((g * 2 + run) * 2 + 0) * kSpecK + tr] = alpha;
      gts[((g * 2 + run) * 2 + 1) * kSpecK + tr] = beta;
    }
  }
  __syncthreads();

  // ---- 4. run coefficients: thread -> (own head, run, column s = -1..n-1)
  {
    const int ng = g_hi - g_lo;
    for (int idx = tid; idx < ng * 2 * (kSpecK + 1); idx += kSpecThreads) {
      const int g = g_lo + idx / (2 * (kSpecK + 1));
      const int run = (idx / (kSpecK + 1)) & 1;
      const int s = idx % (kSpecK + 1) - 1;
      const int n = run ? n_c : n_r;
      if (s >= n) continue;
      RunCoef& C = coef[g * 2 + run];
      const float* al = gts + ((g * 2 + run) * 2 + 0) * kSpecK;
      const float* be = gts + ((g * 2 + run) * 2 + 1) * kSpecK;
      auto ik_of = [&](int t) {
        return rsqrtf(__fadd_rn(run ? D.kkc[t][t] : D.kkr[t][t], P.eps));
      };
      if (s < 0) {
        float r = 1.0f;
        for (int t = 0; t < n; ++t) {
          r = __fmul_rn(r, al[t]);
          C.gam[t] = r;
          C.gk[t] = __fmul_rn(r, ik_of(t));
          C.gq[t] = run ? __fmul_rn(r, rsqrtf(__fadd_rn(D.qqc[t], P.eps))) : 0.0f;
          C.beta[t] = be[t];
        }
      } else {
        const float iks = ik_of(s);
        float r = 1.0f;
        for (int t = s; t < n; ++t) {
          if (t > s) r = __fmul_rn(r, al[t]);
          C.rk[t][s] = __fmul_rn(r, iks);
          if (t > s) {
            const float kk = run ? D.kkc[t][s] : D.kkr[t][s];
            C.aneg[t][s] = -__fmul_rn(r, __fmul_rn(__fmul_rn(kk, iks), ik_of(t)));
          }
          if (run) {
            const float iqt = rsqrtf(__fadd_rn(D.qqc[t], P.eps));
            C.bco[t][s] = __fmul_rn(r, __fmul_rn(__fmul_rn(D.kqc[t][s], iks), iqt));
          }
        }
      }
    }
  }
  __syncthreads();

  // ---- 5. items: no block-wide barrier from here on ---------------------
  // An item's state comes from the stage (copied by this thread alone). The
  // one-page modes request the next item's copy as soon as the first dot
  // products have consumed the current one; the slot layout keeps the stage
  // for the whole item (it rebuilds each candidate's state from it).
  if (active && (n_all > 0 || MODE == SPEC_SLOTS)) {
    const IO* vraw = raw + 2 * DK;
    for (int it = it0; it < it1; ++it) {
      const int g = it / nCB, cb = it % nCB, h = h0 + g;
      ST* col0 = item_col0(it);
      if (MODE == SPEC_SLOTS && it > it0) spec_stage_async<DK, ST>(stage, col0, r4, tid);
      spec_stage_wait();
      SpecS<DK> S;
      spec_unstage<DK, ST>(S, stage, tid);
      bool ahead = (MODE == SPEC_SLOTS) || (it + 1 >= it1);
      auto prefetch = [&]() {
        if (!ahead) {
          spec_stage_async<DK, ST>(stage, item_col0(it + 1), r4, tid);
          ahead = true;
        }
      };
      const int vcol = g * DV + cb * BVI + colw + (b1 ? 1 : 0);   // this lane's v column

      if (n_r > 0) {
        const RunCoef& C = coef[g * 2 + 0];
        float dk[kSpecK], v[kSpecK], u[kSpecK], uo[kSpecK];
#pragma unroll
        for (int t = 0; t < kSpecK; t += 2) {
          if (t < n_r) {
            const float* xr[2] = {kx + t * DKP, kx + (t + 1) * DKP};
            float out[2];
            spec_dots<DK, ST, 2>(S, xr, r4, b1, out);
            dk[t] = out[0];
            dk[t + 1] = out[1];
            if (t == 0) prefetch();
          }
        }
#pragma unroll
        for (int t = 0; t < kSpecK; ++t) v[t] = (t < n_r) ? to_f(vraw[(size_t)t * RW + vcol]) : 0.0f;
        spec_u(C, n_r, v, dk, u);
#pragma unroll
        for (int t = 0; t < kSpecK; ++t) uo[t] = __shfl_xor_sync(0xffffffffu, u[t], 2);
        float u0[kSpecK], u1[kSpecK];
#pragma unroll
        for (int t = 0; t < kSpecK; ++t) {
          u0[t] = b1 ? uo[t] : u[t];
          u1[t] = b1 ? u[t] : uo[t];
        }
        spec_advance<DK, ST>(S, C, n_r - 1, kx, DKP, u0, u1, r4);
        spec_store<DK, ST>(col0, S, r4);
        // continue from exactly what was stored (a bf16 page rounds here)
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int p = 0; p < M::P; ++p)
            S.s[m][p] = make_float2(through<ST>(S.s[m][p].x), through<ST>(S.s[m][p].y));
      }

      if (n_c > 0) {
        const RunCoef& C = coef[g * 2 + 1];
        float dk[kSpecK], dq[kSpecK], v[kSpecK], u[kSpecK];
        const float* kc = kx + n_r * DKP;
#pragma unroll
        for (int t = 0; t < kSpecK; t += 2) {
          if (t < n_c) {
            const float* xr[4] = {kc + t * DKP, kc + (t + 1) * DKP, qx + t * DKP,
                                  qx + (t + 1) * DKP};
            float out[4];
            spec_dots<DK, ST, 4>(S, xr, r4, b1, out);
            dk[t] = out[0];
            dk[t + 1] = out[1];
            dq[t] = out[2];
            dq[t + 1] = out[3];
            if (t == 0) prefetch();
          }
        }
#pragma unroll
        for (int t = 0; t < kSpecK; ++t)
          v[t] = (t < n_c) ? to_f(vraw[(size_t)(n_r + t) * RW + vcol]) : 0.0f;
        spec_u(C, n_c, v, dk, u);
        // outputs: lane bit 0 picks the rows t = 2 tt + b0
        const size_t ocol = (size_t)h * DV + (size_t)cb * BVI + colw + (b1 ? 1 : 0);
#pragma unroll
        for (int tt = 0; tt < kSpecK / 2; ++tt) {
          const int t = 2 * tt + (b0 ? 1 : 0);
          if (t < n_c) {
            const float dqt = b0 ? dq[2 * tt + 1] : dq[2 * tt];
            float acc = __fmul_rn(C.gq[t], dqt);
#pragma unroll
            for (int s = 0; s <= 2 * tt + 1; ++s)
              if (s <= t) acc = __fmaf_rn(C.bco[t][s], u[s], acc);
            store_out(o, out_f32, ((size_t)q.start + t) * G.Hv * DV + ocol,
                      __fmul_rn(P.scale, acc));
          }
        }
        if constexpr (MODE == SPEC_SLOTS) {
          // the state after every candidate goes to its slot, each rebuilt
          // from the staged starting state
          float uo[kSpecK], u0[kSpecK], u1[kSpecK];
#pragma unroll
          for (int t = 0; t < kSpecK; ++t) uo[t] = __shfl_xor_sync(0xffffffffu, u[t], 2);
#pragma unroll
          for (int t = 0; t < kSpecK; ++t) {
            u0[t] = b1 ? uo[t] : u[t];
            u1[t] = b1 ? u[t] : uo[t];
          }
          const size_t off = (size_t)(col0 - Sbase);
          for (int t = 0; t < n_c; ++t) {
            SpecS<DK> T;
            spec_unstage<DK, ST>(T, stage, tid);
            spec_advance<DK, ST>(T, C, t, kc, DKP, u0, u1, r4);
            ST* dst = reinterpret_cast<ST*>(pg + (size_t)t * SG.slot_bytes + SG.state_off) + off;
            spec_store<DK, ST>(dst, T, r4);
          }
        }
      }
      prefetch();   // (a run with no rows never consumed the stage)
    }
  }
  spec_stage_wait();   // no copy outlives the CTA's shared memory

  // ---- 6. the last CTA of the request publishes the new flag word -------
  // No fence orders the page data first: only later launches read it. The
  // counter needs none either: every CTA read the flag before its own
  // increment of the same word, so the publish follows every read.
  if constexpr (MODE != SPEC_SLOTS) {
    if (tid == 0) {
      const uint32_t total = (uint32_t)(G.Hk * splits);
      const uint32_t old = atomicAdd(flagp, 256u);
      if ((old >> 8) == total - 1) {
        const int nl = (n_c > 0) ? 1 - live : live;
        atomicExch(flagp, make_flag(nl, 1 - parity, n_c));
      }
    }
  }
}

// Dynamic shared memory the spec kernel needs, and the most any launch may
// ask for (the kernels' attribute is raised to it once per device).
constexpr int kSpecSmemMax = 200 * 1024;

template <int DK>
cudaError_t launch_spec_dk(int mode, const Geom& G, const Batch& B, const Params& P,
                           const SlotGeom& SG, int io_bf16, int state_bf16, int out_f32,
                           const void* rows, const void* conv_w, const void* a, const void* b,
                           void* o, void* pages, int32_t* status, int splits,
                           cudaStream_t stream) {
  const int Gh = G.Hv / G.Hk;
  const SpecSmem L = spec_smem(DK, DK, Gh, io_bf16 ? 2 : 4, state_bf16 ? 2 : 4);
  if ((int)L.total > kSpecSmemMax) return cudaErrorInvalidConfiguration;
  dim3 grid(G.Hk * splits, B.R);
  dim3 block(kSpecThreads);
#define GDN_SPEC_LAUNCH(IO, ST, MODE)                                                           \
  do {                                                                                          \
    cudaError_t e = ensure_smem_limit<spec_kernel<IO, ST, DK, MODE>>(kSpecSmemMax);             \
    if (e != cudaSuccess) return e;                                                             \
    return launch_pdl(spec_kernel<IO, ST, DK, MODE>, grid, block, L.total, stream, G, B, P, SG, \
                      static_cast<const IO*>(rows), static_cast<const IO*>(conv_w),             \
                      static_cast<const IO*>(a), static_cast<const IO*>(b), o, out_f32, pages,  \
                      status, splits);                                                          \
  } while (0)
#define GDN_SPEC_MODES(IO, ST)                                          \
  if (mode == SPEC_VERIFY) GDN_SPEC_LAUNCH(IO, ST, SPEC_VERIFY);        \
  else if (mode == SPEC_FUSED) GDN_SPEC_LAUNCH(IO, ST, SPEC_FUSED);     \
  else GDN_SPEC_LAUNCH(IO, ST, SPEC_SLOTS);
  if (io_bf16) {
    if (state_bf16) { GDN_SPEC_MODES(bf16, bf16) } else { GDN_SPEC_MODES(bf16, float) }
  } else {
    if (state_bf16) { GDN_SPEC_MODES(float, bf16) } else { GDN_SPEC_MODES(float, float) }
  }
#undef GDN_SPEC_MODES
#undef GDN_SPEC_LAUNCH
}

}  // namespace gdn
