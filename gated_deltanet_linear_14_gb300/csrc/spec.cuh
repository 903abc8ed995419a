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
// The recurrence for u is a unit lower-triangular system in the run's rows:
// with c_t = v_t - G_t S^T k^_t and L[t][s] = -beta_t R[t][s] (k^_s.k^_t),
// u = (I - L)^-1 diag(beta) c =: M c, and the outputs are
// o = scale (G S^T q^ + N c) with N = B M, B[t][s] = R[t][s] (k^_s.q^_t).
// M and N depend only on the rows (not on S or the value column), so a CTA
// forms them once per value head; every column then needs only independent
// short dot products with its c. A run so costs one read of S for all its
// dot products and (only where a state is kept) one rank-n update. M's
// leading block is the inverse of L's leading block, so a run of the first
// a + 1 rows sees exactly the coefficients the longer run had; the record
// keeps the candidates' G/|k|, G, R/|k| and M beside their rows, and the
// next step's replay uses them as they are. The verify runs two such runs:
// the replayed rows (state only: the checkpoint is S_a) and the candidates
// (outputs only). The slot layout runs the candidates and stores every S_t.
// Both compute each quantity with the same code and in the same order from
// the same inputs (a replayed row and the candidate row it was are the same
// bits, its dot products come from the same stored state), so the one-page
// checkpoint equals the slot that was kept for it, bit for bit, and so do
// all outputs.
//
// Work decomposition. One CTA per (request, q/k head kh, split): the Hv/Hk
// value heads that read q/k head kh, in items of 64 value columns; a
// request's items may be split over several CTAs when the batch alone would
// not fill the GPU (not with the conv fused in: every CTA of a group reads
// the q/k window columns that the group's writer rolls, so the fused step
// runs one CTA per group). A CTA stages the group's rows, forms the
// candidates' Gram products and gates once, and derives their run
// coefficients per head in shared memory. Items then run with no block-wide
// barrier: 4 warps x 16 columns; inside a warp, 4 groups of 4 columns x 8
// lanes, a lane holding 4 columns x Dk/8 entries of S in registers (chunks
// of 16 bytes at Dk index VEC (8 i + r8)). Each 16-byte shared load of a q/k
// row by an 8-lane quarter of the warp reads 128 distinct bytes and feeds 4
// columns. The per-column scalar work (c, u = M c, the outputs) goes through
// a small per-warp scratch: the dot products land there, then each lane
// takes one column and half of the rows, which keeps the per-column arrays
// out of registers (161 of them, 3 CTAs per SM). The next item's state is
// copied into shared memory by the thread that will read it (cp.async)
// while the current one is computed.
#pragma once

#include "common.cuh"

namespace gdn {

enum SpecMode { SPEC_VERIFY = 0, SPEC_FUSED = 1, SPEC_SLOTS = 2 };

constexpr int kSpecThreads = 128;
constexpr int kSpecBV = 64;   // value columns per item
constexpr int kSpecK = 8;     // rows in a run at most (max_candidates)
constexpr int kSpecScr = 3 * kSpecK * 16;   // per-warp scratch floats

template <int DK, class ST>
struct SpecMap {
  static constexpr int E = DK / 8;                      // entries per column per lane
  static constexpr int VEC0 = 16 / (int)sizeof(ST);
  static constexpr int VEC = (E < VEC0) ? E : VEC0;     // contiguous entries per chunk
  static constexpr int NI = E / VEC;                    // chunks per column
  static constexpr int P = E / 2;                       // float2 pairs per column
  static constexpr int CB = VEC * (int)sizeof(ST);      // bytes per chunk (8 or 16)
  __device__ static int idx(int r8, int i) { return VEC * (8 * i + r8); }
  // where a q/k row keeps the 4 entries a lane multiplies with pair p0 .. p0+1
  // of chunk i (piece h = 0 .. VEC/4-1): the rows are stored so that the 8
  // lanes of a quarter-warp read 128 contiguous bytes
  __device__ static int xoff(int r8, int i, int h) { return 4 * (8 * (VEC / 4) * i + 8 * h + r8); }
};

// Storage position of Dk entry d in a staged q/k row (see SpecMap::xoff).
template <int DK, class ST>
__device__ __forceinline__ int spec_xpos(int d) {
  using M = SpecMap<DK, ST>;
  const int i = d / (8 * M::VEC), r8 = (d / M::VEC) % 8, e = d % M::VEC;
  return M::xoff(r8, i, e / 4) + (d % 4);
}

// A lane's part of S: 4 columns x E entries, as float2 pairs.
template <int DK>
struct SpecS {
  float2 s[4][DK / 16];
};

// Coefficients of one run (one value head): see the header comment.
struct RunCoef {
  float gk[kSpecK];            // G_t / |k_t|
  float gq[kSpecK];            // G_t / |q_t|
  float gam[kSpecK];           // G_t
  float beta[kSpecK];          // beta_t
  float l[kSpecK][kSpecK];     // L[t][s] = -beta_t R[t][s] k^_s.k^_t   (s < t)
  float bco[kSpecK][kSpecK];   // B[t][s] = R[t][s] k^_s.q^_t          (s <= t)
  float rk[kSpecK][kSpecK];    // R[t][s] / |k_s|                       (s <= t)
  float m[kSpecK][kSpecK];     // M = (I - L)^-1 diag(beta)             (s <= t)
  float nq[kSpecK][kSpecK];    // N = B M                               (s <= t)
};

// The record keeps, per value head, the fields the next step's replay needs
// (gk, gam, rk, m: kRunCoefFloats values) in this order.
static_assert(offsetof(RunCoef, gk) == 0 && offsetof(RunCoef, gam) == 64 &&
                  offsetof(RunCoef, rk) == 640 && offsetof(RunCoef, m) == 896,
              "record coefficient copy offsets");
static_assert(kRunCoefFloats == 8 + 8 + 64 + 64, "record coefficient block");

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
  uint32_t scr;     // per warp: [2 Kc][16] dot products, [Kc][16] u of its columns
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
  L.stage = off; off = spec_al16(off + (uint32_t)(DK / 2 * st_bytes * kSpecThreads));
  L.scr = off;   off = spec_al16(off + (uint32_t)((kSpecThreads / 32) * kSpecScr * 4));
  L.total = off;
  return L;
}

// A lane's state chunks (column m, chunk i) are c = m NI + i. They are
// staged in shared memory thread-major (chunk c of thread t at (c threads +
// t) CB bytes), so a warp's accesses are contiguous, and each thread reads
// back only what it copied itself: its own cp.async wait is the only
// synchronisation.
template <int DK, class ST>
__device__ __forceinline__ void spec_stage_async(uint8_t* stage, const ST* col0, int r8, int tid) {
  using M = SpecMap<DK, ST>;
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int i = 0; i < M::NI; ++i) {
      const uint32_t dst = (uint32_t)__cvta_generic_to_shared(
          stage + ((size_t)(m * M::NI + i) * kSpecThreads + tid) * M::CB);
      const ST* src = col0 + (size_t)m * DK + M::idx(r8, i);
      if constexpr (M::CB == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
      else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
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
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int i = 0; i < M::NI; ++i)
      load_f<ST, M::VEC>(reinterpret_cast<const ST*>(
                             stage + ((size_t)(m * M::NI + i) * kSpecThreads + tid) * M::CB),
                         reinterpret_cast<float*>(&S.s[m][0]) + i * M::VEC);
}

template <int DK, class ST>
__device__ __forceinline__ void spec_store(ST* col0, const SpecS<DK>& S, int r8) {
  using M = SpecMap<DK, ST>;
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int i = 0; i < M::NI; ++i)
      store_f<ST, M::VEC>(col0 + (size_t)m * DK + M::idx(r8, i),
                          reinterpret_cast<const float*>(&S.s[m][0]) + i * M::VEC);
}

// The complete dot products of the lane's column (column 2 b2 + b1 of its
// group of 4) with NG rows of X (fp32, rows at x[g], stored by spec_xpos):
// per-lane partial sums over its entries, then across the 8 lanes of the
// group: lane bit 2 first (it also hands each lane a pair of columns), then
// bit 1 (one column), then bit 0. Every dot product, whichever rows it is
// grouped with, is summed in this one order.
template <int DK, class ST, int NG>
__device__ __forceinline__ void spec_dots(const SpecS<DK>& S, const float* const (&x)[NG], int r8,
                                          bool b2, bool b1, float (&out)[NG]) {
  using M = SpecMap<DK, ST>;
  float2 acc[4][NG];
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int m = 0; m < 4; ++m) acc[m][g] = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < M::NI; ++i)
#pragma unroll
    for (int h = 0; h < M::VEC / 4; ++h) {
      const int p = (i * M::VEC + 4 * h) / 2;
      // the rows' loads first, then every low-half product, then every
      // high-half one: products into one accumulator are 4 NG apart
      float4 v[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) v[g] = *reinterpret_cast<const float4*>(x[g] + M::xoff(r8, i, h));
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int m = 0; m < 4; ++m)
          acc[m][g] = __ffma2_rn(S.s[m][p], make_float2(v[g].x, v[g].y), acc[m][g]);
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int m = 0; m < 4; ++m)
          acc[m][g] = __ffma2_rn(S.s[m][p + 1], make_float2(v[g].z, v[g].w), acc[m][g]);
    }
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    float pm[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) pm[m] = __fadd_rn(acc[m][g].x, acc[m][g].y);
    const float k0 = b2 ? pm[2] : pm[0], s0 = b2 ? pm[0] : pm[2];
    const float k1 = b2 ? pm[3] : pm[1], s1 = b2 ? pm[1] : pm[3];
    const float v0 = __fadd_rn(k0, __shfl_xor_sync(0xffffffffu, s0, 4));
    const float v1 = __fadd_rn(k1, __shfl_xor_sync(0xffffffffu, s1, 4));
    const float kk = b1 ? v1 : v0, ss = b1 ? v0 : v1;
    float w = __fadd_rn(kk, __shfl_xor_sync(0xffffffffu, ss, 2));
    w = __fadd_rn(w, __shfl_xor_sync(0xffffffffu, w, 1));
    out[g] = w;
  }
}

// S <- the state after row a of a run that started from S:
//   G_a S + sum_{s<=a} k_s (R[a][s] / |k_s|) u_s^T,
// k rows (raw, fp32, stored by spec_xpos) at kx + s * kstride; us[s * 16 +
// m] holds u_s of the lane's column m (its warp's scratch).
template <int DK, class ST>
__device__ __forceinline__ void spec_advance(SpecS<DK>& S, const RunCoef& C, int a,
                                             const float* kx, int kstride, const float* us,
                                             int r8) {
  using M = SpecMap<DK, ST>;
  const float gm = C.gam[a];
  const float2 g2 = make_float2(gm, gm);
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int p = 0; p < M::P; ++p) S.s[m][p] = __fmul2_rn(g2, S.s[m][p]);
#pragma unroll
  for (int s = 0; s < kSpecK; ++s) {
    if (s <= a) {
      const float c = C.rk[a][s];
      const float4 u4 = *reinterpret_cast<const float4*>(us + s * 16);
      const float uu[4] = {u4.x, u4.y, u4.z, u4.w};
      float2 w2[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float w = __fmul_rn(c, uu[m]);
        w2[m] = make_float2(w, w);
      }
      const float* xr = kx + s * kstride;
#pragma unroll
      for (int i = 0; i < M::NI; ++i)
#pragma unroll
        for (int h = 0; h < M::VEC / 4; ++h) {
          const int p = (i * M::VEC + 4 * h) / 2;
          const float4 v = *reinterpret_cast<const float4*>(xr + M::xoff(r8, i, h));
          const float2 lo = make_float2(v.x, v.y), hi = make_float2(v.z, v.w);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            S.s[m][p] = __ffma2_rn(lo, w2[m], S.s[m][p]);
            S.s[m][p + 1] = __ffma2_rn(hi, w2[m], S.s[m][p + 1]);
          }
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


__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// All of this thread's copy groups but the most recent one have landed.
__device__ __forceinline__ void cp_async_wait_all_but_one() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// The verify runs 3 CTAs per SM (161 registers): measured faster than 2 (the
// item loop is bound by latency, not by a pipe) and than 4 (which spills).
// The slot layout keeps every candidate's state in registers on its way out
// and spilled 280 bytes at 3 per SM; at 2 per SM (240 registers) it does not
// spill and runs 244 us per 64-request step, against 294 us.
template <class IO, class ST, int DK, int MODE>
__global__ void __launch_bounds__(kSpecThreads, MODE == SPEC_SLOTS ? 2 : 3)
spec_kernel(Geom G, Batch B, Params P, SlotGeom SG, const IO* __restrict__ rows_in,
            const IO* __restrict__ conv_w, const IO* __restrict__ a_in,
            const IO* __restrict__ b_in, void* o, int out_f32, void* pages, int32_t* status,
            int splits) {
  using M = SpecMap<DK, ST>;
  constexpr int DV = DK;
  constexpr int CR = kSpecK;                       // first row of the candidates
  constexpr int VE = 16 / (int)sizeof(IO);         // io elements per 16-byte piece
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
  const int r8 = lane & 7, cg = lane >> 3;
  const bool b2 = (r8 & 4) != 0, b1 = (r8 & 2) != 0, b0 = (r8 & 1) != 0;
  const int colw = 16 * warp + 4 * cg;             // the lane's first column in an item
  const int cown = 2 * (b2 ? 1 : 0) + (b1 ? 1 : 0); // the column its dot products end in
  const bool active = colw < BVI;
  const bool reporter = (blockIdx.x == 0 && tid == 0);

  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  if (MODE != SPEC_SLOTS && !q.spec) return;

  const SpecSmem L = spec_smem(DK, DV, Gh, (int)sizeof(IO), (int)sizeof(ST));
  IO* raw = reinterpret_cast<IO*>(smem + L.raw);
  float* abs_ = reinterpret_cast<float*>(smem + L.ab);
  float* kx = reinterpret_cast<float*>(smem + L.kx);
  float* qx = reinterpret_cast<float*>(smem + L.qx);
  RunDots& D = *reinterpret_cast<RunDots*>(smem + L.dots);
  float* gts = reinterpret_cast<float*>(smem + L.gates);
  RunCoef* coef = reinterpret_cast<RunCoef*>(smem + L.coef);
  uint8_t* stage = smem + L.stage;
  const int RW = L.RW, DKP = L.DKP;
  const int g_lo = it0 / nCB, g_hi = (it1 > it0) ? (it1 - 1) / nCB + 1 : g_lo;  // own heads
  const int ng = g_hi - g_lo;
  const int q_off = kh * DK, k_off = G.Hk * DK + kh * DK, v_off = 2 * G.Hk * DK + h0 * DV;
  const int n_c = q.len;
  // channel of row element c (q | k | v of the group's heads) in a packed row
  auto chan = [&](int c) {
    return (c < DK) ? q_off + c : (c < 2 * DK) ? k_off + (c - DK) : v_off + (c - 2 * DK);
  };
  const int row_els = 2 * DK + Gh * DV;
  const int pieces = row_els / VE;

  // ---- 1. this step's candidate rows start copying (they do not depend on
  // the page), then the page is checked ---------------------------------
  if constexpr (MODE != SPEC_FUSED) {
    if (q.len <= G.Kc) {
      for (int idx = tid; idx < n_c * pieces; idx += kSpecThreads) {
        const int t = idx / pieces, c = (idx % pieces) * VE;
        cp_async16(raw + (size_t)(CR + t) * RW + c, rows_in + (size_t)(q.start + t) * G.C + chan(c));
      }
    }
  }
  cp_async_commit();

  char* pg = page_ptr(G, pages, q.page);
  ST* Sbase;
  int n_r = 0, live = 0, parity = 0;
  uint32_t* flagp = nullptr;
  int err = 0;
  if constexpr (MODE == SPEC_SLOTS) {
    const int src = B.n_accepted ? B.n_accepted[q.r] : -1;
    if (src < 0 || src >= G.Kc) err = GDN_DEV_BAD_ACCEPTED;
    else if (q.len > G.Kc) err = GDN_DEV_TOO_MANY_CANDIDATES;
    pg = reinterpret_cast<char*>(pages) + (size_t)q.page * SG.pool_bytes;
    Sbase = reinterpret_cast<ST*>(pg + (size_t)(err ? 0 : src) * SG.slot_bytes + SG.state_off);
  } else {
    Sbase = reinterpret_cast<ST*>(pg + G.state_off);
    flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
    const uint32_t flag = *reinterpret_cast<volatile uint32_t*>(flagp);
    SpecState ss = spec_state(G, B, q, flag);
    if (q.fresh) ss.err = GDN_DEV_BAD_FLAG;
    err = ss.err;
    n_r = (ss.width > 0) ? ss.accepted + 1 : 0;
    live = ss.live;
    parity = ss.parity;
  }
  if (err) {
    if (reporter) report(status, err);
    asm volatile("cp.async.wait_all;" ::: "memory");   // nothing lands after the CTA is gone
    return;
  }
  const int n_all = n_r + n_c;
  IO* rec = reinterpret_cast<IO*>(pg + G.record_off);   // one-page modes only
  // head g's record gates and conv channels are written by the CTA holding
  // its first item; the q/k channels by split 0
  auto owns_head = [&](int g) { return (g * nCB) / per == split; };
  auto item_col0 = [&](int it) -> ST* {
    const int h = h0 + it / nCB, cb = it % nCB;
    return Sbase + ((size_t)h * DV + (size_t)cb * BVI + colw) * DK;
  };

  // ---- 2. replayed rows (k and v from the live record slot), the fused
  // conv, gate inputs; the first item's state starts copying last ---------
  for (int idx = tid; idx < n_r * pieces; idx += kSpecThreads) {
    const int t = idx / pieces, c = (idx % pieces) * VE;
    if (c < DK) continue;                            // a replayed row's q is not used
    cp_async16(raw + (size_t)t * RW + c, rec + ((size_t)live * G.Kc + t) * G.rec_row + chan(c));
  }
  // the replay's run coefficients: those the previous step derived for the
  // same rows as its candidates (the leading block is the same whatever the
  // run's length), kept in the record slot beside them
  if (n_r > 0) {
    const float* rc = reinterpret_cast<const float*>(pg + G.rcoef_off) + (size_t)live * G.Hv * kRunCoefFloats;
    for (int idx = tid; idx < ng * 36; idx += kSpecThreads) {
      const int g = g_lo + idx / 36, k = idx % 36;
      const float* src = rc + (size_t)(h0 + g) * kRunCoefFloats;
      float* dst = reinterpret_cast<float*>(&coef[g * 2 + 0]);
      // pieces 0-1: gk, 2-3: gam, 4-19: rk, 20-35: m (4 floats each)
      const int so = 4 * k;
      const int dofs = (k < 2) ? so : (k < 4) ? 16 + (so - 8) : (k < 20) ? 160 + (so - 16) : 224 + (so - 80);
      cp_async16(dst + dofs, src + so);
    }
  }
  cp_async_commit();
  if (active && it0 < it1) spec_stage_async<DK, ST>(stage, item_col0(it0), r8, tid);
  else cp_async_commit();   // keep "all but the newest group" meaning the rows

  if constexpr (MODE == SPEC_FUSED) {
    // the conv of the group's channels for this step's candidates, exactly
    // as gdn_conv computes it for a spec request: history = window columns
    // n_r .. n_r+W-2 (the record's accepted rows rolled out), taps oldest
    // first, own SiLU, rounded to the io dtype. Every load of a channel
    // vector is issued before its arithmetic.
    const int nvec = row_els / 4;
    IO* win = reinterpret_cast<IO*>(pg + G.window_off);
    IO* rec_out = rec + (size_t)(1 - live) * G.Kc * G.rec_row;
    for (int vi = tid; vi < nvec; vi += kSpecThreads) {
      const int c4 = 4 * vi;
      const int gg = (c4 < 2 * DK) ? -1 : (c4 - 2 * DK) / DV;
      if (gg >= 0 && (gg < g_lo || gg >= g_hi)) continue;   // another split's head
      const bool owner = (gg < 0) ? (split == 0) : owns_head(gg);
      const int ch = chan(c4);
      float wt[4][4], hcol[3][4], h0c[3][4], xr[kSpecK][4];
      {
        float tmp[16];
        load_f<IO, 16>(conv_w + (size_t)ch * 4, tmp);
#pragma unroll
        for (int v = 0; v < 4; ++v)
#pragma unroll
          for (int j = 0; j < 4; ++j) wt[j][v] = tmp[v * 4 + j];
      }
#pragma unroll
      for (int j = 0; j < 3; ++j) load_f<IO, 4>(win + (size_t)(n_r + j) * G.C + ch, hcol[j]);
#pragma unroll
      for (int t = 0; t < kSpecK; ++t)
        if (t < n_c) load_f<IO, 4>(rows_in + (size_t)(q.start + t) * G.C + ch, xr[t]);
#pragma unroll
      for (int j = 0; j < 3; ++j)
#pragma unroll
        for (int v = 0; v < 4; ++v) h0c[j][v] = hcol[j][v];
#pragma unroll
      for (int t = 0; t < kSpecK; ++t) {
        if (t < n_c) {
          float yv[4];
#pragma unroll
          for (int v = 0; v < 4; v += 2) {
            float2 acc = P.conv_bias ? make_float2(P.conv_bias[ch + v], P.conv_bias[ch + v + 1])
                                     : make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < 3; ++j)
              acc = __ffma2_rn(make_float2(wt[j][v], wt[j][v + 1]),
                               make_float2(hcol[j][v], hcol[j][v + 1]), acc);
            acc = __ffma2_rn(make_float2(wt[3][v], wt[3][v + 1]),
                             make_float2(xr[t][v], xr[t][v + 1]), acc);
            const float2 y2 = own_silu2(acc);
            yv[v] = y2.x;
            yv[v + 1] = y2.y;
          }
          store_f<IO, 4>(raw + (size_t)(CR + t) * RW + c4, yv);
          if (owner) {
            store_f<IO, 4>(rec_out + (size_t)t * G.rec_row + ch, yv);
            store_f<IO, 4>(win + (size_t)(3 + t) * G.C + ch, xr[t]);
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            hcol[0][v] = hcol[1][v];
            hcol[1][v] = hcol[2][v];
            hcol[2][v] = xr[t][v];
          }
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
  for (int idx = tid; idx < n_all * ng; idx += kSpecThreads) {
    const int t = idx / ng, g = g_lo + idx % ng, h = h0 + g;
    const int row = (t < n_r) ? t : CR + (t - n_r);
    float av, bv;
    if (t < n_r) {
      const IO* rr = rec + ((size_t)live * G.Kc + t) * G.rec_row;
      av = to_f(rr[G.C + h]);
      bv = to_f(rr[G.C + G.Hv + h]);
    } else {
      const size_t rn = (size_t)q.start + (t - n_r);
      av = to_f(a_in[rn * G.Hv + h]);
      bv = to_f(b_in[rn * G.Hv + h]);
      if (MODE != SPEC_SLOTS && owns_head(g)) {
        // the candidates' gates go next to their conv'd rows in the other slot
        IO* rr = rec + ((size_t)(1 - live) * G.Kc + (t - n_r)) * G.rec_row;
        rr[G.C + h] = a_in[rn * G.Hv + h];
        rr[G.C + G.Hv + h] = b_in[rn * G.Hv + h];
      }
    }
    abs_[row * 2 * Gh + g] = av;
    abs_[row * 2 * Gh + Gh + g] = bv;
  }
  cp_async_wait_all_but_one();   // the rows (not the state) have landed
  __syncthreads();

  // ---- 3. fp32 copies of the k rows (all) and q rows (candidates), each
  // in the order the lanes read it (spec_xpos); the Gram products below sum
  // over that order too ---------------------------------------------------
  {
    constexpr int Q4 = DK / 4;
    const int nk = n_all * Q4;
    for (int idx = tid; idx < nk + n_c * Q4; idx += kSpecThreads) {
      float f[4];
      if (idx < nk) {
        const int r = idx / Q4, d = (idx % Q4) * 4;
        const int row = (r < n_r) ? r : CR + (r - n_r);
        load_f<IO, 4>(raw + (size_t)row * RW + DK + d, f);
        *reinterpret_cast<float4*>(kx + row * DKP + spec_xpos<DK, ST>(d)) =
            make_float4(f[0], f[1], f[2], f[3]);
      } else {
        const int t = (idx - nk) / Q4, d = ((idx - nk) % Q4) * 4;
        load_f<IO, 4>(raw + (size_t)(CR + t) * RW + d, f);
        *reinterpret_cast<float4*>(qx + t * DKP + spec_xpos<DK, ST>(d)) =
            make_float4(f[0], f[1], f[2], f[3]);
      }
    }
  }
  __syncthreads();

  // ---- 4. Gram products and norms (one per thread), gates ---------------
  {
    const int A = 0, Bc = n_c * (n_c + 1) / 2;   // (the replay's come from the record)
    int k = tid;
    if (k < A) {
      int s, t;
      spec_tri(k, s, t);
      D.kkr[t][s] = spec_rowdot<DK>(kx + s * DKP, kx + t * DKP);
    } else if ((k -= A) < Bc) {
      int s, t;
      spec_tri(k, s, t);
      D.kkc[t][s] = spec_rowdot<DK>(kx + (CR + s) * DKP, kx + (CR + t) * DKP);
    } else if ((k -= Bc) < Bc) {
      int s, t;
      spec_tri(k, s, t);
      D.kqc[t][s] = spec_rowdot<DK>(kx + (CR + s) * DKP, qx + t * DKP);
    } else if ((k -= Bc) < n_c) {
      D.qqc[k] = spec_rowdot<DK>(qx + k * DKP, qx + k * DKP);
    }
    // gates of own heads for the candidates: thread -> (head, row); and the
    // candidate run's coefficient blocks start from zero (the entries past
    // the run stay zero wherever they are stored)
    for (int idx = tid; idx < ng * n_c; idx += kSpecThreads) {
      const int g = g_lo + idx / n_c, t = idx % n_c;
      const int row = CR + t;
      float alpha, beta;
      gates(P, h0 + g, abs_[row * 2 * Gh + g], abs_[row * 2 * Gh + Gh + g], alpha, beta);
      gts[((g * 2 + 1) * 2 + 0) * kSpecK + t] = alpha;
      gts[((g * 2 + 1) * 2 + 1) * kSpecK + t] = beta;
    }
    for (int idx = tid; idx < ng * (int)(sizeof(RunCoef) / 16); idx += kSpecThreads) {
      const int g = g_lo + idx / (int)(sizeof(RunCoef) / 16), k = idx % (int)(sizeof(RunCoef) / 16);
      reinterpret_cast<float4*>(&coef[g * 2 + 1])[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __syncthreads();

  // ---- 5. run coefficients per own head and run --------------------------
  {
    // (a) thread -> (head, run, column s = -1..7): decay products R[.][s], G,
    // and the columns of L, B and R/|k|. Loops run to kSpecK with guards, so
    // every array index is a compile-time constant.
    for (int idx = tid; idx < ng * (kSpecK + 1); idx += kSpecThreads) {
      const int g = g_lo + idx / (kSpecK + 1);
      const int run = 1;
      const int s = idx % (kSpecK + 1) - 1;
      const int n = run ? n_c : n_r;
      if (s >= n) continue;
      RunCoef& C = coef[g * 2 + run];
      const float* al = gts + ((g * 2 + run) * 2 + 0) * kSpecK;
      const float* be = gts + ((g * 2 + run) * 2 + 1) * kSpecK;
      float ik[kSpecK], iq[kSpecK];
#pragma unroll
      for (int t = 0; t < kSpecK; ++t) {
        ik[t] = (t < n) ? rsqrtf(__fadd_rn(run ? D.kkc[t][t] : D.kkr[t][t], P.eps)) : 0.0f;
        iq[t] = (run && t < n) ? rsqrtf(__fadd_rn(D.qqc[t], P.eps)) : 0.0f;
      }
      if (s < 0) {
        float r = 1.0f;
#pragma unroll
        for (int t = 0; t < kSpecK; ++t) {
          if (t < n) {
            r = __fmul_rn(r, al[t]);
            C.gam[t] = r;
            C.gk[t] = __fmul_rn(r, ik[t]);
            C.gq[t] = __fmul_rn(r, iq[t]);
            C.beta[t] = be[t];
          }
        }
      } else {
        float iks = 0.0f;
#pragma unroll
        for (int t = 0; t < kSpecK; ++t) iks = (t == s) ? ik[t] : iks;
        float r = 1.0f;
#pragma unroll
        for (int t = 0; t < kSpecK; ++t) {
          if (t >= s && t < n) {
            if (t > s) r = __fmul_rn(r, al[t]);
            C.rk[t][s] = __fmul_rn(r, iks);
            if (t > s) {
              const float kk = run ? D.kkc[t][s] : D.kkr[t][s];
              C.l[t][s] = -__fmul_rn(be[t], __fmul_rn(r, __fmul_rn(__fmul_rn(kk, iks), ik[t])));
            }
            if (run) C.bco[t][s] = __fmul_rn(r, __fmul_rn(__fmul_rn(D.kqc[t][s], iks), iq[t]));
          }
        }
      }
    }
    __syncthreads();
    // (b) thread -> (head, run, column s): column s of (I - L)^-1 by forward
    // substitution (rows in increasing order, terms r = s .. t-1), times beta_s
    for (int idx = tid; idx < ng * kSpecK; idx += kSpecThreads) {
      const int g = g_lo + idx / kSpecK;
      const int run = 1;
      const int s = idx % kSpecK;
      const int n = run ? n_c : n_r;
      if (s >= n) continue;
      RunCoef& C = coef[g * 2 + run];
      float Lr[kSpecK][kSpecK];
#pragma unroll
      for (int t = 0; t < kSpecK; ++t)
#pragma unroll
        for (int r = 0; r < t; ++r) Lr[t][r] = (t < n && r >= s) ? C.l[t][r] : 0.0f;
      float col[kSpecK];   // col[t] = (I - L)^-1 [t][s]
      const float bs = C.beta[s];
#pragma unroll
      for (int t = 0; t < kSpecK; ++t) {
        if (t < s) {
          col[t] = 0.0f;
        } else if (t == s) {
          col[t] = 1.0f;
          C.m[t][s] = bs;
        } else if (t < n) {
          float acc = 0.0f;
          bool first = true;
#pragma unroll
          for (int r = 0; r < t; ++r) {
            if (r >= s) {
              acc = first ? __fmul_rn(Lr[t][r], col[r]) : __fmaf_rn(Lr[t][r], col[r], acc);
              first = false;
            }
          }
          col[t] = acc;
          C.m[t][s] = __fmul_rn(acc, bs);
        }
      }
    }
    __syncthreads();
    // (c) thread -> (head, candidate row t, column s): N[t][s] = sum_r B[t][r] M[r][s]
    for (int idx = tid; idx < ng * kSpecK * kSpecK; idx += kSpecThreads) {
      const int g = g_lo + idx / (kSpecK * kSpecK);
      const int t = (idx / kSpecK) % kSpecK, s = idx % kSpecK;
      if (t >= n_c || s > t) continue;
      RunCoef& C = coef[g * 2 + 1];
      float acc = __fmul_rn(C.bco[t][s], C.m[s][s]);
      for (int r = s + 1; r <= t; ++r) acc = __fmaf_rn(C.bco[t][r], C.m[r][s], acc);
      C.nq[t][s] = acc;
    }
  }
  __syncthreads();
  if constexpr (MODE != SPEC_SLOTS) {
    // the candidates' run coefficients go beside their rows in the other
    // slot, for the next step's replay
    if (n_c > 0) {
      float* rc = reinterpret_cast<float*>(pg + G.rcoef_off) + (size_t)(1 - live) * G.Hv * kRunCoefFloats;
      for (int idx = tid; idx < ng * 36; idx += kSpecThreads) {
        const int g = g_lo + idx / 36, k = idx % 36;
        if (!owns_head(g)) continue;
        const float* src = reinterpret_cast<const float*>(&coef[g * 2 + 1]);
        const int so = 4 * k;
        const int sofs = (k < 2) ? so : (k < 4) ? 16 + (so - 8) : (k < 20) ? 160 + (so - 16) : 224 + (so - 80);
        *reinterpret_cast<float4*>(rc + (size_t)(h0 + g) * kRunCoefFloats + so) =
            *reinterpret_cast<const float4*>(src + sofs);
      }
    }
  }

  // ---- 6. items: no block-wide barrier from here on ---------------------
  // An item's state comes from the stage (copied by this thread alone). The
  // one-page modes request the next item's copy as soon as the first dot
  // products have consumed the current one; the slot layout keeps the stage
  // for the whole item (it rebuilds each candidate's state from it).
  if (active && (n_all > 0 || MODE == SPEC_SLOTS)) {
    const IO* vraw = raw + 2 * DK;
    for (int it = it0; it < it1; ++it) {
      const int g = it / nCB, cb = it % nCB, h = h0 + g;
      ST* col0 = item_col0(it);
      if (MODE == SPEC_SLOTS && it > it0) spec_stage_async<DK, ST>(stage, col0, r8, tid);
      spec_stage_wait();
      SpecS<DK> S;
      spec_unstage<DK, ST>(S, stage, tid);
      bool ahead = (MODE == SPEC_SLOTS) || (it + 1 >= it1);
      auto prefetch = [&]() {
        if (!ahead) {
          spec_stage_async<DK, ST>(stage, item_col0(it + 1), r8, tid);
          ahead = true;
        }
      };
      // per-warp scratch: dsc[r][j] the dot products of row r (k rows 0..7,
      // candidate q rows 8..15) with the warp's column j; usc[t][j] = u
      float* dsc = reinterpret_cast<float*>(smem + L.scr) + warp * kSpecScr;
      float* usc = dsc + 2 * kSpecK * 16;
      const int jw = 4 * cg + cown;                 // this lane's column in the warp
      const bool writer = (r8 & 1) == 0;            // one of the column's two lanes
      // the scalar phase maps lane -> (column jc of the warp, row half th)
      const int jc = lane & 15, th = lane >> 4;
      const int vcol = g * DV + cb * BVI + 16 * warp + jc;   // v column of jc

      if (n_r > 0) {
        const RunCoef& C = coef[g * 2 + 0];
#pragma unroll
        for (int t = 0; t < kSpecK; t += 2) {
          if (t < n_r) {
            const float* xr[2] = {kx + t * DKP, kx + (t + 1) * DKP};
            float out[2];
            spec_dots<DK, ST, 2>(S, xr, r8, b2, b1, out);
            if (writer) {
              dsc[t * 16 + jw] = out[0];
              dsc[(t + 1) * 16 + jw] = out[1];
            }
            if (t == 0) prefetch();
          }
        }
        __syncwarp();
        // c_t = v_t - G_t dk_t for column jc; u_t = sum_s M[t][s] c_s for
        // the rows t of half th
        {
          float c[kSpecK];
#pragma unroll
          for (int t = 0; t < kSpecK; ++t)
            c[t] = (t < n_r) ? __fmaf_rn(-C.gk[t], dsc[t * 16 + jc],
                                         to_f(vraw[(size_t)t * RW + vcol])) : 0.0f;
#pragma unroll
          for (int tt = 0; tt < kSpecK / 2; ++tt) {
            const int t = 2 * tt + th;
            if (t < n_r) {
              float acc = __fmul_rn(C.m[t][0], c[0]);
#pragma unroll
              for (int s = 1; s <= 2 * tt + 1; ++s)
                if (s <= t) acc = __fmaf_rn(C.m[t][s], c[s], acc);
              usc[t * 16 + jc] = acc;
            }
          }
        }
        __syncwarp();
        spec_advance<DK, ST>(S, C, n_r - 1, kx, DKP, usc + 4 * cg, r8);
        spec_store<DK, ST>(col0, S, r8);
        // continue from exactly what was stored (a bf16 page rounds here)
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int p = 0; p < M::P; ++p)
            S.s[m][p] = make_float2(through<ST>(S.s[m][p].x), through<ST>(S.s[m][p].y));
        __syncwarp();   // usc is read again only after this
      }

      if (n_c > 0) {
        const RunCoef& C = coef[g * 2 + 1];
        const float* kc = kx + CR * DKP;
#pragma unroll
        for (int t = 0; t < kSpecK; t += 2) {
          if (t < n_c) {
            const float* xr[4] = {kc + t * DKP, kc + (t + 1) * DKP, qx + t * DKP,
                                  qx + (t + 1) * DKP};
            float out[4];
            spec_dots<DK, ST, 4>(S, xr, r8, b2, b1, out);
            if (writer) {
              dsc[t * 16 + jw] = out[0];
              dsc[(t + 1) * 16 + jw] = out[1];
              dsc[(kSpecK + t) * 16 + jw] = out[2];
              dsc[(kSpecK + t + 1) * 16 + jw] = out[3];
            }
            if (t == 0) prefetch();
          }
        }
        __syncwarp();
        float c[kSpecK];
#pragma unroll
        for (int t = 0; t < kSpecK; ++t)
          c[t] = (t < n_c) ? __fmaf_rn(-C.gk[t], dsc[t * 16 + jc],
                                       to_f(vraw[(size_t)(CR + t) * RW + vcol])) : 0.0f;
        // outputs o_t = scale (G_t S^T q^_t + sum_s N[t][s] c_s), column jc,
        // the rows of half th
        const size_t ocol = (size_t)h * DV + (size_t)cb * BVI + 16 * warp + jc;
#pragma unroll
        for (int tt = 0; tt < kSpecK / 2; ++tt) {
          const int t = 2 * tt + th;
          if (t < n_c) {
            float acc = __fmul_rn(C.gq[t], dsc[(kSpecK + t) * 16 + jc]);
#pragma unroll
            for (int s = 0; s <= 2 * tt + 1; ++s)
              if (s <= t) acc = __fmaf_rn(C.nq[t][s], c[s], acc);
            store_out(o, out_f32, ((size_t)q.start + t) * G.Hv * DV + ocol,
                      __fmul_rn(P.scale, acc));
          }
        }
        if constexpr (MODE == SPEC_SLOTS) {
          // u of the candidates, then the state after every candidate goes
          // to its slot, each rebuilt from the staged starting state
#pragma unroll
          for (int tt = 0; tt < kSpecK / 2; ++tt) {
            const int t = 2 * tt + th;
            if (t < n_c) {
              float acc = __fmul_rn(C.m[t][0], c[0]);
#pragma unroll
              for (int s = 1; s <= 2 * tt + 1; ++s)
                if (s <= t) acc = __fmaf_rn(C.m[t][s], c[s], acc);
              usc[t * 16 + jc] = acc;
            }
          }
          __syncwarp();
          const size_t off = (size_t)(col0 - Sbase);
          for (int t = 0; t < n_c; ++t) {
            SpecS<DK> T;
            spec_unstage<DK, ST>(T, stage, tid);
            spec_advance<DK, ST>(T, C, t, kc, DKP, usc + 4 * cg, r8);
            ST* dst = reinterpret_cast<ST*>(pg + (size_t)t * SG.slot_bytes + SG.state_off) + off;
            spec_store<DK, ST>(dst, T, r8);
          }
        }
        __syncwarp();   // dsc / usc are written again only after this
      }
      prefetch();   // (a run with no rows never consumed the stage)
    }
  }
  spec_stage_wait();   // no copy outlives the CTA's shared memory

  // ---- 7. the last CTA of the request publishes the new flag word -------
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
