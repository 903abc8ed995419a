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
// M and N depend only on the rows (not on S or the value column), so they
// are formed once per value head; every column then needs only independent
// short dot products with its c. M's leading block is the inverse of L's
// leading block, so a run of the first a + 1 rows sees exactly the
// coefficients and the u the longer run had.
//
// The one-page step so keeps, in the record slot beside the candidates'
// rows, their coefficients (G/|k|, G/|q|, G, R/|k|, M, N) and their u per
// value column (fp32). The next step's replay of the first a + 1 of them is
// then only the rank-(a+1) update S_a = G_a S + sum_s (R[a][s]/|k_s|) k_s u_s^T
// of the stored state: the u it needs are the ones the candidate run formed
// from that same stored state. The slot layout runs the candidates and
// stores every S_t. All three entry points compute each quantity with the
// same code and in the same order from the same inputs, so the one-page
// checkpoint equals the slot that was kept for it, bit for bit, and so do
// all outputs.
//
// Kernels.
// - spec_coef_kernel, one CTA per (request, q/k head kh): stages the
//   candidates' q and k rows of kh, forms their Gram products and gates
//   once, derives the run coefficients of every value head of the group,
//   and stores them in the record slot the candidates go to.
// - spec_item_kernel, one CTA per (request, value head) with the head's
//   items of 64 value columns (two at Dv = 128): copies the first item's
//   state while it reads the flag word and the replay's inputs, then (after
//   the coefficient kernel, which it follows as a programmatic dependent
//   launch) the candidates' rows and coefficients; per item replays and
//   stores the checkpoint, runs the candidates and stores their outputs and
//   u, with the next item's state copied meanwhile. The last CTA of a
//   request publishes the new flag word.
// - spec_step_kernel (gdn_spec_step), one CTA per (request, q/k head kh):
//   the conv of the group's q, k and v channels for this step's candidates
//   (rows into the record, the window rolled), the coefficient kernel's work
//   for the group, then the item kernel's work for every item of the group,
//   in one launch.
// - spec_slots_kernel, one CTA per (request, q/k head, split): the slot
//   layout. It forms the coefficients with the coefficient kernel's code,
//   then per item runs the candidates from the source slot and rebuilds and
//   stores the state after each one.
//
// Inside an item: 4 warps x 16 columns; inside a warp, 4 groups of 4
// columns x 8 lanes, a lane holding 4 columns x Dk/8 entries of S in
// registers (chunks of 16 bytes at Dk index VEC (8 i + r8)). Each 16-byte
// shared load of a q/k row by an 8-lane quarter of the warp reads 128
// distinct bytes and feeds 4 columns. The per-column scalar work (c, u = M c,
// the outputs) goes through a small per-warp scratch: the dot products land
// there, then each lane takes one column and half of the rows, which keeps
// the per-column arrays out of registers. A state item is copied into shared
// memory by the thread that will read it (cp.async).
#pragma once

#include "common.cuh"

namespace gdn {

enum SpecMode { SPEC_VERIFY = 0, SPEC_FUSED = 1, SPEC_SLOTS = 2 };
// Shared memory layouts of spec_smem (see there).
enum SpecLayout { LAYOUT_ITEMS = 0, LAYOUT_COEF = 1, LAYOUT_SLOTS = 2 };

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

// The record keeps, per value head, gk gq gam (24 floats) and rk m nq (192
// floats): kRunCoefFloats values, in 16-byte pieces. Piece k of the record
// block sits at float spec_coef_piece(k) of a RunCoef: gk 0-1, gq 2-3,
// gam 4-5, rk 6-21, m 22-37, nq 38-53.
static_assert(offsetof(RunCoef, gk) == 0 && offsetof(RunCoef, gam) == 64 &&
                  offsetof(RunCoef, beta) == 96 && offsetof(RunCoef, rk) == 640 &&
                  offsetof(RunCoef, nq) == 1152 && sizeof(RunCoef) == 1408,
              "record coefficient copy offsets");
static_assert(kRunCoefFloats == 24 + 192, "record coefficient block");
constexpr int kCoefPieces = (int)kRunCoefFloats / 4;
__host__ __device__ constexpr int spec_coef_piece(int k) { return k < 6 ? 4 * k : 160 + 4 * (k - 6); }

// Raw dot products of the candidate rows (k_s.k_t and k_s.q_t with s <= t,
// q_t.q_t).
struct RunDots {
  float kkc[kSpecK][kSpecK];   // [t][s]
  float kqc[kSpecK][kSpecK];   // k_s.q_t at [t][s]
  float qqc[kSpecK];
  float ik[kSpecK];            // 1 / |k_t| = rsqrt(k_t.k_t + eps)
  float iq[kSpecK];            // 1 / |q_t|
};

__host__ __device__ inline uint32_t spec_al16(uint32_t x) { return (x + 15u) & ~15u; }

// Dynamic shared memory of the three kernels (byte offsets, 16-byte aligned;
// a region a kernel does not use has size 0).
struct SpecSmem {
  uint32_t raw;     // coef / slots: [Kc][RW] io dtype, the candidates' rows
  uint32_t ab;      // coef / slots: [Kc][2 Gh] float: a then b per head
  uint32_t hc;      // coef / slots: [Gh][2] float: A_log, dt_bias per head
  uint32_t kx;      // [NK][DKP] float: k rows (items: replayed 0..7, candidates 8..15)
  uint32_t qx;      // [Kc][DKP] float: candidate q rows
  uint32_t dots;    // coef / slots: RunDots
  uint32_t gates;   // coef / slots: [Gh][2][Kc] float: alpha, beta
  uint32_t coef;    // RunCoef: coef / slots [Gh]; items [3] (record slots 0 and 1, candidates)
  uint32_t rawk;    // items: [3 Kc][DK] io dtype (record slots 0 and 1, candidates)
  uint32_t rawq;    // items: [Kc][DK] io dtype
  uint32_t rawv;    // items: [Kc][VW] io dtype, the candidates' v of the CTA's columns
  uint32_t ur;      // items: [Kc][VW] float, the record's u of the CTA's columns
  uint32_t stage;   // items / slots: [NC][threads] 16-byte chunks of one item's state
  uint32_t scr;     // items / slots: per warp [2 Kc][16] dot products, [Kc][16] u
  uint32_t total;
  int RW, DKP, VW;
};

// kind: LAYOUT_ITEMS = the item kernel (VW value columns per CTA),
// LAYOUT_COEF = the coefficient kernel, LAYOUT_SLOTS = the slot kernel.
__host__ __device__ inline SpecSmem spec_smem(int kind, int DK, int DV, int Gh, int io_bytes,
                                               int st_bytes, int VW) {
  SpecSmem L;
  L.DKP = DK + 4;
  L.RW = (kind == LAYOUT_SLOTS) ? (2 * DK + Gh * DV + 7) / 8 * 8 : 2 * DK;
  L.VW = VW;
  const bool items = (kind == LAYOUT_ITEMS), coef = (kind == LAYOUT_COEF);
  const uint32_t K = kSpecK;
  uint32_t off = 0;
  auto take = [&](uint32_t& at, uint32_t bytes) {
    at = off;
    off = spec_al16(off + bytes);
  };
  take(L.raw, items ? 0u : K * L.RW * io_bytes);
  take(L.ab, items ? 0u : K * 2 * Gh * 4);
  take(L.hc, items ? 0u : Gh * 2 * 4);
  take(L.kx, (items ? 2 * K : K) * L.DKP * 4);
  take(L.qx, K * L.DKP * 4);
  take(L.dots, items ? 0u : (uint32_t)sizeof(RunDots));
  take(L.gates, items ? 0u : Gh * 2 * K * 4);
  take(L.coef, (items ? 3u : (uint32_t)Gh) * (uint32_t)sizeof(RunCoef));
  take(L.rawk, items ? 3 * K * DK * io_bytes : 0u);
  take(L.rawq, items ? K * DK * io_bytes : 0u);
  take(L.rawv, items ? K * VW * io_bytes : 0u);
  take(L.ur, items ? K * VW * 4 : 0u);
  take(L.stage, coef ? 0u : (uint32_t)(DK / 2 * st_bytes * kSpecThreads));
  take(L.scr, coef ? 0u : (uint32_t)((kSpecThreads / 32) * kSpecScr * 4));
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
// k rows (raw, fp32, stored by spec_xpos) at kx + s * kstride; us[s * ustride
// + m] holds u_s of the lane's column m; C is any block with gam and rk laid
// out as in RunCoef (a RunCoef, or the replay's RepCoef).
template <int DK, class ST, class CT>
__device__ __forceinline__ void spec_advance(SpecS<DK>& S, const CT& C, int a,
                                             const float* kx, int kstride, const float* us,
                                             int ustride, int r8) {
  using M = SpecMap<DK, ST>;
  const float gm = C.gam[a];
  const float2 g2 = make_float2(gm, gm);
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int p = 0; p < M::P; ++p) S.s[m][p] = __fmul2_rn(g2, S.s[m][p]);
  // a loop over the run's rows only (a fully unrolled loop to kSpecK would
  // issue the rows past a as predicated-off instructions)
#pragma unroll 1
  for (int s = 0; s <= a; ++s) {
    const float c = C.rk[a][s];
    const float4 u4 = *reinterpret_cast<const float4*>(us + s * ustride);
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

// Plain dot product of two fp32 rows in shared memory, in a fixed order:
// four running sums (entries d = 0, 1, 2, 3 mod 4, as two packed pairs), then
// (x + y) + (z + w).
template <int DK>
__device__ __forceinline__ float spec_rowdot(const float* a, const float* b) {
  float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
#pragma unroll 8
  for (int d = 0; d < DK; d += 4) {
    const float4 x = *reinterpret_cast<const float4*>(a + d);
    const float4 y = *reinterpret_cast<const float4*>(b + d);
    lo = __ffma2_rn(make_float2(x.x, x.y), make_float2(y.x, y.y), lo);
    hi = __ffma2_rn(make_float2(x.z, x.w), make_float2(y.z, y.w), hi);
  }
  return __fadd_rn(__fadd_rn(lo.x, lo.y), __fadd_rn(hi.x, hi.y));
}

// fp32 copies of n rows (io dtype, DK apart from src, q/k entries at column
// 0) in the order the lanes read them, dst rows DKP apart. Block-wide loop
// over NT threads.
template <int DK, class ST, class IO, int NT>
__device__ __forceinline__ void spec_rows_f32(float* dst, int DKP, const IO* src, int sstride,
                                              int n) {
  constexpr int Q4 = DK / 4;
  for (int idx = threadIdx.x; idx < n * Q4; idx += NT) {
    const int t = idx / Q4, d = (idx % Q4) * 4;
    float f[4];
    load_f<IO, 4>(src + (size_t)t * sstride + d, f);
    *reinterpret_cast<float4*>(dst + t * DKP + spec_xpos<DK, ST>(d)) =
        make_float4(f[0], f[1], f[2], f[3]);
  }
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
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// All of this thread's copy groups but the most recent one have landed.
__device__ __forceinline__ void cp_async_wait_all_but_one() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// The candidates' Gram products, gates and run coefficients for the value
// heads g_lo .. g_lo+ng-1 of a group. Block-wide over NT threads: every
// thread calls it, with the rows, gate inputs and head constants in shared
// memory and visible to all.
//   kx, qx [n_c][DKP] float: the k and q rows, stored by spec_xpos (the Gram
//          products sum in that order)
//   abs_  [n_c][2 Gh] float: a of head g at g, b at Gh + g
//   hc    [Gh][2] float: A_log, dt_bias of head g
//   coef  [Gh] RunCoef: coef[g] receives head g's candidate coefficients
// Loops over rows run to kSpecK with guards, so every array index is a
// compile-time constant.
template <int DK, int NT>
__device__ void spec_candidate_coefs(const Params& P, int Gh, int g_lo, int ng, int n_c,
                                     const float* kx, const float* qx, int DKP,
                                     const float* abs_, const float* hc, RunDots& D, float* gts,
                                     RunCoef* coef) {
  const int tid = threadIdx.x;
  // Gram products and norms; gates of the heads, thread -> (head, row); the
  // coefficient blocks start from zero (the entries past the run stay zero
  // wherever they are stored)
  {
    const int Bc = n_c * (n_c + 1) / 2;
    for (int k0 = tid; k0 < 2 * Bc + n_c; k0 += NT) {
      int k = k0;
      if (k < Bc) {
        int s, t;
        spec_tri(k, s, t);
        const float kk = spec_rowdot<DK>(kx + s * DKP, kx + t * DKP);
        D.kkc[t][s] = kk;
        if (s == t) D.ik[t] = rsqrtf(__fadd_rn(kk, P.eps));
      } else if ((k -= Bc) < Bc) {
        int s, t;
        spec_tri(k, s, t);
        D.kqc[t][s] = spec_rowdot<DK>(kx + s * DKP, qx + t * DKP);
      } else {
        k -= Bc;
        const float qq = spec_rowdot<DK>(qx + k * DKP, qx + k * DKP);
        D.qqc[k] = qq;
        D.iq[k] = rsqrtf(__fadd_rn(qq, P.eps));
      }
    }
    for (int idx = tid; idx < ng * n_c; idx += NT) {
      const int g = g_lo + idx / n_c, t = idx % n_c;
      float alpha, beta;
      gates_v(P.gate_mode, hc[2 * g], hc[2 * g + 1], abs_[t * 2 * Gh + g],
              abs_[t * 2 * Gh + Gh + g], alpha, beta);
      gts[(g * 2 + 0) * kSpecK + t] = alpha;
      gts[(g * 2 + 1) * kSpecK + t] = beta;
    }
    constexpr int C4 = (int)(sizeof(RunCoef) / 16);
    for (int idx = tid; idx < ng * C4; idx += NT) {
      const int g = g_lo + idx / C4, k4 = idx % C4;
      reinterpret_cast<float4*>(&coef[g])[k4] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __syncthreads();
  // (a) thread -> (head, task): task t < kSpecK forms G_t (the product
  // alpha_0 ... alpha_t, left to right), G_t/|k_t| and G_t/|q_t|; the other
  // tasks take one pair s <= t each: the decay product R[t][s] = alpha_{s+1}
  // ... alpha_t (left to right) and the entries of L, B and R/|k| at [t][s]
  constexpr int kTasks = kSpecK + kSpecK * (kSpecK + 1) / 2;
  for (int idx = tid; idx < ng * kTasks; idx += NT) {
    const int g = g_lo + idx / kTasks;
    const int task = idx % kTasks;
    RunCoef& C = coef[g];
    const float* al = gts + (g * 2 + 0) * kSpecK;
    const float* be = gts + (g * 2 + 1) * kSpecK;
    if (task < kSpecK) {
      const int t = task;
      if (t >= n_c) continue;
      float r = 1.0f;
      for (int q = 0; q <= t; ++q) r = __fmul_rn(r, al[q]);
      C.gam[t] = r;
      C.gk[t] = __fmul_rn(r, D.ik[t]);
      C.gq[t] = __fmul_rn(r, D.iq[t]);
      C.beta[t] = be[t];
    } else {
      int s, t;
      spec_tri(task - kSpecK, s, t);
      if (t >= n_c) continue;
      float r = 1.0f;
      for (int q = s + 1; q <= t; ++q) r = __fmul_rn(r, al[q]);
      const float iks = D.ik[s];
      C.rk[t][s] = __fmul_rn(r, iks);
      if (t > s)
        C.l[t][s] = -__fmul_rn(be[t], __fmul_rn(r, __fmul_rn(__fmul_rn(D.kkc[t][s], iks), D.ik[t])));
      C.bco[t][s] = __fmul_rn(r, __fmul_rn(__fmul_rn(D.kqc[t][s], iks), D.iq[t]));
    }
  }
  __syncthreads();
  // (b) thread -> (head, column s): column s of (I - L)^-1 by forward
  // substitution (rows in increasing order, terms r = s .. t-1), times beta_s
  for (int idx = tid; idx < ng * kSpecK; idx += NT) {
    const int g = g_lo + idx / kSpecK;
    const int s = idx % kSpecK;
    const int n = n_c;
    if (s >= n) continue;
    RunCoef& C = coef[g];
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
  // (c) thread -> (head, row t, column s): N[t][s] = sum_r B[t][r] M[r][s]
  for (int idx = tid; idx < ng * kSpecK * kSpecK; idx += NT) {
    const int g = g_lo + idx / (kSpecK * kSpecK);
    const int t = (idx / kSpecK) % kSpecK, s = idx % kSpecK;
    if (t >= n_c || s > t) continue;
    RunCoef& C = coef[g];
    float acc = __fmul_rn(C.bco[t][s], C.m[s][s]);
    for (int r = s + 1; r <= t; ++r) acc = __fmaf_rn(C.bco[t][r], C.m[r][s], acc);
    C.nq[t][s] = acc;
  }
  __syncthreads();
}

// The candidates' dot products with the item's state (k rows at kc, q rows
// at qx, DKP apart) into the warp's scratch (dsc[t][j]: k rows at t, q rows
// at kSpecK + t); after the first pair, after_first() runs (S is then in
// registers, so the next item's copy may start).
template <int DK, class ST, class F>
__device__ __forceinline__ void spec_candidate_dots(const SpecS<DK>& S, const float* kc,
                                                    const float* qx, int DKP, int n_c, int r8,
                                                    bool b2, bool b1, float* dsc, int jw,
                                                    bool writer, F&& after_first) {
#pragma unroll
  for (int t = 0; t < kSpecK; t += 2) {
    if (t < n_c) {
      const float* xr[4] = {kc + t * DKP, kc + (t + 1) * DKP, qx + t * DKP, qx + (t + 1) * DKP};
      float out[4];
      spec_dots<DK, ST, 4>(S, xr, r8, b2, b1, out);
      if (writer) {
        dsc[t * 16 + jw] = out[0];
        dsc[(t + 1) * 16 + jw] = out[1];
        dsc[(kSpecK + t) * 16 + jw] = out[2];
        dsc[(kSpecK + t + 1) * 16 + jw] = out[3];
      }
      if (t == 0) after_first();
    }
  }
}

// The candidates' per-column work of one item once their dot products are in
// the warp's scratch: c_t = v_t - G_t/|k_t| (S^T k_t), the outputs
// o_t = scale (G_t/|q_t| (S^T q_t) + sum_s N[t][s] c_s), then
// u_t = sum_s M[t][s] c_s, for column jc of the warp and the rows
// t = 2 tt + th. v_t of the column at vsrc[t * vstride]; o_t at
// o0 + t * ostride; u_t is handed to put_u(t, u).
template <class IO, class PutU>
__device__ __forceinline__ void spec_candidate_columns(const RunCoef& C, const float* dsc, int jc,
                                                       int th, int n_c, const IO* vsrc,
                                                       int vstride, float scale, void* o,
                                                       int out_f32, size_t o0, size_t ostride,
                                                       PutU&& put_u) {
  float c[kSpecK];
#pragma unroll
  for (int t = 0; t < kSpecK; ++t)
    c[t] = (t < n_c) ? __fmaf_rn(-C.gk[t], dsc[t * 16 + jc], to_f(vsrc[(size_t)t * vstride]))
                     : 0.0f;
#pragma unroll
  for (int tt = 0; tt < kSpecK / 2; ++tt) {
    const int t = 2 * tt + th;
    if (t < n_c) {
      float acc = __fmul_rn(C.gq[t], dsc[(kSpecK + t) * 16 + jc]);
#pragma unroll
      for (int s = 0; s <= 2 * tt + 1; ++s)
        if (s <= t) acc = __fmaf_rn(C.nq[t][s], c[s], acc);
      store_out(o, out_f32, o0 + (size_t)t * ostride, __fmul_rn(scale, acc));
    }
  }
#pragma unroll
  for (int tt = 0; tt < kSpecK / 2; ++tt) {
    const int t = 2 * tt + th;
    if (t < n_c) {
      float acc = __fmul_rn(C.m[t][0], c[0]);
#pragma unroll
      for (int s = 1; s <= 2 * tt + 1; ++s)
        if (s <= t) acc = __fmaf_rn(C.m[t][s], c[s], acc);
      put_u(t, acc);
    }
  }
}

// ---------------------------------------------------------------------------
// One-page step, part 1: the candidates' run coefficients per value head.
template <class IO, class ST, int DK>
__global__ void __launch_bounds__(kSpecThreads)
spec_coef_kernel(Geom G, Batch B, Params P, const IO* __restrict__ rows_in,
                 const IO* __restrict__ a_in, const IO* __restrict__ b_in, void* pages,
                 int32_t* status) {
  constexpr int NT = kSpecThreads;
  constexpr int DV = DK;
  constexpr int VE = 16 / (int)sizeof(IO);
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_begin();

  const int Gh = G.Hv / G.Hk;
  const int kh = blockIdx.x, h0 = kh * Gh;
  const int tid = threadIdx.x;
  const bool reporter = (blockIdx.x == 0 && tid == 0);
  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  if (!q.spec) return;

  const SpecSmem L = spec_smem(LAYOUT_COEF, DK, DV, Gh, (int)sizeof(IO), (int)sizeof(ST), 0);
  IO* raw = reinterpret_cast<IO*>(smem + L.raw);
  float* abs_ = reinterpret_cast<float*>(smem + L.ab);
  float* hc = reinterpret_cast<float*>(smem + L.hc);
  const int RW = L.RW;
  const int q_off = kh * DK, k_off = G.Hk * DK + kh * DK;
  const int n_c = (q.len <= G.Kc) ? q.len : 0;   // (more is an error, found below)
  // channel of row element c (q | k of the group)
  auto chan = [&](int c) { return (c < DK) ? q_off + c : k_off + (c - DK); };

  // ---- the candidates' q and k rows start copying; the flag word, the gate
  // inputs and the heads' constants are loaded together (none depends on
  // another), then the page is checked
  {
    constexpr int pieces = 2 * DK / VE;
    for (int idx = tid; idx < n_c * pieces; idx += NT) {
      const int t = idx / pieces, c = (idx % pieces) * VE;
      cp_async16(raw + (size_t)t * RW + c, rows_in + (size_t)(q.start + t) * G.C + chan(c));
    }
  }
  cp_async_commit();
  char* pg = page_ptr(G, pages, q.page);
  uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
  const uint32_t flag = *reinterpret_cast<volatile uint32_t*>(flagp);
  for (int idx = tid; idx < n_c * Gh; idx += NT) {
    const int t = idx / Gh, g = idx % Gh;
    const size_t rn = ((size_t)q.start + t) * G.Hv + h0 + g;
    abs_[t * 2 * Gh + g] = to_f(a_in[rn]);
    abs_[t * 2 * Gh + Gh + g] = to_f(b_in[rn]);
  }
  for (int g = tid; g < Gh; g += NT) {
    hc[2 * g] = P.A_log[h0 + g];
    hc[2 * g + 1] = P.dt_bias[h0 + g];
  }
  SpecState ss = spec_state(G, B, q, flag);
  if (q.fresh) ss.err = GDN_DEV_BAD_FLAG;
  if (ss.err) {
    if (reporter) report(status, ss.err);
    cp_async_wait_all();   // nothing lands after the CTA is gone
    return;
  }
  IO* rec_out = reinterpret_cast<IO*>(pg + G.record_off) + (size_t)(1 - ss.live) * G.Kc * G.rec_row;

  // the candidates' gate inputs go next to their conv'd rows in the record slot
  for (int idx = tid; idx < n_c * Gh; idx += NT) {
    const int t = idx / Gh, g = idx % Gh, h = h0 + g;
    const size_t rn = ((size_t)q.start + t) * G.Hv + h;
    IO* rr = rec_out + (size_t)t * G.rec_row;
    rr[G.C + h] = a_in[rn];
    rr[G.C + G.Hv + h] = b_in[rn];
  }
  cp_async_wait_all();
  __syncthreads();
  if (n_c == 0) return;

  float* kx = reinterpret_cast<float*>(smem + L.kx);
  float* qx = reinterpret_cast<float*>(smem + L.qx);
  spec_rows_f32<DK, ST, IO, NT>(kx, L.DKP, raw + DK, RW, n_c);
  spec_rows_f32<DK, ST, IO, NT>(qx, L.DKP, raw, RW, n_c);
  __syncthreads();
  RunCoef* coef = reinterpret_cast<RunCoef*>(smem + L.coef);
  spec_candidate_coefs<DK, NT>(P, Gh, 0, Gh, n_c, kx, qx, L.DKP, abs_, hc,
                               *reinterpret_cast<RunDots*>(smem + L.dots),
                               reinterpret_cast<float*>(smem + L.gates), coef);
  // the record's coefficient blocks of the slot the candidates go to
  float* rc = reinterpret_cast<float*>(pg + G.rcoef_off) + (size_t)(1 - ss.live) * G.Hv * kRunCoefFloats;
  for (int idx = tid; idx < Gh * kCoefPieces; idx += NT) {
    const int g = idx / kCoefPieces, k = idx % kCoefPieces;
    *reinterpret_cast<float4*>(rc + (size_t)(h0 + g) * kRunCoefFloats + 4 * k) =
        *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(&coef[g]) +
                                         spec_coef_piece(k));
  }
}

// ---------------------------------------------------------------------------
// One-page step, part 2: replay, checkpoint and the candidates, per item.
// rows_in: the candidates' conv'd rows. nsplit CTAs per value head, each
// with Dv / (BVI nsplit) items of BVI columns.
//
// 3 CTAs per SM (150 registers at fp32 state, 70 KB of shared memory; at bf16
// state a fourth CTA, at 128 registers with small spills, ran no faster).
template <class IO, class ST, int DK>
__global__ void __launch_bounds__(kSpecThreads, 3)
spec_item_kernel(Geom G, Batch B, Params P, const IO* __restrict__ rows_in, void* o, int out_f32,
                 void* pages, int32_t* status, int nsplit) {
  using M = SpecMap<DK, ST>;
  constexpr int DV = DK;
  constexpr int VE = 16 / (int)sizeof(IO);
  extern __shared__ __align__(16) uint8_t smem[];

  const int Gh = G.Hv / G.Hk;
  const int h = blockIdx.x / nsplit, sp = blockIdx.x % nsplit, kh = h / Gh;
  const int BVI = DV < kSpecBV ? DV : kSpecBV;     // columns per item
  const int per = DV / BVI / nsplit;               // items per CTA
  const int cb0 = sp * per;                        // first column block
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r8 = lane & 7, cg = lane >> 3;
  const bool b2 = (r8 & 4) != 0, b1 = (r8 & 2) != 0;
  const int colw = 16 * warp + 4 * cg;             // the lane's first column in an item
  const int cown = 2 * (b2 ? 1 : 0) + (b1 ? 1 : 0); // the column its dot products end in
  const bool active = colw < BVI;
  const bool reporter = (blockIdx.x == 0 && tid == 0);

  // Until the wait on the coefficient kernel, this kernel uses only what the
  // launches before that kernel wrote (it lets this one start only once they
  // have completed): the request, the state, the flag word, the live record
  // slot, the record's u and the caller's rows. (It also copies the other
  // record slot, which the coefficient kernel may be writing, and ignores it.)
  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  if (!q.spec) return;

  const SpecSmem L = spec_smem(LAYOUT_ITEMS, DK, DV, Gh, (int)sizeof(IO), (int)sizeof(ST), per * BVI);
  IO* rawk = reinterpret_cast<IO*>(smem + L.rawk);
  IO* rawq = reinterpret_cast<IO*>(smem + L.rawq);
  IO* rawv = reinterpret_cast<IO*>(smem + L.rawv);
  float* ur = reinterpret_cast<float*>(smem + L.ur);
  float* kx = reinterpret_cast<float*>(smem + L.kx);
  float* qx = reinterpret_cast<float*>(smem + L.qx);
  RunCoef* coef = reinterpret_cast<RunCoef*>(smem + L.coef);   // slots 0, 1; candidates
  uint8_t* stage = smem + L.stage;
  const int DKP = L.DKP, VW = L.VW;
  const int q_off = kh * DK, k_off = G.Hk * DK + kh * DK;
  const int v_off = 2 * G.Hk * DK + h * DV + cb0 * BVI;     // the CTA's first v column
  const int n_c = q.len;

  char* pg = page_ptr(G, pages, q.page);
  ST* Sbase = reinterpret_cast<ST*>(pg + G.state_off);
  auto item_col0 = [&](int cb) -> ST* {
    return Sbase + ((size_t)h * DV + (size_t)cb * BVI + colw) * DK;
  };

  // ---- 1. everything the setup reads from memory, at once: the first
  // item's state, the flag word and the accepted count, both record slots' k
  // rows and G, R/|k| blocks (which one is live comes with the flag), the
  // record's u of the CTA's columns, and the caller's candidate rows
  if (active) spec_stage_async<DK, ST>(stage, item_col0(cb0), r8, tid);
  uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
  const int acc = B.n_accepted ? B.n_accepted[q.r] : -1;
  const uint32_t flag = *reinterpret_cast<volatile uint32_t*>(flagp);
  const IO* rec = reinterpret_cast<const IO*>(pg + G.record_off);
  constexpr int RP = DK / VE;   // 16-byte pieces per q or k row
  const int VP = VW / VE;
  const int per_row = 2 * RP + VP;
  for (int idx = tid; idx < 2 * G.Kc * RP; idx += kSpecThreads) {
    const int st = idx / (G.Kc * RP), t = (idx / RP) % G.Kc, c = (idx % RP) * VE;
    cp_async16(rawk + (size_t)(st * kSpecK + t) * DK + c,
               rec + ((size_t)st * G.Kc + t) * G.rec_row + k_off + c);
  }
  for (int idx = tid; idx < 2 * 18; idx += kSpecThreads) {   // gam, rk of both slots
    const int st = idx / 18, k = 4 + idx % 18;
    const float* rc = reinterpret_cast<const float*>(pg + G.rcoef_off) +
                      ((size_t)st * G.Hv + h) * kRunCoefFloats;
    cp_async16(reinterpret_cast<float*>(&coef[st]) + spec_coef_piece(k), rc + 4 * k);
  }
  float* urec = reinterpret_cast<float*>(pg + G.ru_off) + (size_t)h * G.Kc * DV + cb0 * BVI;
  {
    const int UP = VW / 4;
    for (int idx = tid; idx < G.Kc * UP; idx += kSpecThreads) {
      const int s = idx / UP, c = (idx % UP) * 4;
      cp_async16(ur + (size_t)s * VW + c, urec + (size_t)s * DV + c);
    }
  }
  // where the candidates' piece p of row t goes, and where it comes from
  auto cand_dst = [&](int t, int p) -> IO* {
    return (p < RP) ? rawq + (size_t)t * DK + p * VE
         : (p < 2 * RP) ? rawk + (size_t)(2 * kSpecK + t) * DK + (p - RP) * VE
                        : rawv + (size_t)t * VW + (p - 2 * RP) * VE;
  };
  auto cand_src = [&](const IO* row, int p) -> const IO* {
    return row + ((p < RP) ? q_off + p * VE : (p < 2 * RP) ? k_off + (p - RP) * VE
                                                           : v_off + (p - 2 * RP) * VE);
  };
  if (n_c <= G.Kc) {
    for (int idx = tid; idx < n_c * per_row; idx += kSpecThreads) {
      const int t = idx / per_row, p = idx % per_row;
      cp_async16(cand_dst(t, p), cand_src(rows_in + (size_t)(q.start + t) * G.C, p));
    }
  }
  cp_async_commit();
  SpecState ss = spec_state_acc(G, q, flag, acc);
  if (q.fresh) ss.err = GDN_DEV_BAD_FLAG;
  if (ss.err) {
    if (reporter) report(status, ss.err);
    cp_async_wait_all();   // nothing lands after the CTA is gone
    return;
  }
  const int n_r = (ss.width > 0) ? ss.accepted + 1 : 0;
  const int live = ss.live, parity = ss.parity;
  // what the coefficient kernel wrote: the candidates' coefficients
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (n_c > 0) {
    const float* rc = reinterpret_cast<const float*>(pg + G.rcoef_off) +
                      ((size_t)(1 - live) * G.Hv + h) * kRunCoefFloats;
    for (int i = tid; i < 36; i += kSpecThreads) {   // gk, gq, m, nq
      const int k = (i < 4) ? i : 18 + i;
      cp_async16(reinterpret_cast<float*>(&coef[2]) + spec_coef_piece(k), rc + 4 * k);
    }
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();

  // ---- 2. fp32 copies of the rows, in the order the lanes read them: the
  // live slot's replayed k rows at 0.., candidates' k rows at kSpecK.., q rows
  spec_rows_f32<DK, ST, IO, kSpecThreads>(kx, DKP, rawk + (size_t)live * kSpecK * DK, DK, n_r);
  spec_rows_f32<DK, ST, IO, kSpecThreads>(kx + kSpecK * DKP, DKP, rawk + 2 * kSpecK * DK, DK, n_c);
  spec_rows_f32<DK, ST, IO, kSpecThreads>(qx, DKP, rawq, DK, n_c);
  __syncthreads();

  // ---- 3. items: no block-wide barrier from here on. The next item's state
  // starts copying once this one's is in registers.
  const bool work = active && (n_r + n_c > 0);
  float* dsc = reinterpret_cast<float*>(smem + L.scr) + warp * kSpecScr;
  const int jw = 4 * cg + cown;                 // this lane's column in the warp
  const bool writer = (r8 & 1) == 0;            // one of the column's two lanes
  // the per-column phase maps lane -> (column jc of the warp, row half th)
  const int jc = lane & 15, th = lane >> 4;
  // the candidates' u replace the replayed rows' u (read above) in the record
  float* uout = reinterpret_cast<float*>(pg + G.ru_off) + (size_t)h * G.Kc * DV;
  for (int it = 0; it < per; ++it) {
    const int cb = cb0 + it;
    ST* col0 = item_col0(cb);
    SpecS<DK> S;
    bool ahead = !work || (it + 1 >= per);
    auto prefetch = [&]() {
      if (!ahead) {
        spec_stage_async<DK, ST>(stage, item_col0(cb + 1), r8, tid);
        ahead = true;
      }
    };
    if (work) {
      spec_stage_wait();
      spec_unstage<DK, ST>(S, stage, tid);
    }
    if (work && n_r > 0) {
      // the replay: S_a from the stored u of the accepted rows
      spec_advance<DK, ST>(S, coef[live], n_r - 1, kx, DKP, ur + it * BVI + colw, VW, r8);
      prefetch();
      spec_store<DK, ST>(col0, S, r8);
      // continue from exactly what was stored (a bf16 page rounds here)
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int p = 0; p < M::P; ++p)
          S.s[m][p] = make_float2(through<ST>(S.s[m][p].x), through<ST>(S.s[m][p].y));
    }
    if (work && n_c > 0) {
      spec_candidate_dots<DK, ST>(S, kx + kSpecK * DKP, qx, DKP, n_c, r8, b2, b1, dsc, jw,
                                  writer, prefetch);
      __syncwarp();
      const int col = cb * BVI + 16 * warp + jc;   // the column of jc in the head
      spec_candidate_columns<IO>(
          coef[2], dsc, jc, th, n_c, rawv + it * BVI + 16 * warp + jc, VW, P.scale, o, out_f32,
          (size_t)q.start * G.Hv * DV + (size_t)h * DV + col, (size_t)G.Hv * DV,
          [&](int t, float u) { uout[(size_t)t * DV + col] = u; });
      __syncwarp();   // dsc is written again only after this
    }
    prefetch();   // (a run with no rows never consumed the stage)
  }
  spec_stage_wait();   // no copy outlives the CTA's shared memory

  // ---- 4. the last CTA of the request publishes the new flag word -------
  // No fence orders the page data first: only later launches read it. The
  // counter needs none either: every CTA read the flag before its own
  // increment of the same word, so the publish follows every read.
  if (tid == 0) {
    const uint32_t total = (uint32_t)(G.Hv * nsplit);
    const uint32_t old = atomicAdd(flagp, 256u);
    if ((old >> 8) == total - 1) {
      const int nl = (n_c > 0) ? 1 - live : live;
      atomicExch(flagp, make_flag(nl, 1 - parity, n_c));
    }
  }
}

// ---------------------------------------------------------------------------
// The fused step (gdn_spec_step) in one launch: one CTA per (request, q/k
// head kh) convolves the group's channels for this step's candidates (as the
// coefficient kernel's fused form does), forms the group's run coefficients,
// and then runs every item of the group as the item kernel does, with the
// same helpers: the same bits as gdn_conv + gdn_spec_verify, pages included.

// The replay's G and R/|k| of one value head, as the record keeps them
// (floats 16 .. 87 of its coefficient block).
struct RepCoef {
  float gam[kSpecK];
  float rk[kSpecK][kSpecK];
};
static_assert(sizeof(RepCoef) == 72 * 4, "record floats 16..87");

struct StepSmem {
  uint32_t raw;     // [Kc][RW] io dtype: the candidates' conv'd q | k | v of the group
  uint32_t ab;      // [Kc][2 Gh] float: a then b per head
  uint32_t hc;      // [Gh][2] float: A_log, dt_bias per head
  uint32_t kx;      // [2 Kc][DKP] float: replayed k rows 0.., candidates' k rows kSpecK..
  uint32_t qx;      // [Kc][DKP] float: candidates' q rows
  uint32_t dots;    // RunDots
  uint32_t gates;   // [Gh][2][Kc] float
  uint32_t coef;    // [Gh] RunCoef: the candidates'
  uint32_t rep;     // [Gh] RepCoef: the replay's
  uint32_t rawr;    // [Kc][DK] io dtype: the replayed k rows
  uint32_t ur;      // [Gh][Kc][DV] float: the replayed rows' u
  uint32_t stage;   // [NC][threads] 16-byte chunks of one item's state
  uint32_t scr;     // per warp [2 Kc][16] dot products
  uint32_t total;
  int RW, DKP;
};

__host__ __device__ inline StepSmem step_smem(int DK, int DV, int Gh, int io_bytes, int st_bytes) {
  StepSmem L;
  const uint32_t K = kSpecK;
  L.DKP = DK + 4;
  L.RW = (2 * DK + Gh * DV + 7) / 8 * 8;
  uint32_t off = 0;
  auto take = [&](uint32_t& at, uint32_t bytes) {
    at = off;
    off = spec_al16(off + bytes);
  };
  take(L.raw, K * L.RW * io_bytes);
  take(L.ab, K * 2 * Gh * 4);
  take(L.hc, Gh * 2 * 4);
  take(L.kx, 2 * K * L.DKP * 4);
  take(L.qx, K * L.DKP * 4);
  take(L.dots, (uint32_t)sizeof(RunDots));
  take(L.gates, Gh * 2 * K * 4);
  take(L.coef, (uint32_t)Gh * (uint32_t)sizeof(RunCoef));
  take(L.rep, (uint32_t)Gh * (uint32_t)sizeof(RepCoef));
  take(L.rawr, K * DK * io_bytes);
  take(L.ur, Gh * K * DV * 4);
  take(L.stage, (uint32_t)(DK / 2 * st_bytes * kSpecThreads));
  take(L.scr, (uint32_t)((kSpecThreads / 32) * 2 * kSpecK * 16 * 4));
  L.total = off;
  return L;
}

// 3 CTAs per SM at Dk = Dv = 128 with Gh = 2 (about 72 KB of shared memory).
template <class IO, class ST, int DK>
__global__ void __launch_bounds__(kSpecThreads, 3)
spec_step_kernel(Geom G, Batch B, Params P, const IO* __restrict__ x_in,
                 const IO* __restrict__ conv_w, const IO* __restrict__ a_in,
                 const IO* __restrict__ b_in, void* o, int out_f32, void* pages,
                 int32_t* status) {
  using M = SpecMap<DK, ST>;
  constexpr int DV = DK;
  constexpr int VE = 16 / (int)sizeof(IO);
  constexpr int BVI = DV < kSpecBV ? DV : kSpecBV;   // columns per item
  constexpr int nCB = DV / BVI;
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_begin();

  const int Gh = G.Hv / G.Hk;
  const int kh = blockIdx.x, h0 = kh * Gh;
  const int n_items = Gh * nCB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r8 = lane & 7, cg = lane >> 3;
  const bool b2 = (r8 & 4) != 0, b1 = (r8 & 2) != 0;
  const int colw = 16 * warp + 4 * cg;             // the lane's first column in an item
  const int cown = 2 * (b2 ? 1 : 0) + (b1 ? 1 : 0);
  const bool active = colw < BVI;
  const bool reporter = (blockIdx.x == 0 && tid == 0);
  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  if (!q.spec) return;

  const StepSmem L = step_smem(DK, DV, Gh, (int)sizeof(IO), (int)sizeof(ST));
  IO* raw = reinterpret_cast<IO*>(smem + L.raw);
  float* abs_ = reinterpret_cast<float*>(smem + L.ab);
  float* hc = reinterpret_cast<float*>(smem + L.hc);
  float* kx = reinterpret_cast<float*>(smem + L.kx);
  float* qx = reinterpret_cast<float*>(smem + L.qx);
  RunCoef* coef = reinterpret_cast<RunCoef*>(smem + L.coef);
  RepCoef* rep = reinterpret_cast<RepCoef*>(smem + L.rep);
  IO* rawr = reinterpret_cast<IO*>(smem + L.rawr);
  float* ur = reinterpret_cast<float*>(smem + L.ur);
  uint8_t* stage = smem + L.stage;
  const int RW = L.RW, DKP = L.DKP;
  const int q_off = kh * DK, k_off = G.Hk * DK + kh * DK, v_off = 2 * G.Hk * DK + h0 * DV;
  // channel of group element c (q | k | v of the group's heads)
  auto chan = [&](int c) {
    return (c < DK) ? q_off + c : (c < 2 * DK) ? k_off + (c - DK) : v_off + (c - 2 * DK);
  };

  char* pg = page_ptr(G, pages, q.page);
  ST* Sbase = reinterpret_cast<ST*>(pg + G.state_off);
  auto item_col0 = [&](int it) -> ST* {
    return Sbase + ((size_t)(h0 + it / nCB) * DV + (size_t)(it % nCB) * BVI + colw) * DK;
  };
  // ---- 1. the first item's state starts copying; the flag word and the
  // heads' constants are loaded, then the page is checked
  if (active) spec_stage_async<DK, ST>(stage, item_col0(0), r8, tid);
  uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
  const uint32_t flag = *reinterpret_cast<volatile uint32_t*>(flagp);
  for (int g = tid; g < Gh; g += kSpecThreads) {
    hc[2 * g] = P.A_log[h0 + g];
    hc[2 * g + 1] = P.dt_bias[h0 + g];
  }
  SpecState ss = spec_state(G, B, q, flag);
  if (q.fresh) ss.err = GDN_DEV_BAD_FLAG;
  if (ss.err) {
    if (reporter) report(status, ss.err);
    cp_async_wait_all();   // nothing lands after the CTA is gone
    return;
  }
  const int n_r = (ss.width > 0) ? ss.accepted + 1 : 0;
  const int n_c = q.len;
  const int live = ss.live, parity = ss.parity;
  IO* rec = reinterpret_cast<IO*>(pg + G.record_off);
  const IO* rslot = rec + (size_t)live * G.Kc * G.rec_row;
  IO* rec_out = rec + (size_t)(1 - live) * G.Kc * G.rec_row;

  // ---- 2. the replay's inputs from the live record slot: its k rows, per
  // head G and R/|k|, and the u of the accepted rows
  constexpr int RP = DK / VE;   // 16-byte pieces per k row
  for (int idx = tid; idx < n_r * RP; idx += kSpecThreads) {
    const int t = idx / RP, c = (idx % RP) * VE;
    cp_async16(rawr + (size_t)t * DK + c, rslot + (size_t)t * G.rec_row + k_off + c);
  }
  if (n_r > 0) {
    constexpr int RQ = (int)sizeof(RepCoef) / 16;
    for (int idx = tid; idx < Gh * RQ; idx += kSpecThreads) {
      const int g = idx / RQ, k = idx % RQ;
      const float* rc = reinterpret_cast<const float*>(pg + G.rcoef_off) +
                        ((size_t)live * G.Hv + h0 + g) * kRunCoefFloats;
      cp_async16(reinterpret_cast<float*>(&rep[g]) + 4 * k, rc + 16 + 4 * k);
    }
    constexpr int UP = DV / 4;
    const float* us = reinterpret_cast<const float*>(pg + G.ru_off) + (size_t)h0 * G.Kc * DV;
    for (int idx = tid; idx < Gh * n_r * UP; idx += kSpecThreads) {
      const int g = idx / (n_r * UP), s = (idx / UP) % n_r, c = (idx % UP) * 4;
      cp_async16(ur + ((size_t)g * kSpecK + s) * DV + c, us + ((size_t)g * G.Kc + s) * DV + c);
    }
  }
  cp_async_commit();

  // ---- 3. the conv of the group's channels for this step's candidates,
  // exactly as gdn_conv computes it for a spec request: history = window
  // columns n_r .. n_r+W-2, taps oldest first, own SiLU, rounded to the io
  // dtype; the rows go to shared memory and the record slot, the window rolls
  {
    const int nvec = (2 * DK + Gh * DV) / 4;
    IO* win = reinterpret_cast<IO*>(pg + G.window_off);
    for (int vi = tid; vi < nvec; vi += kSpecThreads) {
      const int c4 = 4 * vi;
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
        if (t < n_c) load_f<IO, 4>(x_in + (size_t)(q.start + t) * G.C + ch, xr[t]);
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
          store_f<IO, 4>(raw + (size_t)t * RW + c4, yv);
          store_f<IO, 4>(rec_out + (size_t)t * G.rec_row + ch, yv);
          store_f<IO, 4>(win + (size_t)(3 + t) * G.C + ch, xr[t]);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            hcol[0][v] = hcol[1][v];
            hcol[1][v] = hcol[2][v];
            hcol[2][v] = xr[t][v];
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 3; ++j) store_f<IO, 4>(win + (size_t)j * G.C + ch, h0c[j]);
    }
  }
  // gate inputs per candidate and head; they also go next to the
  // candidates' conv'd rows in the record slot
  for (int idx = tid; idx < n_c * Gh; idx += kSpecThreads) {
    const int t = idx / Gh, g = idx % Gh, h = h0 + g;
    const size_t rn = ((size_t)q.start + t) * G.Hv + h;
    abs_[t * 2 * Gh + g] = to_f(a_in[rn]);
    abs_[t * 2 * Gh + Gh + g] = to_f(b_in[rn]);
    IO* rr = rec_out + (size_t)t * G.rec_row;
    rr[G.C + h] = a_in[rn];
    rr[G.C + G.Hv + h] = b_in[rn];
  }
  cp_async_wait_all();
  __syncthreads();

  // ---- 4. fp32 rows in the lanes' order (replayed k rows at 0.., the
  // candidates' k rows at kSpecK.., their q rows), then the candidates'
  // coefficients, which also go to the record slot they are written to
  spec_rows_f32<DK, ST, IO, kSpecThreads>(kx, DKP, rawr, DK, n_r);
  spec_rows_f32<DK, ST, IO, kSpecThreads>(kx + kSpecK * DKP, DKP, raw + DK, RW, n_c);
  spec_rows_f32<DK, ST, IO, kSpecThreads>(qx, DKP, raw, RW, n_c);
  __syncthreads();
  if (n_c > 0) {
    spec_candidate_coefs<DK, kSpecThreads>(P, Gh, 0, Gh, n_c, kx + kSpecK * DKP, qx, DKP, abs_,
                                           hc, *reinterpret_cast<RunDots*>(smem + L.dots),
                                           reinterpret_cast<float*>(smem + L.gates), coef);
    float* rc = reinterpret_cast<float*>(pg + G.rcoef_off) + (size_t)(1 - live) * G.Hv * kRunCoefFloats;
    for (int idx = tid; idx < Gh * kCoefPieces; idx += kSpecThreads) {
      const int g = idx / kCoefPieces, k = idx % kCoefPieces;
      *reinterpret_cast<float4*>(rc + (size_t)(h0 + g) * kRunCoefFloats + 4 * k) =
          *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(&coef[g]) +
                                           spec_coef_piece(k));
    }
  }

  // ---- 5. items (value head g, column block cb): no block-wide barrier
  // from here on. The next item's state starts copying once this one's is in
  // registers.
  if (active && n_r + n_c > 0) {
    float* dsc = reinterpret_cast<float*>(smem + L.scr) + warp * 2 * kSpecK * 16;
    const int jw = 4 * cg + cown;
    const bool writer = (r8 & 1) == 0;
    const int jc = lane & 15, th = lane >> 4;
    for (int it = 0; it < n_items; ++it) {
      const int g = it / nCB, cb = it % nCB, h = h0 + g;
      ST* col0 = item_col0(it);
      spec_stage_wait();
      SpecS<DK> S;
      spec_unstage<DK, ST>(S, stage, tid);
      bool ahead = (it + 1 >= n_items);
      auto prefetch = [&]() {
        if (!ahead) {
          spec_stage_async<DK, ST>(stage, item_col0(it + 1), r8, tid);
          ahead = true;
        }
      };
      if (n_r > 0) {
        // the replay: S_a from the stored u of the accepted rows
        spec_advance<DK, ST>(S, rep[g], n_r - 1, kx, DKP,
                             ur + (size_t)g * kSpecK * DV + cb * BVI + colw, DV, r8);
        prefetch();
        spec_store<DK, ST>(col0, S, r8);
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int p = 0; p < M::P; ++p)
            S.s[m][p] = make_float2(through<ST>(S.s[m][p].x), through<ST>(S.s[m][p].y));
      }
      if (n_c > 0) {
        spec_candidate_dots<DK, ST>(S, kx + kSpecK * DKP, qx, DKP, n_c, r8, b2, b1, dsc, jw,
                                    writer, prefetch);
        __syncwarp();
        const int col = cb * BVI + 16 * warp + jc;   // the column of jc in the head
        float* uout = reinterpret_cast<float*>(pg + G.ru_off) + (size_t)h * G.Kc * DV;
        spec_candidate_columns<IO>(coef[g], dsc, jc, th, n_c, raw + 2 * DK + g * DV + col, RW,
                                   P.scale, o, out_f32,
                                   (size_t)q.start * G.Hv * DV + (size_t)h * DV + col,
                                   (size_t)G.Hv * DV,
                                   [&](int t, float u) { uout[(size_t)t * DV + col] = u; });
        __syncwarp();   // dsc is written again only after this
      }
      prefetch();
    }
  }
  spec_stage_wait();   // no copy outlives the CTA's shared memory

  // ---- 6. the last CTA of the request publishes the new flag word (every
  // CTA read the flag before its own increment of the same word)
  if (tid == 0) {
    const uint32_t total = (uint32_t)G.Hk;
    const uint32_t old = atomicAdd(flagp, 256u);
    if ((old >> 8) == total - 1) {
      const int nl = (n_c > 0) ? 1 - live : live;
      atomicExch(flagp, make_flag(nl, 1 - parity, n_c));
    }
  }
}

// ---------------------------------------------------------------------------
// Slot-per-candidate layout. 2 CTAs per SM (240 registers): the per-candidate
// rebuild keeps a second state in registers, and at 3 per SM it spilled 280
// bytes and ran 294 us per 64-request step, against 244 us at 2.
template <class IO, class ST, int DK>
__global__ void __launch_bounds__(kSpecThreads, 2)
spec_slots_kernel(Geom G, Batch B, Params P, SlotGeom SG, const IO* __restrict__ rows_in,
                  const IO* __restrict__ a_in, const IO* __restrict__ b_in, void* o,
                  int out_f32, void* pools, int32_t* status, int splits) {
  constexpr int DV = DK;
  constexpr int VE = 16 / (int)sizeof(IO);
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
  const bool b2 = (r8 & 4) != 0, b1 = (r8 & 2) != 0;
  const int colw = 16 * warp + 4 * cg;
  const int cown = 2 * (b2 ? 1 : 0) + (b1 ? 1 : 0);
  const bool active = colw < BVI;
  const bool reporter = (blockIdx.x == 0 && tid == 0);

  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }

  const SpecSmem L = spec_smem(LAYOUT_SLOTS, DK, DV, Gh, (int)sizeof(IO), (int)sizeof(ST), 0);
  IO* raw = reinterpret_cast<IO*>(smem + L.raw);
  float* abs_ = reinterpret_cast<float*>(smem + L.ab);
  float* kx = reinterpret_cast<float*>(smem + L.kx);
  float* qx = reinterpret_cast<float*>(smem + L.qx);
  RunCoef* coef = reinterpret_cast<RunCoef*>(smem + L.coef);
  uint8_t* stage = smem + L.stage;
  const int RW = L.RW, DKP = L.DKP;
  const int g_lo = it0 / nCB, g_hi = (it1 > it0) ? (it1 - 1) / nCB + 1 : g_lo;  // own heads
  const int ng = g_hi - g_lo;
  const int q_off = kh * DK, k_off = G.Hk * DK + kh * DK, v_off = 2 * G.Hk * DK + h0 * DV;
  const int n_c = q.len;
  auto chan = [&](int c) {
    return (c < DK) ? q_off + c : (c < 2 * DK) ? k_off + (c - DK) : v_off + (c - 2 * DK);
  };
  const int pieces = (2 * DK + Gh * DV) / VE;

  // ---- 1. the candidates' rows start copying, then the source slot is checked
  if (q.len <= G.Kc) {
    for (int idx = tid; idx < n_c * pieces; idx += kSpecThreads) {
      const int t = idx / pieces, c = (idx % pieces) * VE;
      cp_async16(raw + (size_t)t * RW + c, rows_in + (size_t)(q.start + t) * G.C + chan(c));
    }
  }
  cp_async_commit();
  const int src = B.n_accepted ? B.n_accepted[q.r] : -1;
  int err = 0;
  if (src < 0 || src >= G.Kc) err = GDN_DEV_BAD_ACCEPTED;
  else if (q.len > G.Kc) err = GDN_DEV_TOO_MANY_CANDIDATES;
  if (err) {
    if (reporter) report(status, err);
    cp_async_wait_all();   // nothing lands after the CTA is gone
    return;
  }
  char* pg = reinterpret_cast<char*>(pools) + (size_t)q.page * SG.pool_bytes;
  ST* Sbase = reinterpret_cast<ST*>(pg + (size_t)src * SG.slot_bytes + SG.state_off);
  auto item_col0 = [&](int it) -> ST* {
    const int hh = h0 + it / nCB, cb = it % nCB;
    return Sbase + ((size_t)hh * DV + (size_t)cb * BVI + colw) * DK;
  };
  if (active && it0 < it1) spec_stage_async<DK, ST>(stage, item_col0(it0), r8, tid);
  else cp_async_commit();   // keep "all but the newest group" meaning the rows

  // ---- 2. gate inputs and constants of own heads
  float* hc = reinterpret_cast<float*>(smem + L.hc);
  for (int idx = tid; idx < n_c * ng; idx += kSpecThreads) {
    const int t = idx / ng, g = g_lo + idx % ng, hh = h0 + g;
    const size_t rn = (size_t)q.start + t;
    abs_[t * 2 * Gh + g] = to_f(a_in[rn * G.Hv + hh]);
    abs_[t * 2 * Gh + Gh + g] = to_f(b_in[rn * G.Hv + hh]);
  }
  for (int g = g_lo + tid; g < g_hi; g += kSpecThreads) {
    hc[2 * g] = P.A_log[h0 + g];
    hc[2 * g + 1] = P.dt_bias[h0 + g];
  }
  cp_async_wait_all_but_one();   // the rows (not the state) have landed
  __syncthreads();

  // ---- 3. fp32 copies of the k and q rows, then the coefficients, with the
  // one-page step's code
  spec_rows_f32<DK, ST, IO, kSpecThreads>(kx, DKP, raw + DK, RW, n_c);
  spec_rows_f32<DK, ST, IO, kSpecThreads>(qx, DKP, raw, RW, n_c);
  __syncthreads();
  spec_candidate_coefs<DK, kSpecThreads>(P, Gh, g_lo, ng, n_c, kx, qx, DKP, abs_, hc,
                                         *reinterpret_cast<RunDots*>(smem + L.dots),
                                         reinterpret_cast<float*>(smem + L.gates), coef);

  // ---- 4. items: the candidates from the source slot's state, then the
  // state after every candidate to its slot, each rebuilt from the staged
  // starting state
  if (active && n_c > 0) {
    const IO* vraw = raw + 2 * DK;
    float* dsc = reinterpret_cast<float*>(smem + L.scr) + warp * kSpecScr;
    float* usc = dsc + 2 * kSpecK * 16;
    const int jw = 4 * cg + cown;
    const bool writer = (r8 & 1) == 0;
    const int jc = lane & 15, th = lane >> 4;
    for (int it = it0; it < it1; ++it) {
      const int g = it / nCB, cb = it % nCB, hh = h0 + g;
      ST* col0 = item_col0(it);
      if (it > it0) spec_stage_async<DK, ST>(stage, col0, r8, tid);
      spec_stage_wait();
      SpecS<DK> S;
      spec_unstage<DK, ST>(S, stage, tid);
      const RunCoef& C = coef[g];
      spec_candidate_dots<DK, ST>(S, kx, qx, DKP, n_c, r8, b2, b1, dsc, jw, writer, [] {});
      __syncwarp();
      const int col = cb * BVI + 16 * warp + jc;
      spec_candidate_columns<IO>(C, dsc, jc, th, n_c, vraw + g * DV + col, RW, P.scale, o,
                                 out_f32, (size_t)q.start * G.Hv * DV + (size_t)hh * DV + col,
                                 (size_t)G.Hv * DV, [&](int t, float u) { usc[t * 16 + jc] = u; });
      __syncwarp();
      const size_t off = (size_t)(col0 - Sbase);
      for (int t = 0; t < n_c; ++t) {
        SpecS<DK> T;
        spec_unstage<DK, ST>(T, stage, tid);
        spec_advance<DK, ST>(T, C, t, kx, DKP, usc + 4 * cg, 16, r8);
        ST* dst = reinterpret_cast<ST*>(pg + (size_t)t * SG.slot_bytes + SG.state_off) + off;
        spec_store<DK, ST>(dst, T, r8);
      }
      __syncwarp();   // dsc / usc are written again only after this
    }
  }
  spec_stage_wait();   // no copy outlives the CTA's shared memory
}

// Dynamic shared memory the spec kernels may ask for (their attribute is
// raised to it once per device).
constexpr int kSpecSmemMax = 200 * 1024;

// Items per CTA of the item kernel: two (one CTA per value head at Dv = 128)
// measured faster than one, whose setup (flag, record, coefficients) was
// exposed as often as its item.
#ifndef GDN_SPEC_ITEMS_PER_CTA
#define GDN_SPEC_ITEMS_PER_CTA 2
#endif

// CTAs per value head of the item kernel.
__host__ inline int spec_item_nsplit(int DV) {
  const int bvi = DV < kSpecBV ? DV : kSpecBV;
  const int ncb = DV / bvi;
  const int ipc = GDN_SPEC_ITEMS_PER_CTA;
  return (ipc >= 1 && ipc <= ncb && ncb % ipc == 0) ? ncb / ipc : ncb;
}

// The shared memory an entry point's kernels need for a shape: the
// coefficient and item kernels (SPEC_VERIFY), the one-launch step
// (SPEC_FUSED) or the slot kernel (SPEC_SLOTS).
__host__ inline uint32_t spec_smem_need(int mode, int DK, int Gh, int io_bytes, int st_bytes) {
  if (mode == SPEC_FUSED) return step_smem(DK, DK, Gh, io_bytes, st_bytes).total;
  if (mode == SPEC_SLOTS) return spec_smem(LAYOUT_SLOTS, DK, DK, Gh, io_bytes, st_bytes, 0).total;
  const uint32_t a =
      spec_smem(LAYOUT_ITEMS, DK, DK, Gh, io_bytes, st_bytes, DK / spec_item_nsplit(DK)).total;
  const uint32_t b = spec_smem(LAYOUT_COEF, DK, DK, Gh, io_bytes, st_bytes, 0).total;
  return a > b ? a : b;
}

template <int DK>
cudaError_t launch_spec_dk(int mode, const Geom& G, const Batch& B, const Params& P,
                           const SlotGeom& SG, int io_bf16, int state_bf16, int out_f32,
                           const void* rows, const void* conv_w, const void* a, const void* b,
                           void* o, void* pages, int32_t* status, int splits,
                           cudaStream_t stream) {
  const int Gh = G.Hv / G.Hk;
  const int iob = io_bf16 ? 2 : 4, stb = state_bf16 ? 2 : 4;
  if ((int)spec_smem_need(mode, DK, Gh, iob, stb) > kSpecSmemMax) return cudaErrorInvalidConfiguration;
  const dim3 block(kSpecThreads);
  const int nsplit = spec_item_nsplit(DK);
  const SpecSmem Lc = spec_smem(LAYOUT_COEF, DK, DK, Gh, iob, stb, 0);
  const SpecSmem Li = spec_smem(LAYOUT_ITEMS, DK, DK, Gh, iob, stb, DK / nsplit);
  const SpecSmem Ls = spec_smem(LAYOUT_SLOTS, DK, DK, Gh, iob, stb, 0);
  const StepSmem Lf = step_smem(DK, DK, Gh, iob, stb);
#define GDN_SPEC_ONE_PAGE(IO, ST)                                                              \
  do {                                                                                         \
    cudaError_t e = ensure_smem_limit<spec_coef_kernel<IO, ST, DK>>(kSpecSmemMax);             \
    if (e == cudaSuccess) e = ensure_smem_limit<spec_item_kernel<IO, ST, DK>>(kSpecSmemMax);   \
    if (e != cudaSuccess) return e;                                                            \
    e = launch_pdl(spec_coef_kernel<IO, ST, DK>, dim3(G.Hk, B.R), block, Lc.total, stream, G,  \
                   B, P, static_cast<const IO*>(rows), static_cast<const IO*>(a),              \
                   static_cast<const IO*>(b), pages, status);                                  \
    if (e != cudaSuccess) return e;                                                            \
    return launch_pdl(spec_item_kernel<IO, ST, DK>, dim3(G.Hv * nsplit, B.R), block, Li.total, \
                      stream, G, B, P, static_cast<const IO*>(rows), o, out_f32, pages,        \
                      status, nsplit);                                                         \
  } while (0)
#define GDN_SPEC_STEP(IO, ST)                                                                  \
  do {                                                                                         \
    cudaError_t e = ensure_smem_limit<spec_step_kernel<IO, ST, DK>>(kSpecSmemMax);             \
    if (e != cudaSuccess) return e;                                                            \
    return launch_pdl(spec_step_kernel<IO, ST, DK>, dim3(G.Hk, B.R), block, Lf.total, stream,  \
                      G, B, P, static_cast<const IO*>(rows), static_cast<const IO*>(conv_w),   \
                      static_cast<const IO*>(a), static_cast<const IO*>(b), o, out_f32, pages, \
                      status);                                                                 \
  } while (0)
#define GDN_SPEC_SLOTS(IO, ST)                                                                 \
  do {                                                                                         \
    cudaError_t e = ensure_smem_limit<spec_slots_kernel<IO, ST, DK>>(kSpecSmemMax);            \
    if (e != cudaSuccess) return e;                                                            \
    return launch_pdl(spec_slots_kernel<IO, ST, DK>, dim3(G.Hk * splits, B.R), block,          \
                      Ls.total, stream, G, B, P, SG, static_cast<const IO*>(rows),             \
                      static_cast<const IO*>(a), static_cast<const IO*>(b), o, out_f32, pages, \
                      status, splits);                                                         \
  } while (0)
#define GDN_SPEC_MODES(IO, ST)                                          \
  if (mode == SPEC_VERIFY) GDN_SPEC_ONE_PAGE(IO, ST);                   \
  else if (mode == SPEC_FUSED) GDN_SPEC_STEP(IO, ST);                   \
  else GDN_SPEC_SLOTS(IO, ST);
  if (io_bf16) {
    if (state_bf16) { GDN_SPEC_MODES(bf16, bf16) } else { GDN_SPEC_MODES(bf16, float) }
  } else {
    if (state_bf16) { GDN_SPEC_MODES(float, bf16) } else { GDN_SPEC_MODES(float, float) }
  }
#undef GDN_SPEC_MODES
#undef GDN_SPEC_SLOTS
#undef GDN_SPEC_STEP
#undef GDN_SPEC_ONE_PAGE
}

}  // namespace gdn
