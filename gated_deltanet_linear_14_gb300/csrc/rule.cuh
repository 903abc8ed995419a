// Token-by-token gated delta rule: gdn_seq, gdn_spec_verify and the
// slot-per-candidate layout (sm_103a).
//
// r9700-stack v0.2.3, section 1 (r9k_gdn_seq: any number of tokens, the state
// in registers, the batch's own rows); v0.2.4, "What it does" (one page per
// request: replay the accepted rows from the record, checkpoint, run the
// candidates; bit-identical to the slot design); vllm.cpp PR #155 (q/k L2
// norm and gates fused per token).
//
// Work decomposition. One CTA = (request, value head h, block of BV = 32
// value columns); 4 warps of 8 columns; inside a warp 4 column groups of 8
// lanes, each lane holding M = 2 columns x E = Dk/8 entries of S in
// registers. The Dk entries a lane owns are chunks of VEC contiguous
// elements, chunk i of lane r at Dk index VEC*(8i + r), so a warp's loads of
// a column are contiguous 16-byte vectors. Every reduction over Dk is a
// 3-level xor butterfly inside the 8-lane group (all lanes end with the same
// bits), with no shared memory and no atomics on data.
//
// Per token (one HBM-free step once S is in registers):
//   k^ = k / sqrt(|k|^2 + eps), q^ likewise (butterfly over the 8 lanes)
//   sk = S^T k^, sq = S^T q^ from the OLD S, kq = k^.q^
//   u  = beta (v - alpha sk),  o = scale (alpha sq + u kq)
//   S  = alpha S + k^ u^T
// which is the rule S <- alpha S; u = beta (v - S^T k^); S <- S + k^ u^T;
// o = scale S^T q^ with the decay folded into the two dot products, so S is
// read once and written once per token. All arithmetic uses explicit
// round-to-nearest intrinsics: the compiler cannot contract differently in
// the three kernels, which is what makes the one-page verify bit-identical to
// the slot layout.
#pragma once

#include "common.cuh"

namespace gdn {

enum RuleMode { MODE_SEQ = 0, MODE_VERIFY = 1, MODE_SLOTS = 2 };

constexpr int kRuleWarps = 4;
constexpr int kColsPerLane = 2;                         // M
constexpr int kBV = kRuleWarps * 4 * kColsPerLane;      // columns per CTA

template <int DK, class ST>
struct LaneMap {
  static constexpr int E = DK / 8;                      // entries per lane per column
  static constexpr int VEC0 = 16 / (int)sizeof(ST);
  static constexpr int VEC = (E < VEC0) ? E : VEC0;     // contiguous entries per chunk
  static constexpr int NI = E / VEC;                    // chunks
  __device__ static int idx(int r8, int i) { return VEC * (8 * i + r8); }
};

__device__ __forceinline__ float group8_sum(float v) {
  v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
  return v;
}

// One token's inputs for one lane.
template <int E>
struct TokenIn {
  float q[E], k[E];
  float v[kColsPerLane];
  float a, b;
};

template <int DK, class IO, class ST>
__device__ __forceinline__ void load_token(TokenIn<DK / 8>& in, const IO* row, const IO* a_ptr,
                                           const IO* b_ptr, int kh, int h, const Geom& G,
                                           const int* col, int r8) {
  using L = LaneMap<DK, ST>;
  const IO* qp = row + (size_t)kh * DK;
  const IO* kp = row + (size_t)G.Hk * DK + (size_t)kh * DK;
#pragma unroll
  for (int i = 0; i < L::NI; ++i) {
    load_f<IO, L::VEC>(qp + L::idx(r8, i), in.q + i * L::VEC);
    load_f<IO, L::VEC>(kp + L::idx(r8, i), in.k + i * L::VEC);
  }
  const IO* vp = row + 2 * (size_t)G.Hk * DK + (size_t)h * G.Dv;
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m) in.v[m] = to_f(vp[col[m]]);
  in.a = to_f(*a_ptr);
  in.b = to_f(*b_ptr);
}

// The step. S is updated in place when `update`; o receives the outputs of
// the lane's columns (identical on the 8 lanes of a group).
template <int E>
__device__ __forceinline__ void token_step(float (&S)[kColsPerLane][E], const TokenIn<E>& in,
                                           float alpha, float beta, float scale, float eps,
                                           bool update, float (&o)[kColsPerLane]) {
  float kk = 0.0f, qq = 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    kk = __fmaf_rn(in.k[e], in.k[e], kk);
    qq = __fmaf_rn(in.q[e], in.q[e], qq);
  }
  kk = group8_sum(kk);
  qq = group8_sum(qq);
  const float ik = rsqrtf(__fadd_rn(kk, eps));
  const float iq = rsqrtf(__fadd_rn(qq, eps));
  float kh[E], qh[E];
  float kq = 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    kh[e] = __fmul_rn(in.k[e], ik);
    qh[e] = __fmul_rn(in.q[e], iq);
    kq = __fmaf_rn(kh[e], qh[e], kq);
  }
  kq = group8_sum(kq);
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m) {
    float sk = 0.0f, sq = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      sk = __fmaf_rn(S[m][e], kh[e], sk);
      sq = __fmaf_rn(S[m][e], qh[e], sq);
    }
    sk = group8_sum(sk);
    sq = group8_sum(sq);
    const float u = __fmul_rn(beta, __fsub_rn(in.v[m], __fmul_rn(alpha, sk)));
    o[m] = __fmul_rn(scale, __fmaf_rn(u, kq, __fmul_rn(alpha, sq)));
    if (update) {
#pragma unroll
      for (int e = 0; e < E; ++e) S[m][e] = __fmaf_rn(kh[e], u, __fmul_rn(alpha, S[m][e]));
    }
  }
}

template <int DK, class ST>
__device__ __forceinline__ void load_state(float (&S)[kColsPerLane][DK / 8], const ST* base,
                                           const int* col, int r8) {
  using L = LaneMap<DK, ST>;
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m)
#pragma unroll
    for (int i = 0; i < L::NI; ++i)
      load_f<ST, L::VEC>(base + (size_t)col[m] * DK + L::idx(r8, i), &S[m][i * L::VEC]);
}

template <int DK, class ST>
__device__ __forceinline__ void store_state(ST* base, const float (&S)[kColsPerLane][DK / 8],
                                            const int* col, int r8) {
  using L = LaneMap<DK, ST>;
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m)
#pragma unroll
    for (int i = 0; i < L::NI; ++i)
      store_f<ST, L::VEC>(base + (size_t)col[m] * DK + L::idx(r8, i), &S[m][i * L::VEC]);
}

__device__ __forceinline__ void store_out(void* o, int out_f32, size_t off, float v) {
  if (out_f32) reinterpret_cast<float*>(o)[off] = v;
  else reinterpret_cast<bf16*>(o)[off] = __float2bfloat16_rn(v);
}

template <class IO, class ST, int DK, int MODE>
__global__ void __launch_bounds__(kRuleWarps * 32)
rule_kernel(Geom G, Batch B, Params P, SlotGeom SG, const IO* __restrict__ qkv,
            const IO* __restrict__ a_in, const IO* __restrict__ b_in, void* o, int out_f32,
            void* pages, int32_t* status) {
  constexpr int E = DK / 8;
  const int nCB = G.Dv / kBV;
  const int h = blockIdx.x / nCB;
  const int cb = blockIdx.x % nCB;
  const bool reporter = (blockIdx.x == 0 && threadIdx.x == 0);

  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  if (MODE == MODE_SEQ && q.spec) return;
  if (MODE == MODE_VERIFY && !q.spec) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cg = lane >> 3, r8 = lane & 7;
  int col[kColsPerLane];
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m) col[m] = cb * kBV + warp * 8 + m * 4 + cg;
  const int kh = (int)(((long long)h * G.Hk) / G.Hv);
  const float scale = P.scale;

  float S[kColsPerLane][E];
  float out[kColsPerLane];
  TokenIn<E> in;

  if constexpr (MODE == MODE_SEQ) {
    char* pg = page_ptr(G, pages, q.page);
    uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
    if (!q.fresh && flag_width(*flagp) != 0) {
      if (reporter) report(status, GDN_DEV_RECORD_OPEN);
      return;
    }
    ST* Sb = reinterpret_cast<ST*>(pg + G.state_off) + (size_t)h * G.Dv * DK;
    if (q.fresh) {
#pragma unroll
      for (int m = 0; m < kColsPerLane; ++m)
#pragma unroll
        for (int e = 0; e < E; ++e) S[m][e] = 0.0f;
    } else {
      if (q.len == 0) return;  // nothing to do
      load_state<DK, ST>(S, Sb, col, r8);
    }
    if (q.len > 0) {
      const IO* row0 = qkv + (size_t)q.start * G.C;
      load_token<DK, IO, ST>(in, row0, a_in + (size_t)q.start * G.Hv + h,
                             b_in + (size_t)q.start * G.Hv + h, kh, h, G, col, r8);
    }
    for (int t = 0; t < q.len; ++t) {
      const TokenIn<E> cur = in;
      if (t + 1 < q.len) {
        const size_t rn = (size_t)q.start + t + 1;
        load_token<DK, IO, ST>(in, qkv + rn * G.C, a_in + rn * G.Hv + h, b_in + rn * G.Hv + h, kh,
                               h, G, col, r8);
      }
      float alpha, beta;
      gates(P, h, cur.a, cur.b, alpha, beta);
      token_step<E>(S, cur, alpha, beta, scale, P.eps, true, out);
      if (r8 == 0) {
        const size_t off = ((size_t)(q.start + t) * G.Hv + h) * G.Dv;
#pragma unroll
        for (int m = 0; m < kColsPerLane; ++m) store_out(o, out_f32, off + col[m], out[m]);
      }
    }
    store_state<DK, ST>(Sb, S, col, r8);
    if (q.fresh && blockIdx.x == 0 && threadIdx.x == 0) *flagp = 0u;  // empty record
  } else if constexpr (MODE == MODE_VERIFY) {
    char* pg = page_ptr(G, pages, q.page);
    uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
    const uint32_t flag = *reinterpret_cast<volatile uint32_t*>(flagp);
    SpecState ss = spec_state(G, B, q, flag);
    if (q.fresh) ss.err = GDN_DEV_BAD_FLAG;
    if (ss.err) {
      if (reporter) report(status, ss.err);
      return;
    }
    ST* Sb = reinterpret_cast<ST*>(pg + G.state_off) + (size_t)h * G.Dv * DK;
    const IO* rec = reinterpret_cast<const IO*>(pg + G.record_off);
    load_state<DK, ST>(S, Sb, col, r8);
    if (ss.width > 0) {
      // replay rows 0..a of the live slot, then store the checkpoint
      const IO* slot = rec + (size_t)ss.live * G.Kc * G.rec_row;
      for (int i = 0; i <= ss.accepted; ++i) {
        const IO* row = slot + (size_t)i * G.rec_row;
        load_token<DK, IO, ST>(in, row, row + G.C + h, row + G.C + G.Hv + h, kh, h, G, col, r8);
        float alpha, beta;
        gates(P, h, in.a, in.b, alpha, beta);
        token_step<E>(S, in, alpha, beta, scale, P.eps, true, out);
      }
      store_state<DK, ST>(Sb, S, col, r8);
      // continue from exactly what was stored (a bf16 page rounds here)
#pragma unroll
      for (int m = 0; m < kColsPerLane; ++m)
#pragma unroll
        for (int e = 0; e < E; ++e) S[m][e] = through<ST>(S[m][e]);
    }
    // this step's candidates: outputs only, no per-candidate state
    for (int t = 0; t < q.len; ++t) {
      const size_t rn = (size_t)q.start + t;
      load_token<DK, IO, ST>(in, qkv + rn * G.C, a_in + rn * G.Hv + h, b_in + rn * G.Hv + h, kh,
                             h, G, col, r8);
      float alpha, beta;
      gates(P, h, in.a, in.b, alpha, beta);
      token_step<E>(S, in, alpha, beta, scale, P.eps, t + 1 < q.len, out);
      if (r8 == 0) {
        const size_t off = (rn * G.Hv + h) * G.Dv;
#pragma unroll
        for (int m = 0; m < kColsPerLane; ++m) store_out(o, out_f32, off + col[m], out[m]);
      }
    }
    // the candidates' gates go next to their conv'd rows in the other slot
    if (cb == 0 && threadIdx.x < q.len) {
      IO* row = const_cast<IO*>(rec) + ((size_t)(1 - ss.live) * G.Kc + threadIdx.x) * G.rec_row;
      const size_t rn = (size_t)q.start + threadIdx.x;
      row[G.C + h] = a_in[rn * G.Hv + h];
      row[G.C + G.Hv + h] = b_in[rn * G.Hv + h];
    }
    // last CTA of this request publishes the new flag word
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const uint32_t total = (uint32_t)(G.Hv * nCB);
      const uint32_t old = atomicAdd(flagp, 256u);
      if ((old >> 8) == total - 1) {
        __threadfence();
        const int live = (q.len > 0) ? 1 - ss.live : ss.live;
        atomicExch(flagp, make_flag(live, 1 - ss.parity, q.len));
      }
    }
  } else {  // MODE_SLOTS
    const int src = B.n_accepted ? B.n_accepted[q.r] : -1;
    if (src < 0 || src >= G.Kc) {
      if (reporter) report(status, GDN_DEV_BAD_ACCEPTED);
      return;
    }
    if (q.len > G.Kc) {
      if (reporter) report(status, GDN_DEV_TOO_MANY_CANDIDATES);
      return;
    }
    char* pool = reinterpret_cast<char*>(pages) + (size_t)q.page * SG.pool_bytes;
    auto slot_state = [&](int i) {
      return reinterpret_cast<ST*>(pool + (size_t)i * SG.slot_bytes + SG.state_off) +
             (size_t)h * G.Dv * DK;
    };
    load_state<DK, ST>(S, slot_state(src), col, r8);
    for (int t = 0; t < q.len; ++t) {
      const size_t rn = (size_t)q.start + t;
      load_token<DK, IO, ST>(in, qkv + rn * G.C, a_in + rn * G.Hv + h, b_in + rn * G.Hv + h, kh,
                             h, G, col, r8);
      float alpha, beta;
      gates(P, h, in.a, in.b, alpha, beta);
      token_step<E>(S, in, alpha, beta, scale, P.eps, true, out);
      if (r8 == 0) {
        const size_t off = (rn * G.Hv + h) * G.Dv;
#pragma unroll
        for (int m = 0; m < kColsPerLane; ++m) store_out(o, out_f32, off + col[m], out[m]);
      }
      store_state<DK, ST>(slot_state(t), S, col, r8);
    }
  }
}

template <int DK>
cudaError_t launch_rule_dk(int mode, const Geom& G, const Batch& B, const Params& P,
                           const SlotGeom& SG, int io_bf16, int state_bf16, int out_f32,
                           const void* qkv, const void* a, const void* b, void* o, void* pages,
                           int32_t* status, cudaStream_t stream) {
  dim3 grid(G.Hv * (G.Dv / kBV), B.R);
  dim3 block(kRuleWarps * 32);
#define GDN_RULE_LAUNCH(IO, ST, MODE)                                                         \
  rule_kernel<IO, ST, DK, MODE><<<grid, block, 0, stream>>>(                                  \
      G, B, P, SG, static_cast<const IO*>(qkv), static_cast<const IO*>(a),                   \
      static_cast<const IO*>(b), o, out_f32, pages, status)
#define GDN_RULE_MODES(IO, ST)                       \
  if (mode == MODE_SEQ) GDN_RULE_LAUNCH(IO, ST, MODE_SEQ);          \
  else if (mode == MODE_VERIFY) GDN_RULE_LAUNCH(IO, ST, MODE_VERIFY); \
  else GDN_RULE_LAUNCH(IO, ST, MODE_SLOTS);
  if (io_bf16) {
    if (state_bf16) { GDN_RULE_MODES(bf16, bf16) } else { GDN_RULE_MODES(bf16, float) }
  } else {
    if (state_bf16) { GDN_RULE_MODES(float, bf16) } else { GDN_RULE_MODES(float, float) }
  }
#undef GDN_RULE_MODES
#undef GDN_RULE_LAUNCH
  return cudaGetLastError();
}

}  // namespace gdn
