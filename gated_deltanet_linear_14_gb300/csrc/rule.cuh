// Token-by-token gated delta rule (gdn_seq), plus the staging and token step
// that the fused decode (decode.cu) runs too (sm_103a).
//
// r9700-stack v0.2.3, section 1 (r9k_gdn_seq: any number of tokens, the state
// in registers, the batch's own rows); vllm.cpp PR #155 (q/k L2 norm and
// gates fused per token).
//
// Work decomposition. One CTA = (request, value head h, block of BV = 32
// value columns); 4 warps of 8 columns; inside a warp 4 column groups of 8
// lanes; a lane holds M = 2 adjacent columns x E = Dk/8 entries of S in
// registers (as float2 pairs for the packed f32x2 FMA pipe). The Dk entries a
// lane owns are chunks of VEC contiguous elements, chunk i of lane r at Dk
// index VEC*(8i + r), so a warp's accesses to a column are contiguous.
//
// Tokens are processed in chunks of TC. For each chunk the CTA stages, once,
// in shared memory: q^ and k^ normalised in fp32, the CTA's 32 values of v,
// and per token (alpha = e^g, beta, q^.k^). The raw rows of the next chunk
// are fetched into registers while the current chunk runs. The per-token
// step of a lane is then only
//   sk = S^T k^, sq = S^T q^ (old S, f32x2 partial sums, one 8-lane
//   transpose-reduce of the four sums), u = beta (v - alpha sk),
//   o = scale (alpha sq + u q^.k^), S = alpha S + k^ u^T (f32x2)
// which is the rule S <- alpha S; u = beta (v - S^T k^); S <- S + k^ u^T;
// o = scale S^T q^ with the decay folded into the dot products, so S is read
// once and written once per token. All arithmetic is explicit
// round-to-nearest intrinsics, so the fused decode, which runs the same
// staging and step, is bit-identical to gdn_conv followed by gdn_seq.
#pragma once

#include "common.cuh"

namespace gdn {

constexpr int kRuleWarps = 4;
constexpr int kRuleThreads = kRuleWarps * 32;
constexpr int kColsPerLane = 2;                         // M (adjacent columns)
constexpr int kBV = kRuleWarps * 4 * kColsPerLane;      // columns per CTA
constexpr int kTC = 16;                                 // tokens per staged chunk

template <int DK, class ST>
struct LaneMap {
  static constexpr int E = DK / 8;                      // entries per lane per column
  static constexpr int VEC0 = 16 / (int)sizeof(ST);
  static constexpr int VEC = (E < VEC0) ? E : VEC0;     // contiguous entries per chunk
  static constexpr int NI = E / VEC;                    // chunks
  __device__ static int idx(int r8, int i) { return VEC * (8 * i + r8); }
};

// Where Dk entry d of a staged q^ or k^ row sits in shared memory. When a
// lane's state entries come in runs of 8 (bf16 state: VEC = 8), the row is
// permuted by 16-byte pieces so that the first halves of the 8 lanes' runs
// are contiguous, then the second halves: each 16-byte load of a warp then
// reads one 128-byte line instead of two. With VEC = 4 rows are in order.
template <int DK, class ST>
__device__ __forceinline__ int stage_pos(int d) {
  if constexpr (LaneMap<DK, ST>::VEC == 8) {
    const int m = d >> 2;  // 16-byte piece: m = 2 (8 i + r8) + half
    return ((((m >> 4) << 4) | ((m & 1) << 3) | ((m >> 1) & 7)) << 2) | (d & 3);
  } else {
    return d;
  }
}

template <int DK>
struct Stage {
  float q[kTC][DK];       // q^ (fp32, normalised)
  float k[kTC][DK];       // k^
  float v[kTC][kBV];      // the CTA's value columns
  float4 sc[kTC];         // alpha, beta, q^.k^, unused
};

// Where a chunk's rows come from: packed step rows or a page record.
template <class IO>
struct RowSrc {
  const IO* rows;         // row 0 of the run
  size_t row_stride;      // elements between rows
  const IO* a;            // a of row 0 (head h)
  const IO* b;
  size_t ab_stride;
};

// N elements of T held raw (packed) in registers until they are used.
template <class T, int N>
struct RawVec {
  static constexpr int BYTES = N * (int)sizeof(T);
  static_assert(BYTES % 8 == 0, "raw vectors are whole 8-byte words");
  uint32_t w[BYTES / 4];
  __device__ __forceinline__ void load(const T* p) {
    if constexpr (BYTES >= 16) {
#pragma unroll
      for (int v = 0; v < BYTES / 16; ++v) {
        const uint4 u = reinterpret_cast<const uint4*>(p)[v];
        w[4 * v] = u.x; w[4 * v + 1] = u.y; w[4 * v + 2] = u.z; w[4 * v + 3] = u.w;
      }
    } else {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      w[0] = u.x; w[1] = u.y;
    }
  }
  __device__ __forceinline__ float get(int i) const {
    if constexpr (sizeof(T) == 4) {
      return __uint_as_float(w[i]);
    } else {
      const uint32_t x = w[i >> 1];
      return __uint_as_float((i & 1) ? (x & 0xFFFF0000u) : (x << 16));
    }
  }
};

// The raw inputs one thread fetches for one token of a chunk: entries
// [E*p, E*p + E) of q and k, value columns [4p, 4p+4) of the CTA's block.
template <int DK, class IO>
struct Fetch {
  RawVec<IO, DK / 8> q, k;
  RawVec<IO, 4> v;
  float a, b;
};

template <int DK, class IO>
__device__ __forceinline__ void fetch(Fetch<DK, IO>& f, const RowSrc<IO>& src, int t, int n_t,
                                      int p, int kh, int h, int cb, const Geom& G) {
  constexpr int PE = DK / 8;
  if (t >= n_t) return;
  const IO* row = src.rows + (size_t)t * src.row_stride;
  f.q.load(row + (size_t)kh * DK + PE * p);
  f.k.load(row + (size_t)G.Hk * DK + (size_t)kh * DK + PE * p);
  f.v.load(row + 2 * (size_t)G.Hk * DK + (size_t)h * G.Dv + cb * kBV + 4 * p);
  if (p == 0) {
    f.a = to_f(src.a[(size_t)t * src.ab_stride]);
    f.b = to_f(src.b[(size_t)t * src.ab_stride]);
  }
}

// q^ and k^ of one token from its raw parts, 8 threads per token (thread p
// holds entries [PE p, PE p + PE)): 8-lane butterfly sums of q.q, k.k and
// q.k, then 1/sqrt(x.x + eps). Writes this thread's parts of q^, k^ (entries
// d0 .. d0 + PE - 1 of the staged rows, at stage_pos) and returns q^.k^ (the same value in all 8 threads). Every kernel that stages
// rows for the token step normalises through here, so they all see
// bit-identical q^, k^.
template <int DK, class IO, class ST>
__device__ __forceinline__ float publish_qk(float* qrow, float* krow, int d0,
                                            const RawVec<IO, DK / 8>& rq,
                                            const RawVec<IO, DK / 8>& rk, const Params& P) {
  constexpr int PE = DK / 8;
  float fq[PE], fk[PE];
#pragma unroll
  for (int e = 0; e < PE; ++e) {
    fq[e] = rq.get(e);
    fk[e] = rk.get(e);
  }
  float qq = 0.0f, kk = 0.0f, qk = 0.0f;
#pragma unroll
  for (int e = 0; e < PE; ++e) {
    qq = __fmaf_rn(fq[e], fq[e], qq);
    kk = __fmaf_rn(fk[e], fk[e], kk);
    qk = __fmaf_rn(fq[e], fk[e], qk);
  }
  const unsigned grp = 0xFFu << (threadIdx.x & 24);
#pragma unroll
  for (int d = 1; d < 8; d <<= 1) {
    qq = __fadd_rn(qq, __shfl_xor_sync(grp, qq, d));
    kk = __fadd_rn(kk, __shfl_xor_sync(grp, kk, d));
    qk = __fadd_rn(qk, __shfl_xor_sync(grp, qk, d));
  }
  const float iq = rsqrtf(__fadd_rn(qq, P.eps));
  const float ik = rsqrtf(__fadd_rn(kk, P.eps));
#pragma unroll
  for (int e = 0; e < PE; e += 4) {
    *reinterpret_cast<float4*>(&qrow[stage_pos<DK, ST>(d0 + e)]) =
        make_float4(__fmul_rn(fq[e], iq), __fmul_rn(fq[e + 1], iq), __fmul_rn(fq[e + 2], iq),
                    __fmul_rn(fq[e + 3], iq));
    *reinterpret_cast<float4*>(&krow[stage_pos<DK, ST>(d0 + e)]) =
        make_float4(__fmul_rn(fk[e], ik), __fmul_rn(fk[e + 1], ik), __fmul_rn(fk[e + 2], ik),
                    __fmul_rn(fk[e + 3], ik));
  }
  return __fmul_rn(__fmul_rn(qk, iq), ik);
}

// Normalise and publish one fetched token (8 threads per token).
template <int DK, class IO, class ST>
__device__ __forceinline__ void publish(Stage<DK>& st, const Fetch<DK, IO>& f, int t, int n_t,
                                        int p, int h, const Params& P) {
  constexpr int PE = DK / 8;
  if (t >= n_t) return;  // whole 8-lane groups take this branch together
  const float kq = publish_qk<DK, IO, ST>(st.q[t], st.k[t], PE * p, f.q, f.k, P);
  *reinterpret_cast<float4*>(&st.v[t][4 * p]) =
      make_float4(f.v.get(0), f.v.get(1), f.v.get(2), f.v.get(3));
  if (p == 0) {
    float alpha, beta;
    gates(P, h, f.a, f.b, alpha, beta);
    st.sc[t] = make_float4(alpha, beta, kq, 0.0f);
  }
}

// The state of a lane: M columns x E entries as float2 pairs.
template <int E>
struct LaneState {
  float2 s[kColsPerLane][E / 2];
};

// One token for one lane. Returns this lane's output column value in o (the
// lanes with (r8 & 3) == 0 own column m = r8 >> 2 of their group).
template <int DK, class ST>
__device__ __forceinline__ float token_step(LaneState<DK / 8>& S, const Stage<DK>& st, int t, int r8,
                                            int vcol, float scale, bool update);

// The step on explicit shared-memory rows: q^ and k^ (DK floats each), the
// CTA's value block (vcol indexes it) and (alpha, beta, q^.k^).
template <int DK, class ST>
__device__ __forceinline__ float token_step_rows(LaneState<DK / 8>& S, const float* qrow,
                                                 const float* krow, const float* vrow, float4 sc,
                                                 int r8, int vcol, float scale, bool update) {
  using L = LaneMap<DK, ST>;
  constexpr int E = DK / 8;
  float2 q2[E / 2], k2[E / 2];
#pragma unroll
  for (int i = 0; i < L::NI; ++i) {
#pragma unroll
    for (int e = 0; e < L::VEC; e += 4) {
      const float4 qv = *reinterpret_cast<const float4*>(&qrow[stage_pos<DK, ST>(L::idx(r8, i) + e)]);
      const float4 kv = *reinterpret_cast<const float4*>(&krow[stage_pos<DK, ST>(L::idx(r8, i) + e)]);
      q2[(i * L::VEC + e) / 2] = make_float2(qv.x, qv.y);
      q2[(i * L::VEC + e) / 2 + 1] = make_float2(qv.z, qv.w);
      k2[(i * L::VEC + e) / 2] = make_float2(kv.x, kv.y);
      k2[(i * L::VEC + e) / 2 + 1] = make_float2(kv.z, kv.w);
    }
  }
  const float alpha = sc.x, beta = sc.y, kq = sc.z;
  const float2 vv = *reinterpret_cast<const float2*>(&vrow[vcol]);

  float2 ak0 = make_float2(0.f, 0.f), aq0 = ak0, ak1 = ak0, aq1 = ak0;
#pragma unroll
  for (int j = 0; j < E / 2; ++j) {
    ak0 = __ffma2_rn(S.s[0][j], k2[j], ak0);
    aq0 = __ffma2_rn(S.s[0][j], q2[j], aq0);
    ak1 = __ffma2_rn(S.s[1][j], k2[j], ak1);
    aq1 = __ffma2_rn(S.s[1][j], q2[j], aq1);
  }
  // the four partial sums of this lane
  const float v0 = __fadd_rn(ak0.x, ak0.y), v1 = __fadd_rn(aq0.x, aq0.y);
  const float v2 = __fadd_rn(ak1.x, ak1.y), v3 = __fadd_rn(aq1.x, aq1.y);
  // transpose-reduce over the 8 lanes of the group: afterwards lanes with
  // bit 2 = m hold the full sums of column m (sk if bit 1 = 0, sq if 1)
  const bool b2 = (r8 & 4) != 0, b1 = (r8 & 2) != 0;
  float a0 = b2 ? v2 : v0, a1 = b2 ? v3 : v1;
  const float s0 = b2 ? v0 : v2, s1 = b2 ? v1 : v3;
  a0 = __fadd_rn(a0, __shfl_xor_sync(0xffffffffu, s0, 4));
  a1 = __fadd_rn(a1, __shfl_xor_sync(0xffffffffu, s1, 4));
  float kept = b1 ? a1 : a0;
  const float sent = b1 ? a0 : a1;
  kept = __fadd_rn(kept, __shfl_xor_sync(0xffffffffu, sent, 2));
  kept = __fadd_rn(kept, __shfl_xor_sync(0xffffffffu, kept, 1));
  const float other = __shfl_xor_sync(0xffffffffu, kept, 2);
  const float sk = b1 ? other : kept;
  const float sq = b1 ? kept : other;
  const float vm = b2 ? vv.y : vv.x;
  const float u = __fmul_rn(beta, __fsub_rn(vm, __fmul_rn(alpha, sk)));
  const float o = __fmul_rn(scale, __fmaf_rn(u, kq, __fmul_rn(alpha, sq)));
  if (update) {
    const float u_x = __shfl_xor_sync(0xffffffffu, u, 4);
    const float u0 = b2 ? u_x : u, u1 = b2 ? u : u_x;
    const float2 al = make_float2(alpha, alpha);
    const float2 uu0 = make_float2(u0, u0), uu1 = make_float2(u1, u1);
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
      S.s[0][j] = __ffma2_rn(k2[j], uu0, __fmul2_rn(al, S.s[0][j]));
      S.s[1][j] = __ffma2_rn(k2[j], uu1, __fmul2_rn(al, S.s[1][j]));
    }
  }
  return o;
}

template <int DK, class ST>
__device__ __forceinline__ float token_step(LaneState<DK / 8>& S, const Stage<DK>& st, int t, int r8,
                                            int vcol, float scale, bool update) {
  return token_step_rows<DK, ST>(S, st.q[t], st.k[t], st.v[t], st.sc[t], r8, vcol, scale, update);
}

template <int DK, class ST>
__device__ __forceinline__ void load_state(LaneState<DK / 8>& S, const ST* base, const int* col,
                                           int r8) {
  using L = LaneMap<DK, ST>;
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m)
#pragma unroll
    for (int i = 0; i < L::NI; ++i)
      load_f<ST, L::VEC>(base + (size_t)col[m] * DK + L::idx(r8, i),
                         reinterpret_cast<float*>(&S.s[m][0]) + i * L::VEC);
}

template <int DK, class ST>
__device__ __forceinline__ void store_state(ST* base, const LaneState<DK / 8>& S, const int* col,
                                            int r8) {
  using L = LaneMap<DK, ST>;
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m)
#pragma unroll
    for (int i = 0; i < L::NI; ++i)
      store_f<ST, L::VEC>(base + (size_t)col[m] * DK + L::idx(r8, i),
                          reinterpret_cast<const float*>(&S.s[m][0]) + i * L::VEC);
}

template <int E>
__device__ __forceinline__ void zero_state(LaneState<E>& S) {
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m)
#pragma unroll
    for (int j = 0; j < E / 2; ++j) S.s[m][j] = make_float2(0.f, 0.f);
}

// Run n rows from `src` through the rule. Outputs go to o rows starting at
// out_row (nullptr o: no outputs). The state is updated for every row but
// the last when !update_last. `keep` is called after each row with the row
// index (the slot layout stores the state there).
template <int DK, class IO, class ST, class AfterRow>
__device__ __forceinline__ void run_rows(LaneState<DK / 8>& S, Stage<DK>& st, const RowSrc<IO>& src,
                                         int n, void* o, int out_f32, size_t out_row, int h,
                                         int cb, int kh, const Geom& G, const Params& P,
                                         bool update_last, AfterRow after_row) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, cg = lane >> 3, r8 = lane & 7;
  const int vcol = warp * 8 + cg * 2;                   // first of the lane's 2 columns
  const int ft = tid >> 3, fp = tid & 7;                // fetch: token, part
  Fetch<DK, IO> f;
  fetch<DK, IO>(f, src, ft, n, fp, kh, h, cb, G);
  for (int c0 = 0; c0 < n; c0 += kTC) {
    const int n_t = min(kTC, n - c0);
    __syncthreads();                                    // previous chunk fully read
    publish<DK, IO, ST>(st, f, ft, n_t, fp, h, P);
    __syncthreads();
    if (c0 + kTC < n) {                                 // prefetch the next chunk
      RowSrc<IO> nx = src;
      nx.rows += (size_t)(c0 + kTC) * src.row_stride;
      nx.a += (size_t)(c0 + kTC) * src.ab_stride;
      nx.b += (size_t)(c0 + kTC) * src.ab_stride;
      fetch<DK, IO>(f, nx, ft, n - c0 - kTC, fp, kh, h, cb, G);
    }
    for (int t = 0; t < n_t; ++t) {
      const bool upd = update_last || (c0 + t + 1 < n);
      const float ov = token_step<DK, ST>(S, st, t, r8, vcol, P.scale, upd);
      if (o != nullptr && (r8 & 3) == 0) {
        const size_t off = ((out_row + c0 + t) * G.Hv + h) * G.Dv + cb * kBV + vcol + (r8 >> 2);
        store_out(o, out_f32, off, ov);
      }
      after_row(c0 + t);
    }
  }
}

struct NoAfter {
  __device__ void operator()(int) const {}
};

// 4 CTAs per SM keep the token-by-token kernel near 120 registers (left free,
// the compiler went past 150 and a long prefill's per-token chain measured a
// quarter slower).
template <class IO, class ST, int DK>
__global__ void __launch_bounds__(kRuleThreads, 4)
rule_kernel(Geom G, Batch B, Params P, const IO* __restrict__ qkv, const IO* __restrict__ a_in,
            const IO* __restrict__ b_in, void* o, int out_f32, void* pages, int32_t* status) {
  pdl_begin();
  constexpr int E = DK / 8;
  __shared__ __align__(16) Stage<DK> st;
  const int nCB = G.Dv / kBV;
  const int h = blockIdx.x / nCB;
  const int cb = blockIdx.x % nCB;
  const bool reporter = (blockIdx.x == 0 && threadIdx.x == 0);

  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  if (q.spec) return;
  if (q.len < B.min_len || q.len > B.max_len) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cg = lane >> 3, r8 = lane & 7;
  int col[kColsPerLane];
#pragma unroll
  for (int m = 0; m < kColsPerLane; ++m) col[m] = cb * kBV + warp * 8 + cg * 2 + m;
  const int kh = (int)(((long long)h * G.Hk) / G.Hv);

  LaneState<E> S;
  RowSrc<IO> rows_in;
  rows_in.rows = qkv + (size_t)q.start * G.C;
  rows_in.row_stride = G.C;
  rows_in.a = a_in + (size_t)q.start * G.Hv + h;
  rows_in.b = b_in + (size_t)q.start * G.Hv + h;
  rows_in.ab_stride = G.Hv;

  char* pg = page_ptr(G, pages, q.page);
  uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
  if (!q.fresh && q.len == 0) return;  // nothing to do
  ST* Sb = reinterpret_cast<ST*>(pg + G.state_off) + (size_t)h * G.Dv * DK;
  // the state load is issued before the flag check (one round trip, not
  // two); a refused request only discards it
  if (q.fresh) zero_state<E>(S);
  else load_state<DK, ST>(S, Sb, col, r8);
  if (!q.fresh && flag_width(*flagp) != 0) {
    if (reporter) report(status, GDN_DEV_RECORD_OPEN);
    return;
  }
  run_rows<DK, IO, ST>(S, st, rows_in, q.len, o, out_f32, (size_t)q.start, h, cb, kh, G, P, true,
                       NoAfter());
  store_state<DK, ST>(Sb, S, col, r8);
  if (q.fresh && blockIdx.x == 0 && threadIdx.x == 0) *flagp = 0u;  // empty record
}

template <int DK>
cudaError_t launch_rule_dk(const Geom& G, const Batch& B, const Params& P, int io_bf16,
                           int state_bf16, int out_f32, const void* qkv, const void* a,
                           const void* b, void* o, void* pages, int32_t* status,
                           cudaStream_t stream) {
  dim3 grid(G.Hv * (G.Dv / kBV), B.R);
  dim3 block(kRuleThreads);
#define GDN_RULE_LAUNCH(IO, ST)                                                              \
  return launch_pdl(rule_kernel<IO, ST, DK>, grid, block, 0, stream, G, B, P,               \
                    static_cast<const IO*>(qkv), static_cast<const IO*>(a),                 \
                    static_cast<const IO*>(b), o, out_f32, pages, status)
  if (io_bf16) {
    if (state_bf16) GDN_RULE_LAUNCH(bf16, bf16); else GDN_RULE_LAUNCH(bf16, float);
  } else {
    if (state_bf16) GDN_RULE_LAUNCH(float, bf16); else GDN_RULE_LAUNCH(float, float);
  }
#undef GDN_RULE_LAUNCH
}

}  // namespace gdn
