// Device-side helpers shared by the GDN kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

typedef __nv_bfloat16 bf16;

// ------------------------------------------------------------------ layout

// Everything a kernel needs to address one layer's rows and pages.
struct Geom {
  int Hk, Hv, Dk, Dv, W, Kc;
  int C;              // 2*Hk*Dk + Hv*Dv
  int rec_row;        // record row stride in elements (16-byte padded)
  size_t page_bytes, window_off, state_off, record_off, flag_off;
  size_t rcoef_off;   // the record's run-coefficient blocks ([2][Hv], kRunCoefBytes each)
  size_t ru_off;      // the record's u per value column ([Hv][Kc][Dv] fp32)
};

// Run coefficients of one value head for the rows of one record slot: G_t /
// |k_t|, G_t / |q_t|, G_t, R[t][s] / |k_s|, M = (I - L)^-1 diag(beta) and
// N = B M, fp32, 8 + 8 + 8 + 64 + 64 + 64 values (see spec.cuh). The item
// kernel reads the candidates' from here; the next step's replay reads G and
// R/|k| of the same rows.
constexpr size_t kRunCoefFloats = 8 + 8 + 8 + 64 + 64 + 64;
constexpr size_t kRunCoefBytes = kRunCoefFloats * 4;

struct Batch {
  int R, num_rows, max_rows, num_pages;
  const int32_t* row_start;
  const int32_t* row_len;
  const int32_t* page;
  const uint32_t* flags;
  const int32_t* n_accepted;
  const int32_t* order;
  // plain requests with row counts outside [min_len, max_len] are left to
  // another launch (the prefill dispatch splits a batch this way)
  int min_len, max_len;
};

// Slot pool geometry of the slot-per-candidate layout.
struct SlotGeom {
  size_t pool_bytes, slot_bytes, state_off, window_off;
};

struct Params {
  const float* A_log;
  const float* dt_bias;
  const float* conv_bias;
  float scale;
  float eps;
  int gate_mode;
};

// Flag word: bit 0 live slot, bit 1 parity, bits 2..7 width, 8..31 counter.
__device__ __forceinline__ int flag_live(uint32_t f) { return (int)(f & 1u); }
__device__ __forceinline__ int flag_parity(uint32_t f) { return (int)((f >> 1) & 1u); }
__device__ __forceinline__ int flag_width(uint32_t f) { return (int)((f >> 2) & 63u); }
__device__ __forceinline__ uint32_t make_flag(int live, int parity, int width) {
  return (uint32_t)live | ((uint32_t)parity << 1) | ((uint32_t)width << 2);
}

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Per-request facts every kernel checks the same way.
struct Req {
  int r, start, len, page;
  uint32_t flags;
  bool fresh, spec;
  int err;  // 0 or a gdn_status device code
};

__device__ __forceinline__ Req load_req(const Batch& B, int slot) {
  Req q;
  q.r = B.order ? B.order[slot] : slot;
  q.err = 0;
  if (q.r < 0 || q.r >= B.R) {
    q.err = GDN_DEV_BAD_ROWS;
    q.r = 0;
    q.start = q.len = q.page = 0;
    q.flags = 0;
    q.fresh = q.spec = false;
    return q;
  }
  q.start = B.row_start[q.r];
  q.len = B.row_len[q.r];
  q.page = B.page[q.r];
  q.flags = B.flags[q.r];
  q.fresh = (q.flags & GDN_REQ_FRESH) != 0;
  q.spec = (q.flags & GDN_REQ_SPEC) != 0;
  if (q.page < 0 || q.page >= B.num_pages) q.err = GDN_DEV_BAD_PAGE;
  else if (q.start < 0 || q.len < 0 || q.len > B.max_rows ||
           (long long)q.start + q.len > (long long)B.num_rows)
    q.err = GDN_DEV_BAD_ROWS;
  return q;
}

__device__ __forceinline__ char* page_ptr(const Geom& G, void* pages, int p) {
  return reinterpret_cast<char*>(pages) + (size_t)p * G.page_bytes;
}

// Speculative request facts read from the page flag (validated).
struct SpecState {
  int live, parity, width, accepted;  // accepted = -1 when nothing to replay
  int err;
};

// As spec_state, with the request's accepted count already loaded (-1 when
// the batch has none).
__device__ __forceinline__ SpecState spec_state_acc(const Geom& G, const Req& q, uint32_t flag,
                                                    int accepted) {
  SpecState s;
  s.live = flag_live(flag);
  s.parity = flag_parity(flag);
  s.width = flag_width(flag);
  s.accepted = -1;
  s.err = 0;
  const int want = (q.flags & GDN_REQ_PARITY) ? 1 : 0;
  if (s.width > G.Kc) s.err = GDN_DEV_BAD_FLAG;
  else if (s.parity != want) s.err = GDN_DEV_STALE_STEP;
  else if (q.len > G.Kc) s.err = GDN_DEV_TOO_MANY_CANDIDATES;
  else if (s.width > 0) {
    if (accepted < 0 || accepted >= s.width) s.err = GDN_DEV_BAD_ACCEPTED;
    else s.accepted = accepted;
  }
  return s;
}

__device__ __forceinline__ SpecState spec_state(const Geom& G, const Batch& B, const Req& q,
                                                uint32_t flag) {
  SpecState s;
  s.live = flag_live(flag);
  s.parity = flag_parity(flag);
  s.width = flag_width(flag);
  s.accepted = -1;
  s.err = 0;
  const int want = (q.flags & GDN_REQ_PARITY) ? 1 : 0;
  if (s.width > G.Kc) s.err = GDN_DEV_BAD_FLAG;
  else if (s.parity != want) s.err = GDN_DEV_STALE_STEP;
  else if (q.len > G.Kc) s.err = GDN_DEV_TOO_MANY_CANDIDATES;
  else if (s.width > 0) {
    const int a = B.n_accepted ? B.n_accepted[q.r] : -1;
    if (a < 0 || a >= s.width) s.err = GDN_DEV_BAD_ACCEPTED;
    else s.accepted = a;
  }
  return s;
}

// ------------------------------------------------------------ dtype access

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <class T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// Load N consecutive elements (N * sizeof(T) a multiple of 8 bytes, pointer
// aligned to min(16, N * sizeof(T))) into fp32 registers.
template <class T, int N>
__device__ __forceinline__ void load_f(const T* p, float* out) {
  constexpr int BYTES = N * (int)sizeof(T);
  static_assert(BYTES % 8 == 0, "vector load of at least 8 bytes");
  if constexpr (BYTES >= 16) {
#pragma unroll
    for (int v = 0; v < BYTES / 16; ++v) {
      uint4 u = reinterpret_cast<const uint4*>(p)[v];
      const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int i = 0; i < 16 / (int)sizeof(T); ++i) out[v * (16 / sizeof(T)) + i] = to_f(e[i]);
    }
  } else {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = to_f(e[i]);
  }
}

template <class T, int N>
__device__ __forceinline__ void store_f(T* p, const float* in) {
  constexpr int BYTES = N * (int)sizeof(T);
  static_assert(BYTES % 8 == 0, "vector store of at least 8 bytes");
  if constexpr (sizeof(T) == 2) {
    // bf16: two values per paired round-to-nearest conversion
    uint32_t w[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    if constexpr (BYTES >= 16) {
#pragma unroll
      for (int v = 0; v < BYTES / 16; ++v)
        reinterpret_cast<uint4*>(p)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
    } else {
      *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
    }
  } else if constexpr (BYTES >= 16) {
#pragma unroll
    for (int v = 0; v < BYTES / 16; ++v) {
      uint4 u;
      T* e = reinterpret_cast<T*>(&u);
#pragma unroll
      for (int i = 0; i < 16 / (int)sizeof(T); ++i) e[i] = from_f<T>(in[v * (16 / sizeof(T)) + i]);
      reinterpret_cast<uint4*>(p)[v] = u;
    }
  } else {
    uint2 u;
    T* e = reinterpret_cast<T*>(&u);
#pragma unroll
    for (int i = 0; i < N; ++i) e[i] = from_f<T>(in[i]);
    *reinterpret_cast<uint2*>(p) = u;
  }
}

// One output value, fp32 or bf16 (round to nearest even).
__device__ __forceinline__ void store_out(void* o, int out_f32, size_t off, float v) {
  if (out_f32) reinterpret_cast<float*>(o)[off] = v;
  else reinterpret_cast<bf16*>(o)[off] = __float2bfloat16_rn(v);
}

// Round-trip through the storage type (what a store followed by a load
// returns).
template <class T>
__device__ __forceinline__ float through(float x) { return to_f(from_f<T>(x)); }

// ----------------------------------------------------------- own exp, SiLU
//
// The conv's SiLU must be reproducible bit for bit by a plain CPU program, so
// it uses no CUDA math-library function and no division or reciprocal of the
// compiler: only IEEE additions, multiplications and fused multiply-adds,
// rounded to nearest even, in a fixed order, and exact operations on bit
// patterns.
//
// SiLU(z) = z sigmoid(z). With a = |z| (at most 104), t = e^{-a} in [0, 1]
// and d = 1 + t in [1, 2], sigmoid(z) is t/d for z < 0 and 1 - t/d for
// z >= 0, so with c = max(z, 0)
//     SiLU(z) = c - a (t/d)
// for either sign: exp is only taken of a non-positive argument and the
// reciprocal only of a number in [1, 2]. The chain carries -t, -d and -t/d;
// negation is exact and rounding to nearest is symmetric, so every value has
// the roundings of its positive form.
//
// e^{-a}: Cody and Waite's argument reduction (Cody & Waite, "Software Manual
// for the Elementary Functions", 1980): -a = n ln2 + r with n the integer
// nearest -a log2 e, found by one fused multiply-add against 1.5 2^23 (where
// the spacing of floats is 1: the low bits of the sum's pattern are then n);
// ln2 is split into a high part with its low 12 mantissa bits cleared, so
// that n ln2_hi is exact, and a low correction. e^r, |r| <= ln2/2, comes from
// the degree-6 polynomial of least maximum relative error with its first two
// coefficients held at 1, fitted by the Remez exchange algorithm; the free
// coefficients were rounded to float one at a time from c2 upwards, the
// remaining ones refitted after each rounding, for a relative error of
// 3.31e-9 (2^-28.2) with the rounded values below. Horner's rule in -r (the
// odd coefficients negated) with fused multiply-adds, every coefficient
// scaled by 2^-64 (exactly, so the polynomial comes out as p 2^-64 with p's
// own roundings); then one product with -2^(n+64), which rounds once, and
// only where e^{-a} is subnormal. At a = 104 the result is 0 (e^-104 is under
// half the smallest subnormal). Over every float a in [0, 104] the result is
// within 0.90 ulp of e^{-a} where that is a normal float and within 0.86 of
// the subnormal spacing below.
//
// t/d: the hardware's approximate reciprocal r of d (rcp.approx), the
// quotient t r, then one correction with the exact residual,
// q <- q + r (t - d q) (Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34, 1990). For every
// float t in [0, 1] and d = fl(1 + t) this gives the correctly rounded t/d:
// silu_negquot below was run over all of them on sm_103a against the IEEE
// division, with no difference. The SiLU is therefore c - a fl(t/d), with
// t the exp above.
//
// c = max(z, 0) is taken on the bit pattern (a signed-integer maximum with
// 0): it is z for z > 0 and +0 for every z with the sign bit set. A NaN z
// keeps a = NaN, so the result is NaN; z = +inf gives +inf.
namespace silu_consts {
constexpr float kLog2e = 0x1.715476p+0f;        // float(1 / ln 2)
constexpr float kLn2Hi = 0x1.62ep-1f;           // ln 2, low 12 mantissa bits cleared
constexpr float kLn2Lo = 0x1.0bfbe8p-15f;       // float(ln 2 - kLn2Hi)
constexpr float kRound = 12582912.0f;           // 1.5 2^23
constexpr float kC2 = 0x1.fffffcp-2f, kC3 = 0x1.55548cp-3f, kC4 = 0x1.555858p-5f,
                kC5 = 0x1.123e26p-7f, kC6 = 0x1.6ace9ap-10f;   // c0 = c1 = 1
}  // namespace silu_consts

__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// min(|z|, 104), a NaN stays NaN
__device__ __forceinline__ float silu_arg(float z) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(fabsf(z)), "f"(104.0f));
  return r;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// -t/d, correctly rounded, from nt = -t and nd = -d = -fl(1 + t), t in [0, 1]
// (the method above), on two values.
__device__ __forceinline__ float2 silu_negquot(float2 nt, float2 nd) {
  const float2 rc = make_float2(rcp_approx(-nd.x), rcp_approx(-nd.y));   // ~ 1/d
  const float2 nq = __fmul2_rn(nt, rc);
  return __ffma2_rn(rc, __ffma2_rn(nd, nq, nt), nq);
}

// SiLU on two values (the method above), the floating-point steps in packed
// f32x2 form; each value sees exactly the roundings of the scalar steps.
__device__ __forceinline__ float2 own_silu2(float2 z) {
  using namespace silu_consts;
  constexpr float s = 0x1p-64f;
  const float2 a = make_float2(silu_arg(z.x), silu_arg(z.y));
  const float2 m = __ffma2_rn(a, splat2(-kLog2e), splat2(kRound));
  const float2 n = __fadd2_rn(m, splat2(-kRound));
  float2 r = __ffma2_rn(n, splat2(kLn2Hi), a);   // a + n ln2 = -r
  r = __ffma2_rn(n, splat2(kLn2Lo), r);
  float2 p = splat2(kC6 * s);
  p = __ffma2_rn(p, r, splat2(-kC5 * s));
  p = __ffma2_rn(p, r, splat2(kC4 * s));
  p = __ffma2_rn(p, r, splat2(-kC3 * s));
  p = __ffma2_rn(p, r, splat2(kC2 * s));
  p = __ffma2_rn(p, r, splat2(-1.0f * s));
  p = __ffma2_rn(p, r, splat2(1.0f * s));
  // -2^(n+64): the low 9 bits of m's pattern are n mod 512; 447 = 256 + 191
  // puts 64 + 127 into the exponent field and sets the sign bit
  const float2 negs = make_float2(__uint_as_float((__float_as_uint(m.x) << 23) + (447u << 23)),
                                  __uint_as_float((__float_as_uint(m.y) << 23) + (447u << 23)));
  const float2 nt = __fmul2_rn(p, negs);           // -t
  const float2 nd = __fadd2_rn(nt, splat2(-1.0f));  // -d
  const float2 nq = silu_negquot(nt, nd);           // -t/d
  const float2 c = make_float2(__int_as_float(max(__float_as_int(z.x), 0)),
                               __int_as_float(max(__float_as_int(z.y), 0)));
  return __ffma2_rn(a, nq, c);
}

// ----------------------------------------------------------------- gates

// g (log decay) and beta from the raw inputs, fp32, CUDA math library, with
// the head's A_log and dt_bias already at hand.
__device__ __forceinline__ void gates_v(int gate_mode, float A_log_h, float dt_bias_h, float a_in,
                                        float b_in, float& alpha, float& beta) {
  if (gate_mode == 1) {
    alpha = expf(a_in);
    beta = b_in;
    return;
  }
  const float x = __fadd_rn(a_in, dt_bias_h);
  const float sp = (x > 20.0f) ? x : log1pf(expf(x));
  const float g = -__fmul_rn(expf(A_log_h), sp);
  alpha = expf(g);
  beta = __frcp_rn(__fadd_rn(1.0f, expf(-b_in)));
}

__device__ __forceinline__ void gates(const Params& P, int h, float a_in, float b_in,
                                      float& alpha, float& beta) {
  if (P.gate_mode == 1) {
    gates_v(1, 0.0f, 0.0f, a_in, b_in, alpha, beta);
    return;
  }
  gates_v(0, P.A_log[h], P.dt_bias[h], a_in, b_in, alpha, beta);
}

// g (the log decay) and beta, for the chunked form (which works with prefix
// sums of g rather than with e^g), with the head's constants already in
// registers: eA = e^{A_log[h]} and dtb = dt_bias[h]. The same arithmetic as
// gates() up to e^g.
__device__ __forceinline__ void gate_log_c(int gate_mode, float eA, float dtb, float a_in,
                                           float b_in, float& g, float& beta) {
  if (gate_mode == 1) {
    g = a_in;
    beta = b_in;
    return;
  }
  const float x = __fadd_rn(a_in, dtb);
  const float sp = (x > 20.0f) ? x : log1pf(expf(x));
  g = -__fmul_rn(eA, sp);
  beta = __frcp_rn(__fadd_rn(1.0f, expf(-b_in)));
}

// ------------------------------------------------- programmatic launches
//
// Every kernel of the library starts with pdl_begin(): it waits until the
// previous grid on the stream has completed and its writes are visible (so
// stream order is kept exactly: nothing is read or written before), then lets
// the next grid be scheduled. Launched with launch_pdl, a kernel's blocks can
// be resident while the previous grid finishes, which hides the launch
// latency between back-to-back kernels.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Raise a kernel's dynamic shared memory limit once per device (host side;
// later launches, including ones being captured into a graph, skip the call).
// One instantiation, and so one record of devices done, per kernel.
template <auto kernel>
inline cudaError_t ensure_smem_limit(int bytes) {
  static unsigned long long done = 0;  // bit d: set on device d (benign race)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done |= bit;
  return e;
}

}  // namespace gdn
