// Gated DeltaNet layer core: plain CPU oracle.
//
// TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg load this library. The product path (the CUDA
// library) never calls it, shares no code with it, and fails loudly when its
// own extension is missing.
//
// What it follows:
//  * The recurrence and gates are the gated delta rule as stated for the
//    Gated DeltaNet core: per value head, with state S (Dk x Dv),
//      g_t = -exp(A_log) * softplus(a_t + dt_bias),  beta_t = sigmoid(b_t),
//      S <- exp(g_t) S ;  u = beta_t (v_t - S^T k_t) ;  S <- S + k_t u^T ;
//      o_t = scale * S^T q_t,   with q_t, k_t L2-normalised.
//    It runs token by token, the form the r9700-stack v0.2.3 release notes
//    ("1. Time to first token: the GDN prefill core") check their new core
//    against ("an fp64 token-by-token reference").
//  * The conv is the width-W causal depthwise conv over the concatenated
//    q|k|v channels followed by SiLU, with a rolling window of the last W-1
//    raw input columns (r9700-stack v0.2.3, section 1: r9k_gdn_conv; v0.2.4,
//    "A defect found and fixed before the tag": the window rolls by the
//    number of candidate columns).
//
// Readings where the pages are silent (all stated again in the design notes):
//  * L2 norm:   x_hat = x / sqrt(sum x^2 + eps), eps passed in (1e-6).
//  * softplus:  log(1 + exp(x)).
//  * GQA:       value head h reads q/k head floor(h * Hk / Hv).
//  * channels:  [q (Hk*Dk) | k (Hk*Dk) | v (Hv*Dv)], head-major inside each.
//  * conv taps: y_t[c] = SiLU(bias[c] + sum_j w[c][j] * x_{t-(W-1)+j}[c]),
//               history columns oldest first.
//
// Precision: every floating-point step of the recurrence and of
// oracle_conv_f64 is IEEE double. oracle_conv_f32 is the one deliberate
// exception: it is the fp32-accumulate conv that the GPU conv must match bit
// for bit, so it fixes the accumulation order (bias, then taps j = 0..W-1,
// each a fused multiply-add) and evaluates SiLU with its own exp and an
// IEEE quotient (below), from IEEE additions, multiplications, divisions and
// fused multiply-adds only.
// Build with -ffp-contract=off so the compiler adds no contractions.

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- fp64 parts

double softplus_f64(double x) {
  // log(1 + e^x); for large x rewrite as x + log(1 + e^-x) so e^x cannot
  // overflow. Both are the same function.
  if (x > 30.0) return x + std::log1p(std::exp(-x));
  return std::log1p(std::exp(x));
}

double sigmoid_f64(double x) { return 1.0 / (1.0 + std::exp(-x)); }

double silu_f64(double x) { return x * sigmoid_f64(x); }

// Planted mistakes for the tests that prove the pins can fail. 0 = none.
enum Mutation {
  MUT_NONE = 0,
  MUT_NO_DECAY = 1,        // forget the exp(g) decay
  MUT_U_SIGN = 2,          // u = beta (v + S^T k)
  MUT_OUT_BEFORE_UPDATE = 3,  // read o from the state before the k u^T update
  MUT_GQA_MODULO = 4,      // value head h reads q/k head h % Hk
  MUT_NO_Q_NORM = 5,       // skip the L2 norm of q
  MUT_BETA_NOT_SIGMOID = 6,   // beta = b (raw)
  MUT_SOFTPLUS_SIGN = 7,   // g = +exp(A_log) softplus(...)
  MUT_TRANSPOSED_READ = 8, // o_j = scale * sum_i S[j][i] q_i (needs Dk == Dv)
};

struct SeqArgs {
  int R;
  const int* row_start;
  const int* row_len;
  int Hk, Hv, Dk, Dv;
  const double* qkv;  // [T][C]
  const double* a;    // [T][Hv]
  const double* b;    // [T][Hv]
  const double* A_log;    // [Hv]
  const double* dt_bias;  // [Hv]
  double scale;
  double eps;
  int gate_mode;      // 0: raw a/b; 1: a is g (log decay), b is beta
  const double* S0;   // [R][Hv][Dk][Dv] or nullptr (zero)
  double* S_out;      // [R][Hv][Dk][Dv]
  double* o;          // [T][Hv][Dv]
  int mutate;
};

// One (request, value head) pair, token by token, in the order the rule is
// written: decay, delta-rule correction, rank-1 write, read-out.
void seq_one(const SeqArgs& A, int r, int h) {
  const int Hk = A.Hk, Hv = A.Hv, Dk = A.Dk, Dv = A.Dv;
  const long C = 2L * Hk * Dk + (long)Hv * Dv;
  int kh = (int)(((long)h * Hk) / Hv);
  if (A.mutate == MUT_GQA_MODULO) kh = h % Hk;
  const long state_off = ((long)r * Hv + h) * Dk * Dv;

  std::vector<double> S((size_t)Dk * Dv, 0.0);  // S[i*Dv + j], i over Dk
  if (A.S0) std::memcpy(S.data(), A.S0 + state_off, sizeof(double) * Dk * Dv);

  std::vector<double> q(Dk), k(Dk), v(Dv), u(Dv);
  const int t0 = A.row_start[r];
  for (int t = t0; t < t0 + A.row_len[r]; ++t) {
    const double* row = A.qkv + (long)t * C;
    for (int i = 0; i < Dk; ++i) q[i] = row[(long)kh * Dk + i];
    for (int i = 0; i < Dk; ++i) k[i] = row[(long)Hk * Dk + (long)kh * Dk + i];
    for (int j = 0; j < Dv; ++j) v[j] = row[2L * Hk * Dk + (long)h * Dv + j];

    // L2 normalisation of q and k.
    double qq = 0.0, kk = 0.0;
    for (int i = 0; i < Dk; ++i) { qq += q[i] * q[i]; kk += k[i] * k[i]; }
    const double qn = std::sqrt(qq + A.eps), kn = std::sqrt(kk + A.eps);
    if (A.mutate != MUT_NO_Q_NORM)
      for (int i = 0; i < Dk; ++i) q[i] /= qn;
    for (int i = 0; i < Dk; ++i) k[i] /= kn;

    // Gates.
    double g, beta;
    const double at = A.a[(long)t * Hv + h], bt = A.b[(long)t * Hv + h];
    if (A.gate_mode == 0) {
      double sp = softplus_f64(at + A.dt_bias[h]);
      g = -std::exp(A.A_log[h]) * sp;
      if (A.mutate == MUT_SOFTPLUS_SIGN) g = -g;
      beta = (A.mutate == MUT_BETA_NOT_SIGMOID) ? bt : sigmoid_f64(bt);
    } else {
      g = at;
      beta = bt;
    }

    // S <- exp(g) S
    if (A.mutate != MUT_NO_DECAY) {
      const double alpha = std::exp(g);
      for (auto& s : S) s *= alpha;
    }
    // u = beta (v - S^T k)
    for (int j = 0; j < Dv; ++j) {
      double sk = 0.0;
      for (int i = 0; i < Dk; ++i) sk += S[(size_t)i * Dv + j] * k[i];
      u[j] = (A.mutate == MUT_U_SIGN) ? beta * (v[j] + sk) : beta * (v[j] - sk);
    }
    double* out = A.o + ((long)t * Hv + h) * Dv;
    if (A.mutate == MUT_OUT_BEFORE_UPDATE) {
      for (int j = 0; j < Dv; ++j) {
        double sq = 0.0;
        for (int i = 0; i < Dk; ++i) sq += S[(size_t)i * Dv + j] * q[i];
        out[j] = A.scale * sq;
      }
    }
    // S <- S + k u^T
    for (int i = 0; i < Dk; ++i)
      for (int j = 0; j < Dv; ++j) S[(size_t)i * Dv + j] += k[i] * u[j];
    // o = scale S^T q
    if (A.mutate != MUT_OUT_BEFORE_UPDATE) {
      for (int j = 0; j < Dv; ++j) {
        double sq = 0.0;
        if (A.mutate == MUT_TRANSPOSED_READ)
          for (int i = 0; i < Dk; ++i) sq += S[(size_t)j * Dv + i] * q[i];
        else
          for (int i = 0; i < Dk; ++i) sq += S[(size_t)i * Dv + j] * q[i];
        out[j] = A.scale * sq;
      }
    }
  }
  std::memcpy(A.S_out + state_off, S.data(), sizeof(double) * Dk * Dv);
}

template <class F>
void parallel_for(long n, int threads, F f) {
  if (threads <= 1 || n <= 1) {
    for (long i = 0; i < n; ++i) f(i);
    return;
  }
  if (threads > n) threads = (int)n;
  std::vector<std::thread> pool;
  for (int w = 0; w < threads; ++w) {
    pool.emplace_back([=]() {
      for (long i = w; i < n; i += threads) f(i);
    });
  }
  for (auto& th : pool) th.join();
}

// ------------------------------------------------------- fp32 conv mirror
//
// SiLU(z) = z sigmoid(z) in fp32, with the exp of the GPU conv. With
// a = |z| (lowered to at most 104), t = e^{-a} in [0, 1] and d = 1 + t in
// [1, 2], sigmoid(z) = t/d for z < 0 and 1 - t/d for z >= 0, so with
// c = max(z, 0):
//     SiLU(z) = c - a (t/d)
// for both signs: exp is only taken of a non-positive argument. Each step is
// one fp32 rounding: t (the exp below), d = fl(1 + t), the quotient
// fl(t / d) as an IEEE division, and c - a q as one fused multiply-add. The
// chain carries -t, -d and -t/d (negation is exact, so each value has the
// roundings of its positive form).
//
// e^{-a}: Cody & Waite argument reduction (W. J. Cody and W. Waite,
// "Software Manual for the Elementary Functions", 1980): -a = n ln2 + r with
// n the nearest integer to -a log2(e) (one fused multiply-add against
// 1.5 2^23, where the spacing of floats is 1), ln2 split into a short high
// part and a low correction so n*ln2_hi is exact; e^r from the degree-6
// polynomial of least maximum relative error on |r| <= ln2/2 with its first
// two coefficients held at 1 (Remez exchange, coefficients rounded to float
// one at a time from the highest-order free one, refitting the rest after
// each rounding; relative error 3.31e-9 = 2^-28.2 with the rounded
// coefficients), by Horner's rule with fused multiply-adds, the coefficients
// scaled by 2^-64 (exactly); then one product with -2^(n+64), which rounds
// once, and only where e^{-a} is subnormal. At a = 104 the result is 0.
struct OwnExpConsts {
  float log2e, ln2_hi, ln2_lo;
  float c[7];     // e^r ~ sum c_k r^k, |r| <= ln2/2
  OwnExpConsts() {
    const double ln2 = std::log(2.0);
    log2e = (float)(1.0 / ln2);
    // High part of ln2 with its last 12 mantissa bits cleared, so that
    // n * ln2_hi is exact for |n| < 2^12.
    float hi = (float)ln2;
    uint32_t bits;
    std::memcpy(&bits, &hi, 4);
    bits &= 0xFFFFF000u;
    std::memcpy(&hi, &bits, 4);
    ln2_hi = hi;
    ln2_lo = (float)(ln2 - (double)hi);
    const float fit[7] = {1.0f, 1.0f, 0x1.fffffcp-2f, 0x1.55548cp-3f, 0x1.555858p-5f,
                          0x1.123e26p-7f, 0x1.6ace9ap-10f};
    for (int k = 0; k < 7; ++k) c[k] = fit[k];
  }
};
const OwnExpConsts kExp;

float pow2_exact(int n) {  // 2^n for -126 <= n <= 127, built from the bits
  uint32_t bits = (uint32_t)(n + 127) << 23;
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

// -e^{-a} for 0 <= a <= 104 (the caller clamps).
float own_negexp_f32(float a) {
  const float kRound = 12582912.0f;                    // 1.5 2^23
  const float m = std::fma(a, -kExp.log2e, kRound);   // n + 1.5 2^23, n = round(-a log2 e)
  const float n = m - kRound;                          // exact
  float r = std::fma(n, kExp.ln2_hi, a);               // a + n ln2 = -r
  r = std::fma(n, kExp.ln2_lo, r);
  // Horner in -r with the odd coefficients negated: the same roundings as
  // Horner in r
  const float s = pow2_exact(-64);
  float p = (kExp.c[6] * s);
  for (int k = 5; k >= 0; --k) p = std::fma(p, r, ((k & 1) ? -kExp.c[k] : kExp.c[k]) * s);
  return p * -pow2_exact((int)n + 64);
}

// a = min(|z|, 104); a NaN stays NaN.
float silu_arg(float z) { return std::isnan(z) ? z : std::fmin(std::fabs(z), 104.0f); }

float silu_own_f32(float z) {
  const float a = silu_arg(z);
  const float negt = std::isnan(a) ? a : own_negexp_f32(a);
  const float N = negt - 1.0f;                         // -d
  const float nq = negt / -N;                          // -t/d, correctly rounded
  int32_t zb;
  std::memcpy(&zb, &z, 4);
  const int32_t cb = zb > 0 ? zb : 0;                  // max(z, 0) on the bit pattern
  float c;
  std::memcpy(&c, &cb, 4);
  return std::fma(a, nq, c);
}

// e^x for x <= 0 through the same steps (x NaN is treated as -104).
float own_exp_nonpos_f32(float x) {
  const float a = std::fmin(-x, 104.0f);
  return -own_negexp_f32(std::isnan(a) ? 104.0f : a);
}

}  // namespace

extern "C" {

// Own fp32 exp (of a <= 0), exposed for its own pins.
float oracle_exp_f32(float x) { return own_exp_nonpos_f32(x); }
float oracle_silu_f32(float x) { return silu_own_f32(x); }

// Causal depthwise conv + SiLU, fp32 accumulate, fixed order.
//   x     [T][C]       raw inputs (already io-dtype values)
//   hist  [R][W-1][C]  history columns per request, oldest first
//   w     [C][W]       taps; bias [C] or null
//   y     [T][C]       SiLU(conv)
//   hist_out [R][W-1][C] last W-1 columns of [hist; rows] per request
void oracle_conv_f32(int R, const int* row_start, const int* row_len, int C, int W,
                     const float* x, const float* hist, const float* w,
                     const float* bias, float* y, float* hist_out) {
  const int H = W - 1;
  for (int r = 0; r < R; ++r) {
    const int s = row_start[r], n = row_len[r];
    for (int c = 0; c < C; ++c) {
      // the column sequence [hist; rows] for this channel
      std::vector<float> col((size_t)H + n);
      for (int j = 0; j < H; ++j) col[j] = hist[((long)r * H + j) * C + c];
      for (int t = 0; t < n; ++t) col[H + t] = x[(long)(s + t) * C + c];
      for (int t = 0; t < n; ++t) {
        float acc = bias ? bias[c] : 0.0f;
        for (int j = 0; j < W; ++j) acc = std::fma(w[(long)c * W + j], col[t + j], acc);
        y[(long)(s + t) * C + c] = silu_own_f32(acc);
      }
      for (int j = 0; j < H; ++j) hist_out[((long)r * H + j) * C + c] = col[n + j];
    }
  }
}

// Same conv in fp64 (the value the fp32 paths approximate).
void oracle_conv_f64(int R, const int* row_start, const int* row_len, int C, int W,
                     const double* x, const double* hist, const double* w,
                     const double* bias, double* y, double* hist_out) {
  const int H = W - 1;
  for (int r = 0; r < R; ++r) {
    const int s = row_start[r], n = row_len[r];
    for (int c = 0; c < C; ++c) {
      std::vector<double> col((size_t)H + n);
      for (int j = 0; j < H; ++j) col[j] = hist[((long)r * H + j) * C + c];
      for (int t = 0; t < n; ++t) col[H + t] = x[(long)(s + t) * C + c];
      for (int t = 0; t < n; ++t) {
        double acc = bias ? bias[c] : 0.0;
        for (int j = 0; j < W; ++j) acc += w[(long)c * W + j] * col[t + j];
        y[(long)(s + t) * C + c] = silu_f64(acc);
      }
      for (int j = 0; j < H; ++j) hist_out[((long)r * H + j) * C + c] = col[n + j];
    }
  }
}

// Gated delta rule, token by token, fp64, with the q/k L2 norm and gates
// computed per token. Parallel over (request, value head).
//   S0/S_out: [R][Hv][Dk][Dv] (row i over Dk, column j over Dv)
//   o:        [T][Hv][Dv]
// Returns 0, or -1 on bad arguments.
int oracle_gdn_f64(int R, const int* row_start, const int* row_len,
                   int Hk, int Hv, int Dk, int Dv,
                   const double* qkv, const double* a, const double* b,
                   const double* A_log, const double* dt_bias,
                   double scale, double eps, int gate_mode,
                   const double* S0, double* S_out, double* o,
                   int threads, int mutate) {
  if (R < 0 || Hk <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0 || Hv % Hk != 0) return -1;
  if (mutate == MUT_TRANSPOSED_READ && Dk != Dv) return -1;
  SeqArgs A{R, row_start, row_len, Hk, Hv, Dk, Dv, qkv, a, b, A_log, dt_bias,
            scale, eps, gate_mode, S0, S_out, o, mutate};
  parallel_for((long)R * Hv, threads, [&](long i) { seq_one(A, (int)(i / Hv), (int)(i % Hv)); });
  return 0;
}

}  // extern "C"
