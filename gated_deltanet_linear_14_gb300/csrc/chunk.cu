// Chunked prefill of the gated delta rule on the tcgen05 tensor cores
// (sm_103a): the WY (UT-transform) chunk form, 64 tokens per chunk.
//
// r9700-stack v0.2.3, section 1, names the chunked GDN core used for prompts
// above the token-by-token threshold and its numerics (solves on bf16 q/k
// land at 5e-3 from an fp64 token-by-token reference). The chunk form is not
// written out there; this is its standard statement. Per chunk with state S
// (Dk x Dv), gamma_t = sum_{s<=t} g_s, k^/q^ the L2-normalised rows:
//   A  = strictly_lower(beta_t e^{gamma_t-gamma_s} k^_t.k^_s),  T = (I+A)^-1
//   W  = T diag(beta e^gamma) K^,   U = T diag(beta) V,   Vn = U - W S
//   O  = scale (diag(e^gamma) Q^ S + (Q^ K^T o e^{gamma_t-gamma_s} o causal) Vn)
//   S <- e^{gamma_L} S + (diag(e^{gamma_L-gamma}) K^)^T Vn
//
// Design. One CTA (8 warps) per (request, value head) walks the request's
// chunks. Every contraction is an M = 128 tcgen05.mma with bf16 operands in
// 128B-swizzled shared memory and fp32 accumulators in tensor memory; the
// 128 rows are Dk or Dv (or the 64 q rows stacked on the 64 k rows), so in
// every epilogue a thread owns one TMEM lane (one row) and its warpgroup
// half of the columns:
//   MMA1  [Q;K] K^T          -> QK^T and KK^T (raw bf16: exact products);
//                               |k_t|^2 is the diagonal of KK^T
//   MMA2  K^T T_W^T          -> W^T   (T_W = T diag(beta e^gamma / |k|))
//   MMA3  V^T T_U^T          -> U^T   (T_U = T diag(beta))
//   MMA4  S^T W^T            -> (W S)^T
//   MMA5  S^T Q^T            -> (Q S)^T
//   MMA6  Vn^T P^T           -> (P Vn)^T   (P = masked, gated, normalised QK^T)
//   MMA7  S^T += V'^T K      (V' = diag(e^{gamma_L-gamma} / |k|) Vn), on top
//                               of e^{gamma_L} S written back into TMEM
// Raw q/k/v are exact in bf16; every fp32 operand (T_W, T_U, S, W, Vn, P,
// V') is split into bf16 hi + lo and the products summed (dropping lo x lo),
// which keeps about 2^-16 relative accuracy: fp32-grade results from the
// bf16 tensor pipe. The 64 x 64 unit-lower-triangular inverse T is computed
// on the CUDA cores (16 x 16 diagonal blocks, then two 32 x 32 rounds). The
// state stays fp32 in TMEM for the whole request. Tiles arrive by TMA
// (SWIZZLE_128B) straight into the operand layout; the next chunk's tiles
// are fetched while the current chunk's outputs are written, and its gates
// are formed while this chunk's MMA4/5 run.
#include <cuda.h>

#include "chunk_core.cuh"
#include "kernels.h"

namespace gdn {

using namespace umma;

// Shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t OFF_QK = 0;        // per 64-column atom a (a*16384): Q rows 0..63, K rows 64..127
constexpr uint32_t OFF_V = 32768;     // V atom a at OFF_V + a*8192 (64 rows each)
constexpr uint32_t OFF_P = 49152;     // P hi [64][64] | P lo
constexpr uint32_t OFF_R1 = 65536;    // T_W hi | T_W lo | T_U hi | T_U lo (8 KB each)
                                      //  -> Vn^T hi | lo ([128][64], 16 KB each); solve scratch
constexpr uint32_t OFF_R2 = 98304;    // A, T fp32 [64][64] -> W^T hi | lo -> V'^T hi | lo
constexpr uint32_t OFF_S = 131072;    // S^T hi: atom a at a*16384 ([128][64]); S^T lo at +32768
constexpr uint32_t OFF_VEC = 196608;  // per-token vectors (8 x 64 floats)
constexpr uint32_t kChunkSmem = OFF_VEC + 8 * 64 * 4 + 2048;  // + 1024-byte alignment slack

// TMEM columns (512 allocated).
constexpr uint32_t TM_D1 = 0, TM_W = 64, TM_U = 128, TM_WS = 192, TM_S = 256, TM_OQ = 384,
                   TM_OP = 448;

template <class ST>
__global__ void __launch_bounds__(kChunkThreads, 1)
chunk_kernel(const __grid_constant__ CUtensorMap tm_qkv, Geom G, Batch B, Params P,
             const bf16* __restrict__ a_in, const bf16* __restrict__ b_in, void* o, int out_f32,
             void* pages, int32_t* status) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float gamma_carry;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & 127;    // TMEM lane (row) of this thread
  const int wg = tid >> 7;      // column half this warpgroup handles
  const int h = blockIdx.x;
  const bool reporter = (h == 0 && tid == 0);
  const Req q = load_req(B, blockIdx.y);
  if (q.err) {
    if (reporter) report(status, q.err);
    return;
  }
  if (q.spec) return;
  if (q.len < B.min_len || q.len > B.max_len) return;
  char* pg = page_ptr(G, pages, q.page);
  uint32_t* flagp = reinterpret_cast<uint32_t*>(pg + G.flag_off);
  if (!q.fresh && flag_width(*flagp) != 0) {
    if (reporter) report(status, GDN_DEV_RECORD_OPEN);
    return;
  }
  if (!q.fresh && q.len == 0) return;
  ST* Sb = reinterpret_cast<ST*>(pg + G.state_off) + (size_t)h * kCD * kCD;
  const int kh = (int)(((long long)h * G.Hk) / G.Hv);

  float* s_l2 = reinterpret_cast<float*>(sm + OFF_VEC);   // gamma log2(e)
  float* s_beta = s_l2 + 64;
  float* s_gam = s_beta + 64;
  float* s_iq = s_gam + 64;
  float* s_ik = s_iq + 64;
  float* s_cw = s_ik + 64;   // beta e^gamma / |k|      (columns of T_W)
  float* s_cv = s_cw + 64;   // e^{gamma_L-gamma} / |k| (columns of V')
  float* s_co = s_cv + 64;   // e^gamma / |q|           (rows of the Q S term)
  float* Am = reinterpret_cast<float*>(sm + OFF_R2);
  float* Tm = Am + 64 * 64;
  float* Xs = reinterpret_cast<float*>(sm + OFF_R1);

  const uint32_t bar_tma = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's lanes
  const uint32_t sb = smem_u32(sm);

  // the initial state S^T (row j, columns of this warpgroup's half) into TMEM
  {
    float v[32];
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      const int cc = 2 * wg + c2;
      if (q.fresh) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      } else {
        load_f<ST, 32>(Sb + (size_t)row * kCD + cc * 32, v);
      }
      tmem_st32(trow + TM_S + cc * 32, v);
    }
    tmem_st_wait();
  }

  const int nchunks = (q.len + kCL - 1) / kCL;
  const int xq = kh * kCD, xk = G.Hk * kCD + kh * kCD, xv = 2 * G.Hk * kCD + h * G.Dv;
  // phases issued (by thread 0) and completed, for the drain after a failed wait
  uint32_t tma_iss = 0, tma_done = 0, m_iss = 0, m_done = 0;
  auto issue_tma = [&](int c) {
    ++tma_iss;
    const int y = q.start + c * kCL;
    mbar_expect_tx(bar_tma, 6 * 8192);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      tma_load_2d(sb + OFF_QK + a * 16384, &tm_qkv, xq + 64 * a, y, bar_tma);
      tma_load_2d(sb + OFF_QK + a * 16384 + 8192, &tm_qkv, xk + 64 * a, y, bar_tma);
      tma_load_2d(sb + OFF_V + a * 8192, &tm_qkv, xv + 64 * a, y, bar_tma);
    }
  };
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && nchunks > 0) issue_tma(0);

  // Gates of chunk cc (threads tid < kCL, one token each): beta into s_beta;
  // returns this thread's gamma scanned within its warp (the first warp's
  // total goes to gamma_carry; after a barrier the caller adds it for the
  // second warp and writes s_gam and s_l2 = gamma log2 e).
  auto load_ab = [&](int cc, float& a_v, float& b_v) {
    const int n = min(kCL, q.len - cc * kCL);
    const size_t R = (size_t)q.start + (size_t)cc * kCL;
    a_v = 0.0f;
    b_v = 0.0f;
    if (tid < n) {
      a_v = to_f(a_in[(R + tid) * G.Hv + h]);
      b_v = to_f(b_in[(R + tid) * G.Hv + h]);
    }
  };
  // the head's gate constants, read once
  const float gate_eA = (P.gate_mode == 1) ? 0.0f : expf(P.A_log[h]);
  const float gate_dtb = (P.gate_mode == 1) ? 0.0f : P.dt_bias[h];
  auto gates_scan = [&](int cc, float a_v, float b_v) -> float {
    float g = 0.0f, beta = 0.0f;
    if (tid < min(kCL, q.len - cc * kCL))
      gate_log_c(P.gate_mode, gate_eA, gate_dtb, a_v, b_v, g, beta);
    s_beta[tid] = beta;
    const int lane = tid & 31;
#pragma unroll
    for (int dd = 1; dd < 32; dd <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, g, dd);
      if (lane >= dd) g = __fadd_rn(g, y);
    }
    if (tid == 31) gamma_carry = g;
    return g;
  };
  if (nchunks > 0) {
    float g0 = 0.0f;
    if (tid < kCL) {
      float a0, b0;
      load_ab(0, a0, b0);
      g0 = gates_scan(0, a0, b0);
    }
    __syncthreads();
    if (tid < kCL) {
      s_gam[tid] = (tid >= 32) ? __fadd_rn(g0, gamma_carry) : g0;
      s_l2[tid] = __fmul_rn(s_gam[tid], kLog2e);
    }
  }

  uint32_t mma_count = 0;
  bool fail = false;
  auto wait_mma = [&]() -> bool {
    const bool ok = mbar_wait(bar_mma, mma_count & 1);
    ++mma_count;
    const bool any_fail = __syncthreads_or(!ok);
    tc_fence_after();
    if (!any_fail) ++m_done;
    return !any_fail;
  };

  for (int c = 0; c < nchunks; ++c) {
    const int n_c = min(kCL, q.len - c * kCL);
    const size_t R0 = (size_t)q.start + (size_t)c * kCL;
    // the next chunk's raw gates, used while this chunk's MMA4/5 run
    float a_n = 0.0f, b_n = 0.0f;
    if (c + 1 < nchunks && tid < kCL) load_ab(c + 1, a_n, b_n);
    {
      const bool ok = mbar_wait(bar_tma, c & 1);
      if (__syncthreads_or(!ok)) { fail = true; break; }
      ++tma_done;
    }
    if (n_c < kCL) {
      // rows past the request's end belong to other requests: zero them
      const int nrow = kCL - n_c;
      for (int idx = tid; idx < nrow * 6 * 8; idx += kChunkThreads) {
        const int r = n_c + idx / 48, rest = idx % 48, tile = rest / 8, ch = rest % 8;
        const uint32_t base = (tile < 4) ? OFF_QK + (tile >> 1) * 16384 + (tile & 1) * 8192
                                         : OFF_V + (tile - 4) * 8192;
        *reinterpret_cast<uint4*>(sm + base + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_async_smem();
    }
    __syncthreads();

    // MMA1: [Q;K] K^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t base = sb + OFF_QK + (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16(tmem + TM_D1, sdesc(base, 16, 1024), sdesc(base + 8192, 16, 1024), id, ks > 0);
      }
      mma_commit(bar_mma);
      ++m_iss;
    }
    // q norms while it runs (this chunk's gates are in place already)
    if (tid < kCL) {
      float qq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 u = *reinterpret_cast<const uint4*>(sm + OFF_QK + a * 16384 + sw128_chunk(tid, ch));
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = __uint_as_float(w4[e] << 16), x1 = __uint_as_float(w4[e] & 0xFFFF0000u);
            qq[e] = __fmaf_rn(x0, x0, qq[e]);
            qq[e] = __fmaf_rn(x1, x1, qq[e]);
          }
        }
      s_iq[tid] = rsqrtf(__fadd_rn(__fadd_rn(__fadd_rn(qq[0], qq[1]), __fadd_rn(qq[2], qq[3])), P.eps));
    }
    if (!wait_mma()) { fail = true; break; }

    float d1[32];   // columns [32 wg, 32 wg + 32) of this thread's row of [QK^T; KK^T]
    tmem_ld32(trow + TM_D1 + 32 * wg, d1);
    if (row >= kCL && ((row - kCL) >> 5) == wg) {
      // |k_t|^2 is the diagonal of KK^T: column t sits in this half
      const int t = row - kCL;
      float kk = 0.0f;
#pragma unroll
      for (int s = 0; s < 32; ++s) kk = (s == (t & 31)) ? d1[s] : kk;
      s_ik[t] = rsqrtf(__fadd_rn(kk, P.eps));
    }
    __syncthreads();
    const float gL = s_gam[kCL - 1];
    if (tid < kCL) {
      const float eg = expf(s_gam[tid]);
      s_cw[tid] = __fmul_rn(__fmul_rn(s_beta[tid], eg), s_ik[tid]);
      s_cv[tid] = __fmul_rn(expf(__fsub_rn(gL, s_gam[tid])), s_ik[tid]);
      s_co[tid] = __fmul_rn(eg, s_iq[tid]);
    }
    if (row < kCL) {
      // P row t, columns of this half: masked, gated, normalised q_t . k_s (s <= t < n_c)
      const int t = row;
      const float iq = s_iq[t], lt = s_l2[t];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int s = 32 * wg + i;
        d1[i] = (s <= t && t < n_c)
                    ? __fmul_rn(__fmul_rn(__fmul_rn(d1[i], iq), s_ik[s]), exp2f(__fsub_rn(lt, s_l2[s])))
                    : 0.0f;
      }
      store_half_hilo(sm + OFF_P, sm + OFF_P + 8192, t, wg, d1);
    } else {
      // A row t: beta_t e^{gamma_t - gamma_s} k^_t . k^_s for s < t
      const int t = row - kCL;
      const float ikt = s_ik[t], lt = s_l2[t], bt = s_beta[t];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 v;
        float* vp = &v.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ss = 32 * wg + i + e;
          vp[e] = (ss < t && t < n_c)
                      ? __fmul_rn(__fmul_rn(__fmul_rn(__fmul_rn(d1[i + e], ikt), s_ik[ss]), bt),
                                  exp2f(__fsub_rn(lt, s_l2[ss])))
                      : 0.0f;
        }
        *reinterpret_cast<float4*>(&Am[mat_idx(t, 32 * wg + i)]) = v;
      }
    }
    __syncthreads();
    solve_unit_lower64(Am, Tm, Xs, tid);

    // T_W = T diag(beta e^gamma / |k|), T_U = T diag(beta), hi/lo bf16 tiles
    {
      // thread -> (row t, which of T_W / T_U, column half)
      const int t = tid & 63, which = (tid >> 6) & 1, half = tid >> 7;
      float w[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(&Tm[mat_idx(t, 32 * half + i)]);
        w[i] = v.x; w[i + 1] = v.y; w[i + 2] = v.z; w[i + 3] = v.w;
      }
      const float* colscale = which ? s_beta : s_cw;
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = __fmul_rn(w[i], colscale[32 * half + i]);
      store_half_hilo(sm + OFF_R1 + which * 16384, sm + OFF_R1 + which * 16384 + 8192, t, half, w);
    }
    fence_async_smem();
    __syncthreads();
    // MMA2: W^T = K^T T_W^T ; MMA3: U^T = V^T T_U^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64, 1, 0);
#pragma unroll
      for (int pass = 0; pass < 2; ++pass)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_W, sdesc(sb + OFF_QK + 8192 + ks * 2048, 16384, 1024),
                   sdesc(sb + OFF_R1 + pass * 8192 + ks * 32, 16, 1024), id, (pass | ks) != 0);
#pragma unroll
      for (int pass = 0; pass < 2; ++pass)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_U, sdesc(sb + OFF_V + ks * 2048, 8192, 1024),
                   sdesc(sb + OFF_R1 + 16384 + pass * 8192 + ks * 32, 16, 1024), id, (pass | ks) != 0);
      mma_commit(bar_mma);
      ++m_iss;
    }
    // S^T hi/lo operand tiles, and e^{gamma_L} S^T back into TMEM for MMA7
    {
      const float eL = expf(gL);
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int cc = 2 * wg + c2;
        float v[32];
        tmem_ld32(trow + TM_S + cc * 32, v);
        store_half_hilo(sm + OFF_S + (cc >> 1) * 16384, sm + OFF_S + 32768 + (cc >> 1) * 16384, row,
                        cc & 1, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], eL);
        tmem_st32(trow + TM_S + cc * 32, v);
      }
      tmem_st_wait();
    }
    if (!wait_mma()) { fail = true; break; }

    // W^T rows (MN-major B operand of MMA4)
    {
      {
        float w[32];
        tmem_ld32(trow + TM_W + wg * 32, w);
        store_half_hilo(sm + OFF_R2, sm + OFF_R2 + 16384, row, wg, w);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // MMA4: (W S)^T = S^T W^T (3 hi/lo passes) ; MMA5: (Q S)^T = S^T Q^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id4 = idesc_bf16(128, 64, 0, 1);
      const int sel_s[3] = {0, 0, 1}, sel_w[3] = {0, 1, 0};
#pragma unroll
      for (int pass = 0; pass < 3; ++pass)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16(tmem + TM_WS,
                   sdesc(sb + OFF_S + sel_s[pass] * 32768 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                   sdesc(sb + OFF_R2 + sel_w[pass] * 16384 + ks * 2048, 16384, 1024), id4,
                   (pass | ks) != 0);
      const uint32_t id5 = idesc_bf16(128, 64, 0, 0);
#pragma unroll
      for (int pass = 0; pass < 2; ++pass)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16(tmem + TM_OQ,
                   sdesc(sb + OFF_S + pass * 32768 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                   sdesc(sb + OFF_QK + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024), id5,
                   (pass | ks) != 0);
      mma_commit(bar_mma);
      ++m_iss;
    }
    // the next chunk's gates while they run: past this point the chunk reads
    // none of s_beta, s_gam, s_l2 (its later phases use s_cv and s_co)
    float g_nx = 0.0f;
    if (c + 1 < nchunks && tid < kCL) g_nx = gates_scan(c + 1, a_n, b_n);
    if (!wait_mma()) { fail = true; break; }
    if (c + 1 < nchunks && tid < kCL) {
      s_gam[tid] = (tid >= 32) ? __fadd_rn(g_nx, gamma_carry) : g_nx;
      s_l2[tid] = __fmul_rn(s_gam[tid], kLog2e);
    }

    // Vn^T = U^T - (W S)^T ; V'^T = Vn^T diag(e^{gamma_L - gamma} / |k|)
    {
      {
        const int half = wg;
        float u[32], ws[32];
        tmem_ld32(trow + TM_U + half * 32, u);
        tmem_ld32(trow + TM_WS + half * 32, ws);
#pragma unroll
        for (int s = 0; s < 32; ++s) u[s] = __fsub_rn(u[s], ws[s]);
        store_half_hilo(sm + OFF_R1, sm + OFF_R1 + 16384, row, half, u);
#pragma unroll
        for (int s = 0; s < 32; ++s) u[s] = __fmul_rn(u[s], s_cv[half * 32 + s]);
        store_half_hilo(sm + OFF_R2, sm + OFF_R2 + 16384, row, half, u);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // MMA6: (P Vn)^T = Vn^T P^T ; MMA7: S^T += V'^T K
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id6 = idesc_bf16(128, 64, 0, 0);
      const int sel_v[3] = {0, 0, 1}, sel_p[3] = {0, 1, 0};
#pragma unroll
      for (int pass = 0; pass < 3; ++pass)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_OP, sdesc(sb + OFF_R1 + sel_v[pass] * 16384 + ks * 32, 16, 1024),
                   sdesc(sb + OFF_P + sel_p[pass] * 8192 + ks * 32, 16, 1024), id6,
                   (pass | ks) != 0);
      const uint32_t id7 = idesc_bf16(128, 128, 0, 1);
#pragma unroll
      for (int pass = 0; pass < 2; ++pass)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_S, sdesc(sb + OFF_R2 + pass * 16384 + ks * 32, 16, 1024),
                   sdesc(sb + OFF_QK + 8192 + ks * 2048, 16384, 1024), id7, 1u);
      mma_commit(bar_mma);
      ++m_iss;
    }
    if (!wait_mma()) { fail = true; break; }
    if (tid == 0 && c + 1 < nchunks) issue_tma(c + 1);

    // outputs: O[t][j] = scale (e^{gamma_t} |q_t|^-1 (S^T Q^T)[j][t] + (Vn^T P^T)[j][t]),
    // gathered as a [64][128] tile in shared memory (the Vn^T region, free
    // once MMA6 has read it) and written out as whole 16-byte row pieces
    {
      const int half = wg;
      float oq[32], op[32];
      tmem_ld32(trow + TM_OQ + half * 32, oq);
      tmem_ld32(trow + TM_OP + half * 32, op);
      float* of = reinterpret_cast<float*>(sm + OFF_R1);
      bf16* ob = reinterpret_cast<bf16*>(sm + OFF_R1);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = half * 32 + i;
        const float v = __fmul_rn(P.scale, __fmaf_rn(s_co[t], oq[i], op[i]));
        if (out_f32) of[t * kCD + row] = v;
        else ob[t * kCD + row] = __float2bfloat16_rn(v);
      }
    }
    __syncthreads();
    {
      const int lg = out_f32 ? 5 : 4;                    // log2 of 16-byte pieces per row
      const int per_row = 1 << lg;
      const uint4* src = reinterpret_cast<const uint4*>(sm + OFF_R1);
      for (int idx = tid; idx < (n_c << lg); idx += kChunkThreads) {
        const int t = idx >> lg, piece = idx & (per_row - 1);
        const size_t row_off = ((R0 + t) * G.Hv + h) * G.Dv;
        uint4* dst = out_f32 ? reinterpret_cast<uint4*>(reinterpret_cast<float*>(o) + row_off)
                             : reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(o) + row_off);
        dst[piece] = src[t * per_row + piece];
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (!fail) {
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      const int cc = 2 * wg + c2;
      float v[32];
      tmem_ld32(trow + TM_S + cc * 32, v);
      store_f<ST, 32>(Sb + (size_t)row * kCD + cc * 32, v);
    }
    if (q.fresh && h == 0 && tid == 0) *flagp = 0u;  // empty record
  } else if (tid == 0) {
    report(status, GDN_DEV_TIMEOUT);
    // let the copies and MMAs still in flight finish (each wait bounded)
    // before the shared and tensor memory are given up
    for (uint32_t k = tma_done; k < tma_iss; ++k) mbar_wait(bar_tma, k & 1);
    for (uint32_t k = m_done; k < m_iss; ++k) mbar_wait(bar_mma, k & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t launch_chunk(const void* tmap, const Geom& G, const Batch& B, const Params& P,
                         int state_bf16, int out_f32, const void* a, const void* b, void* o,
                         void* pages, int32_t* status, cudaStream_t stream) {
  const CUtensorMap& tm = *static_cast<const CUtensorMap*>(tmap);
  dim3 grid(G.Hv, B.R);
  if (state_bf16) {
    cudaError_t e = ensure_smem_limit<chunk_kernel<bf16>>((int)kChunkSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(chunk_kernel<bf16>, grid, dim3(kChunkThreads), kChunkSmem, stream, tm, G, B, P,
                   static_cast<const bf16*>(a), static_cast<const bf16*>(b), o, out_f32, pages,
                   status);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = ensure_smem_limit<chunk_kernel<float>>((int)kChunkSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(chunk_kernel<float>, grid, dim3(kChunkThreads), kChunkSmem, stream, tm, G, B,
                   P, static_cast<const bf16*>(a), static_cast<const bf16*>(b), o, out_f32, pages,
                   status);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace gdn
