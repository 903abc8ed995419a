// Chunked prefill in two passes (sm_103a): the same WY (UT-transform) chunk
// form as chunk.cu, with the work that does not depend on the state taken
// off the per-request chain.
//
// r9700-stack v0.2.3, section 1, names the chunked GDN core used for prompts
// above the token-by-token threshold; the chunk form is written out in
// chunk.cu. Of its per-chunk steps only W S, Q S, P Vn and the state update
// read the state; MMA1 ([Q;K] K^T), the A / P epilogue, the triangular solve
// and T_W K, T_U V depend on the chunk's own rows alone.
//
//   pass 1, chunk_prep_kernel: one CTA per (request, value head, chunk), two
//     CTAs per SM. It runs those state-independent steps exactly as the
//     one-kernel form does and writes, per item, the operands the chain will
//     need into the workspace: W^T as bf16 hi/lo tiles in the 128B-swizzled
//     operand layout, Q^T (exact in bf16) beside W^T hi, P as hi/lo tiles,
//     U^T in fp32, and the per-token factors e^{gamma_L - gamma}/|k|,
//     e^gamma/|q| and e^{gamma_L}.
//   pass 2, chunk_seq_kernel: one CTA per (request, value head) walks the
//     chunks with the fp32 state in tensor memory. Per chunk: split S^T into
//     hi/lo operand tiles (and decay it in TMEM), MMA4/5 S^T [W^T | Q^T] (one
//     N = 128 product for both), Vn = U - W S and V', MMA6 Vn^T P^T and MMA7
//     S^T += V'^T K. The operands of chunk c+1 are fetched while chunk c runs
//     (W^T, Q^T and the factors once MMA4/5 have read theirs, P and K once
//     MMA6/7 have), and the outputs of chunk c are formed while MMA4/5 of
//     chunk c+1 run.
//
// Every value is computed by the same operations in the same order as in the
// one-kernel form, so the two forms agree bit for bit.
#include <cuda.h>

#include "chunk_core.cuh"
#include "kernels.h"

namespace gdn {

// ------------------------------------------------------------------ pass 1

// Shared memory of the pre-pass (bytes from a 1024-aligned base). Every
// output is staged in its workspace layout and written by bulk copies.
constexpr uint32_t PP_QK = 0;        // TMA: per atom a (a*16384) Q rows 0..63, K rows 64..127;
                                     //   Q^T rows 0..63 | 64..127 in the Q halves once MMA1
                                     //   and the norms have read Q; W^T lo in the K halves
                                     //   once MMA2 has read K
constexpr uint32_t PP_V = 32768;     // TMA: V atom a at PP_V + a*8192; then W^T hi
constexpr uint32_t PP_P = 49152;     // P hi | lo [64][64]
constexpr uint32_t PP_A = 65536;     // A fp32 [64][64] -> T_W hi | lo -> U^T (with PP_T)
constexpr uint32_t PP_T = 81920;     // T fp32 [64][64] -> T_U hi | lo (in place)
constexpr uint32_t PP_X = 98304;     // solve scratch (4 KB)
constexpr uint32_t PP_VEC = 102400;  // 9 x 64 floats of per-token vectors
constexpr uint32_t kPrepSmem = PP_VEC + 9 * 256 + 1024;

// U^T in the workspace, piece-major: the 16-byte piece q (4 floats) of row
// j's half h sits at ((h * 8 + q) * 128 + j) * 16, so the 32 rows of a warp
// read or write one piece as 512 contiguous bytes.
__device__ __forceinline__ uint32_t ut_piece(int j, int half, int q) {
  return (uint32_t)((((half * 8 + q) << 7) + j) << 4);
}

// A 16-byte load through the read-only path, issued where it is written (the
// chain issues its U^T loads at the top of a chunk and uses them after MMA4/5).
__device__ __forceinline__ float4 ldg_nc_early(const void* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"((uint64_t)dst),
               "r"(src), "r"(bytes)
               : "memory");
}
// commit the bulk stores issued so far and wait until they have read shared
// memory (the writes complete before the grid does)
__device__ __forceinline__ void bulk_store_commit_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait for the previous grid without letting the next one start early: the
// chain that follows holds a whole SM per CTA, and started early it would
// take SMs from this grid's later waves.
__device__ __forceinline__ void pdl_wait_only() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__global__ void __launch_bounds__(kChunkThreads, 2)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_qkv, Geom G, Batch B, Params P,
                  const bf16* __restrict__ a_in, const bf16* __restrict__ b_in, char* ws,
                  int ws_chunks, int32_t* status) {
  pdl_wait_only();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float gamma_carry;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & 127;
  const int wg = tid >> 7;
  const int c = blockIdx.x, h = blockIdx.y;
  const Req q = load_req(B, blockIdx.z);
  // request errors are the chain's to report; its rows need no pre-pass
  if (q.err || q.spec || q.len < B.min_len || q.len > B.max_len) return;
  if (c * kCL >= q.len) return;
  const int n_c = min(kCL, q.len - c * kCL);
  const int kh = (int)(((long long)h * G.Hk) / G.Hv);
  char* item = ws + (((size_t)q.r * G.Hv + h) * ws_chunks + c) * kChunkItemBytes;

  float* s_l2 = reinterpret_cast<float*>(sm + PP_VEC);
  float* s_beta = s_l2 + 64;
  float* s_gam = s_beta + 64;
  float* s_iq = s_gam + 64;
  float* s_ik = s_iq + 64;
  float* s_cw = s_ik + 64;   // beta e^gamma / |k|
  float* s_cv = s_cw + 64;   // e^{gamma_L-gamma} / |k|  } written out
  float* s_co = s_cv + 64;   // e^gamma / |q|            } together
  float* s_el = s_co + 64;   // e^{gamma_L}              } (768 bytes)
  float* Am = reinterpret_cast<float*>(sm + PP_A);
  float* Tm = reinterpret_cast<float*>(sm + PP_T);
  float* Xs = reinterpret_cast<float*>(sm + PP_X);

  const uint32_t bar_tma = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const uint32_t sb = smem_u32(sm);
  constexpr uint32_t TM_D1 = 0, TM_W = 64, TM_U = 128;

  const int xq = kh * kCD, xk = G.Hk * kCD + kh * kCD, xv = 2 * G.Hk * kCD + h * G.Dv;
  const size_t R0 = (size_t)q.start + (size_t)c * kCL;
  if (tid == 0) {
    mbar_expect_tx(bar_tma, 6 * 8192);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      tma_load_2d(sb + PP_QK + a * 16384, &tm_qkv, xq + 64 * a, (int)R0, bar_tma);
      tma_load_2d(sb + PP_QK + a * 16384 + 8192, &tm_qkv, xk + 64 * a, (int)R0, bar_tma);
      tma_load_2d(sb + PP_V + a * 8192, &tm_qkv, xv + 64 * a, (int)R0, bar_tma);
    }
  }

  // gates of the chunk's tokens (threads tid < kCL, one token each)
  {
    float g = 0.0f, beta = 0.0f;
    if (tid < n_c) {
      const float gate_eA = (P.gate_mode == 1) ? 0.0f : expf(P.A_log[h]);
      const float gate_dtb = (P.gate_mode == 1) ? 0.0f : P.dt_bias[h];
      const float a_v = to_f(a_in[(R0 + tid) * G.Hv + h]);
      const float b_v = to_f(b_in[(R0 + tid) * G.Hv + h]);
      gate_log_c(P.gate_mode, gate_eA, gate_dtb, a_v, b_v, g, beta);
    }
    if (tid < kCL) {
      s_beta[tid] = beta;
      const int lane = tid & 31;
#pragma unroll
      for (int dd = 1; dd < 32; dd <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, g, dd);
        if (lane >= dd) g = __fadd_rn(g, y);
      }
      if (tid == 31) gamma_carry = g;
    }
    __syncthreads();
    if (tid < kCL) {
      s_gam[tid] = (tid >= 32) ? __fadd_rn(g, gamma_carry) : g;
      s_l2[tid] = __fmul_rn(s_gam[tid], kLog2e);
    }
  }

  // phases issued and completed, for the drain after a failed wait
  uint32_t tma_done = 0, mma_iss = 0, mma_done = 0;
  bool ok = mbar_wait(bar_tma, 0);
  if (__syncthreads_or(!ok)) goto fail;
  tma_done = 1;
  if (n_c < kCL) {
    // rows past the request's end belong to other requests: zero them
    const int nrow = kCL - n_c;
    for (int idx = tid; idx < nrow * 6 * 8; idx += kChunkThreads) {
      const int r = n_c + idx / 48, rest = idx % 48, tile = rest / 8, ch = rest % 8;
      const uint32_t base = (tile < 4) ? PP_QK + (tile >> 1) * 16384 + (tile & 1) * 8192
                                       : PP_V + (tile - 4) * 8192;
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
      const uint32_t base = sb + PP_QK + (ks >> 2) * 16384 + (ks & 3) * 32;
      mma_bf16(tmem + TM_D1, sdesc(base, 16, 1024), sdesc(base + 8192, 16, 1024), id, ks > 0);
    }
    mma_commit(bar_mma);
    ++mma_iss;
  }
  if (tid < kCL) {
    float qq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 u = *reinterpret_cast<const uint4*>(sm + PP_QK + a * 16384 + sw128_chunk(tid, ch));
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
  // Q^T [128 i][64 t] as an MN-major operand tile (exact in bf16) for the
  // chain's merged W S / Q S product: this thread's row i, half wg of t,
  // gathered from the K-major Q tile while MMA1 runs, then written over the
  // Q halves (rows 0..63 in atom 0's, 64..127 in atom 1's)
  uint32_t qt[16];
  {
    const int ii = row & 63;
    const uint8_t* qa = sm + PP_QK + (row >> 6) * 16384;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int t0 = 32 * wg + 2 * e;
      const uint32_t lo = *reinterpret_cast<const uint16_t*>(
          qa + t0 * 128 + ((((ii >> 3) ^ (t0 & 7)) << 4) | ((ii & 7) << 1)));
      const uint32_t hi = *reinterpret_cast<const uint16_t*>(
          qa + (t0 + 1) * 128 + ((((ii >> 3) ^ ((t0 + 1) & 7)) << 4) | ((ii & 7) << 1)));
      qt[e] = lo | (hi << 16);
    }
  }
  ok = mbar_wait(bar_mma, 0);
  if (__syncthreads_or(!ok)) goto fail;
  mma_done = 1;
  tc_fence_after();
  {
    uint8_t* qdst = sm + PP_QK + (row >> 6) * 16384;
#pragma unroll
    for (int cq = 0; cq < 4; ++cq)
      *reinterpret_cast<uint4*>(qdst + sw128_chunk(row & 63, 4 * wg + cq)) =
          make_uint4(qt[4 * cq], qt[4 * cq + 1], qt[4 * cq + 2], qt[4 * cq + 3]);
  }

  {
    float d1[32];
    tmem_ld32(trow + TM_D1 + 32 * wg, d1);
    if (row >= kCL && ((row - kCL) >> 5) == wg) {
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
      s_el[tid] = (tid == 0) ? expf(gL) : 0.0f;
    }
    if (row < kCL) {
      const int t = row;
      const float iq = s_iq[t], lt = s_l2[t];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int s = 32 * wg + i;
        d1[i] = (s <= t && t < n_c)
                    ? __fmul_rn(__fmul_rn(__fmul_rn(d1[i], iq), s_ik[s]), exp2f(__fsub_rn(lt, s_l2[s])))
                    : 0.0f;
      }
      store_half_hilo(sm + PP_P, sm + PP_P + 8192, t, wg, d1);
    } else {
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
  }
  __syncthreads();
  solve_unit_lower64(Am, Tm, Xs, tid);

  // T_W (into the A region) and T_U (over T itself), hi/lo bf16 tiles: every
  // thread takes its part of T into registers before any tile is written
  {
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
    __syncthreads();
    uint8_t* hi = which ? sm + PP_T : sm + PP_A;
    store_half_hilo(hi, hi + 8192, t, half, w);
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
        mma_bf16(tmem + TM_W, sdesc(sb + PP_QK + 8192 + ks * 2048, 16384, 1024),
                 sdesc(sb + PP_A + pass * 8192 + ks * 32, 16, 1024), id, (pass | ks) != 0);
#pragma unroll
    for (int pass = 0; pass < 2; ++pass)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + TM_U, sdesc(sb + PP_V + ks * 2048, 8192, 1024),
                 sdesc(sb + PP_T + pass * 8192 + ks * 32, 16, 1024), id, (pass | ks) != 0);
    mma_commit(bar_mma);
    ++mma_iss;
  }
  ok = mbar_wait(bar_mma, 1);
  if (__syncthreads_or(!ok)) goto fail;
  mma_done = 2;
  tc_fence_after();

  // staging in the workspace layout: W^T hi over V, W^T lo over the K halves
  // (rows 0..63 in atom 0's, 64..127 in atom 1's: the same swizzle, as a row
  // and its row - 64 share their low bits), U^T over A and T
  {
    float w[32];
    tmem_ld32(trow + TM_W + wg * 32, w);
    store_half_hilo(sm + PP_V, sm + PP_QK + 8192 + (row >> 6) * 8192, row, wg, w);
    tmem_ld32(trow + TM_U + wg * 32, w);
#pragma unroll
    for (int pq = 0; pq < 8; ++pq)
      *reinterpret_cast<float4*>(sm + PP_A + ut_piece(row, wg, pq)) =
          make_float4(w[4 * pq], w[4 * pq + 1], w[4 * pq + 2], w[4 * pq + 3]);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    bulk_store(item + CW_WT, sb + PP_V, 16384);                   // W^T hi
    bulk_store(item + CW_WT + 16384, sb + PP_QK, 8192);           // Q^T rows 0..63
    bulk_store(item + CW_WT + 24576, sb + PP_QK + 16384, 8192);   // Q^T rows 64..127
    bulk_store(item + CW_WT + 32768, sb + PP_QK + 8192, 8192);    // W^T lo rows 0..63
    bulk_store(item + CW_WT + 40960, sb + PP_QK + 24576, 8192);   // W^T lo rows 64..127
    bulk_store(item + CW_P, sb + PP_P, 16384);
    bulk_store(item + CW_UT, sb + PP_A, 32768);
    bulk_store(item + CW_VEC, smem_u32(s_cv), 768);
    bulk_store_commit_wait_read();
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
  return;

fail:
  if (tid == 0) {
    report(status, GDN_DEV_TIMEOUT);
    // let the copies and MMAs still in flight finish (each wait bounded)
    // before the shared and tensor memory are given up
    if (tma_done == 0) mbar_wait(bar_tma, 0);
    for (uint32_t k = mma_done; k < mma_iss; ++k) mbar_wait(bar_mma, k & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------ pass 2

// Shared memory of the chain (bytes from a 1024-aligned base).
constexpr uint32_t SQ_S = 0;          // S^T hi: atom a at a*16384 ([128][64]); lo at +32768
constexpr uint32_t SQ_K = 65536;      // TMA: K atom a at SQ_K + a*8192 ([64 t][64 i])
constexpr uint32_t SQ_WT = 81920;     // W^T hi | Q^T | W^T lo (from the workspace)
constexpr uint32_t SQ_P = 131072;     // P hi | lo (from the workspace)
constexpr uint32_t SQ_VN = 147456;    // Vn^T hi | lo ([128][64] each); then the output tile
constexpr uint32_t SQ_VP = 180224;    // V'^T hi | lo
constexpr uint32_t SQ_VEC = 212992;   // two slots of 768 bytes: cv[64] | co[64] | e^{gamma_L}
constexpr uint32_t kSeqSmem = SQ_VEC + 2 * 768 + 1024;

template <class ST>
__global__ void __launch_bounds__(kChunkThreads, 1)
chunk_seq_kernel(const __grid_constant__ CUtensorMap tm_qkv, Geom G, Batch B, Params P,
                 const char* __restrict__ ws, int ws_chunks, void* o, int out_f32, void* pages,
                 int32_t* status) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t bars[3];
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & 127;
  const int wg = tid >> 7;
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
  const char* items = ws + ((size_t)q.r * G.Hv + h) * ws_chunks * kChunkItemBytes;

  const uint32_t bar_a = smem_u32(&bars[0]), bar_b = smem_u32(&bars[1]),
                 bar_mma = smem_u32(&bars[2]);
  if (tid == 0) {
    mbar_init(bar_a, 1);
    mbar_init(bar_b, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const uint32_t sb = smem_u32(sm);
  // S^T; per chunk parity a [W S | Q S]^T slot of 128 columns and a (P Vn)^T slot of 64
  constexpr uint32_t TM_S = 0, TM_D4 = 128, TM_OP = 384;

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
  const int xk = G.Hk * kCD + kh * kCD;
  // phases issued (by thread 0) and completed, for the drain after a failed wait
  uint32_t a_iss = 0, a_done = 0, b_iss = 0, b_done = 0, m_iss = 0, m_done = 0;
  // operands read by MMA4/5 (and the chunk's factors)
  auto issue_a = [&](int c) {
    ++a_iss;
    const char* it = items + (size_t)c * kChunkItemBytes;
    mbar_expect_tx(bar_a, 49152 + 768);
    bulk_load(sb + SQ_WT, it + CW_WT, 49152, bar_a);
    bulk_load(sb + SQ_VEC + (c & 1) * 768, it + CW_VEC, 768, bar_a);
  };
  // operands read by MMA6/7
  auto issue_b = [&](int c) {
    ++b_iss;
    const int y = q.start + c * kCL;
    const char* it = items + (size_t)c * kChunkItemBytes;
    mbar_expect_tx(bar_b, 2 * 8192 + 16384);
#pragma unroll
    for (int a = 0; a < 2; ++a)
      tma_load_2d(sb + SQ_K + a * 8192, &tm_qkv, xk + 64 * a, y, bar_b);
    bulk_load(sb + SQ_P, it + CW_P, 16384, bar_b);
  };
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && nchunks > 0) {
    issue_a(0);
    issue_b(0);
  }

  uint32_t mma_count = 0;
  bool fail = false;
  auto wait_bar = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool ok = mbar_wait(bar, parity);
    const bool any_fail = __syncthreads_or(!ok);
    tc_fence_after();
    return !any_fail;
  };

  // U^T of chunk c for this thread's row and half. Issued only after the
  // chunk's last tensor-memory load before MMA4/5 completes: a wait for
  // tensor-memory loads also waits for global loads in flight.
  auto load_u = [&](int c, float* u) {
    const char* ut = items + (size_t)c * kChunkItemBytes + CW_UT;
#pragma unroll
    for (int pq = 0; pq < 8; ++pq) {
      const float4 v = ldg_nc_early(ut + ut_piece(row, wg, pq));
      u[4 * pq] = v.x; u[4 * pq + 1] = v.y; u[4 * pq + 2] = v.z; u[4 * pq + 3] = v.w;
    }
  };

  // outputs of chunk c: O[t][j] = scale (co_t (S^T Q^T)[j][t] + (Vn^T P^T)[j][t]),
  // by the second warpgroup alone (its four warps reach all 128 TMEM lanes),
  // so that they run while the first warpgroup's issuing thread queues the
  // next MMAs. Gathered as a [64][128] tile (the Vn^T region, which MMA6 of
  // chunk c has read) and written out as whole 16-byte row pieces. u_next,
  // when given, receives U^T of chunk c+1 after the last tensor-memory load.
  auto outputs = [&](int c, float* u_next) {
    const int n_c = min(kCL, q.len - c * kCL);
    const size_t R0 = (size_t)q.start + (size_t)c * kCL;
    const float* co = reinterpret_cast<const float*>(sm + SQ_VEC + (c & 1) * 768) + 64;
    float* of = reinterpret_cast<float*>(sm + SQ_VN);
    bf16* ob = reinterpret_cast<bf16*>(sm + SQ_VN);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float oq[32], op[32];
      tmem_ld32(trow + TM_D4 + (c & 1) * 128 + 64 + half * 32, oq);
      tmem_ld32(trow + TM_OP + (c & 1) * 64 + half * 32, op);
      if (half == 1 && u_next) load_u(c + 1, u_next);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = half * 32 + i;
        const float v = __fmul_rn(P.scale, __fmaf_rn(co[t], oq[i], op[i]));
        if (out_f32) of[t * kCD + row] = v;
        else ob[t * kCD + row] = __float2bfloat16_rn(v);
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const int lg = out_f32 ? 5 : 4;
    const int per_row = 1 << lg;
    const uint4* src = reinterpret_cast<const uint4*>(sm + SQ_VN);
    for (int idx = tid - 128; idx < (n_c << lg); idx += 128) {
      const int t = idx >> lg, piece = idx & (per_row - 1);
      const size_t row_off = ((R0 + t) * G.Hv + h) * G.Dv;
      uint4* dst = out_f32 ? reinterpret_cast<uint4*>(reinterpret_cast<float*>(o) + row_off)
                           : reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(o) + row_off);
      dst[piece] = src[t * per_row + piece];
    }
  };

  for (int c = 0; c < nchunks; ++c) {
    const int n_c = min(kCL, q.len - c * kCL);
    const float* vec = reinterpret_cast<const float*>(sm + SQ_VEC + (c & 1) * 768);
    if (!wait_bar(bar_a, c & 1)) { fail = true; break; }
    ++a_done;
    float u[32];   // U^T of this thread's row and half, loaded under MMA4/5
    // S^T hi/lo operand tiles, and e^{gamma_L} S^T back into TMEM for MMA7
    {
      const float eL = vec[128];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int cc = 2 * wg + c2;
        float v[32];
        tmem_ld32(trow + TM_S + cc * 32, v);
        store_half_hilo(sm + SQ_S + (cc >> 1) * 16384, sm + SQ_S + 32768 + (cc >> 1) * 16384, row,
                        cc & 1, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], eL);
        tmem_st32(trow + TM_S + cc * 32, v);
      }
      tmem_st_wait();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // MMA4/5 merged: [(W S)^T | (Q S)^T] = S^T [W^T | Q^T]; the W columns take
    // three hi/lo passes (S_hi W_hi, S_hi W_lo, S_lo W_hi), the Q columns two
    // (S_hi Q, S_lo Q), each in the one-kernel form's order
    if (tid == 0) {
      load_u(c, u);
      tc_fence_after();
      const uint32_t d4 = tmem + TM_D4 + (c & 1) * 128;
      const uint32_t id128 = idesc_bf16(128, 128, 0, 1), id64 = idesc_bf16(128, 64, 0, 1);
      auto a_s = [&](int lo, int ks) {
        return sdesc(sb + SQ_S + lo * 32768 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
      };
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(d4, a_s(0, ks), sdesc(sb + SQ_WT + ks * 2048, 16384, 1024), id128, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(d4, a_s(0, ks), sdesc(sb + SQ_WT + 32768 + ks * 2048, 16384, 1024), id64, 1u);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(d4, a_s(1, ks), sdesc(sb + SQ_WT + ks * 2048, 16384, 1024), id128, 1u);
      mma_commit(bar_mma);
      ++m_iss;
    }
    // the previous chunk's outputs while they run
    if (wg == 1 && c > 0) outputs(c - 1, u);
    else if (wg == 1 || tid != 0) load_u(c, u);
    if (!wait_bar(bar_mma, mma_count++ & 1)) { fail = true; break; }
    ++m_done;
    if (tid == 0 && c + 1 < nchunks) issue_a(c + 1);

    // Vn^T = U^T - (W S)^T ; V'^T = Vn^T diag(e^{gamma_L - gamma} / |k|)
    {
      float ws_[32];
      tmem_ld32(trow + TM_D4 + (c & 1) * 128 + wg * 32, ws_);
#pragma unroll
      for (int s = 0; s < 32; ++s) u[s] = __fsub_rn(u[s], ws_[s]);
      store_half_hilo(sm + SQ_VN, sm + SQ_VN + 16384, row, wg, u);
#pragma unroll
      for (int s = 0; s < 32; ++s) u[s] = __fmul_rn(u[s], vec[wg * 32 + s]);
      store_half_hilo(sm + SQ_VP, sm + SQ_VP + 16384, row, wg, u);
    }
    fence_async_smem();
    tc_fence_before();
    if (!wait_bar(bar_b, c & 1)) { fail = true; break; }
    ++b_done;
    if (n_c < kCL) {
      // K rows past the request's end belong to other requests: zero them
      for (int idx = tid; idx < (kCL - n_c) * 16; idx += kChunkThreads) {
        const int r = n_c + (idx >> 4), a = (idx >> 3) & 1, ch = idx & 7;
        *reinterpret_cast<uint4*>(sm + SQ_K + a * 8192 + r * 128 + ch * 16) =
            make_uint4(0, 0, 0, 0);
      }
      fence_async_smem();
      __syncthreads();
    }
    // MMA6: (P Vn)^T = Vn^T P^T ; MMA7: S^T += V'^T K
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id6 = idesc_bf16(128, 64, 0, 0);
      const int sel_v[3] = {0, 0, 1}, sel_p[3] = {0, 1, 0};
#pragma unroll
      for (int pass = 0; pass < 3; ++pass)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_OP + (c & 1) * 64,
                   sdesc(sb + SQ_VN + sel_v[pass] * 16384 + ks * 32, 16, 1024),
                   sdesc(sb + SQ_P + sel_p[pass] * 8192 + ks * 32, 16, 1024), id6,
                   (pass | ks) != 0);
      const uint32_t id7 = idesc_bf16(128, 128, 0, 1);
#pragma unroll
      for (int pass = 0; pass < 2; ++pass)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_S, sdesc(sb + SQ_VP + pass * 16384 + ks * 32, 16, 1024),
                   sdesc(sb + SQ_K + ks * 2048, 8192, 1024), id7, 1u);
      mma_commit(bar_mma);
      ++m_iss;
    }
    if (!wait_bar(bar_mma, mma_count++ & 1)) { fail = true; break; }
    ++m_done;
    if (tid == 0 && c + 1 < nchunks) issue_b(c + 1);
  }
  if (!fail && nchunks > 0 && wg == 1) outputs(nchunks - 1, nullptr);
  __syncthreads();

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
    for (uint32_t k = a_done; k < a_iss; ++k) mbar_wait(bar_a, k & 1);
    for (uint32_t k = b_done; k < b_iss; ++k) mbar_wait(bar_b, k & 1);
    for (uint32_t k = m_done; k < m_iss; ++k) mbar_wait(bar_mma, k & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t launch_chunk2(const void* tmap, const Geom& G, const Batch& B, const Params& P,
                          int state_bf16, int out_f32, const void* a, const void* b, void* o,
                          void* pages, void* ws, int ws_chunks, int32_t* status,
                          cudaStream_t stream) {
  const CUtensorMap& tm = *static_cast<const CUtensorMap*>(tmap);
  if (ws_chunks > 0) {
    cudaError_t e = ensure_smem_limit<chunk_prep_kernel>((int)kPrepSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(chunk_prep_kernel, dim3(ws_chunks, G.Hv, B.R), dim3(kChunkThreads), kPrepSmem,
                   stream, tm, G, B, P, static_cast<const bf16*>(a), static_cast<const bf16*>(b),
                   static_cast<char*>(ws), ws_chunks, status);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(G.Hv, B.R);
  if (state_bf16) {
    cudaError_t e = ensure_smem_limit<chunk_seq_kernel<bf16>>((int)kSeqSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(chunk_seq_kernel<bf16>, grid, dim3(kChunkThreads), kSeqSmem, stream, tm, G, B,
                   P, static_cast<const char*>(ws), ws_chunks, o, out_f32, pages, status);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = ensure_smem_limit<chunk_seq_kernel<float>>((int)kSeqSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(chunk_seq_kernel<float>, grid, dim3(kChunkThreads), kSeqSmem, stream, tm, G, B,
                   P, static_cast<const char*>(ws), ws_chunks, o, out_f32, pages, status);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace gdn
