// Pieces shared by the two forms of the chunked prefill (sm_103a): the chunk
// geometry, the bf16 hi/lo operand split and the 64 x 64 unit-lower-
// triangular solve on the CUDA cores. chunk.cu holds the one-kernel form,
// chunk2.cu the two-pass form (a chunk-parallel pre-pass into a workspace,
// then the state chain).
#pragma once

#include "common.cuh"
#include "umma.cuh"

namespace gdn {

using namespace umma;

constexpr int kCL = 64;               // tokens per chunk
constexpr int kCD = 128;              // Dk = Dv
constexpr int kChunkThreads = 256;      // two warpgroups; warps w and w+4 share TMEM lanes
constexpr float kLog2e = 1.4426950408889634f;

// A pair of fp32 values as two bf16x2 words (element 0 in the low half):
// hi = each value rounded to bf16, lo = the remainder rounded to bf16. One
// paired conversion per word.
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 hb = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(hb);
  const __nv_bfloat162 lb = __floats2bfloat162_rn(__fsub_rn(x0, hf.x), __fsub_rn(x1, hf.y));
  hi = *reinterpret_cast<const uint32_t*>(&hb);
  lo = *reinterpret_cast<const uint32_t*>(&lb);
}

// Write 64 fp32 values as row `row` of two [rows][64] SW128 bf16 tiles: the
// bf16 rounding (hi) and the rounding of the remainder (lo).
__device__ __forceinline__ void store_row_hilo(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                               const float* v) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      split_pair(v[ch * 8 + 2 * e], v[ch * 8 + 2 * e + 1], h[e], l[e]);
    }
    const uint32_t off = sw128_chunk(row, ch);
    *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// The same for 32 values: chunks 4*half .. 4*half+3 of the row.
__device__ __forceinline__ void store_half_hilo(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                                int half, const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      split_pair(v[c * 8 + 2 * e], v[c * 8 + 2 * e + 1], h[e], l[e]);
    }
    const uint32_t off = sw128_chunk(row, 4 * half + c);
    *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// A and T ([64][64] fp32 in shared memory) keep the 16-byte chunk q of row r
// at chunk q ^ (r & 15): threads that each own a row and touch the same
// columns then hit different banks (a plain 256-byte row stride sent all of
// them to the same four banks).
__device__ __forceinline__ int mat_idx(int r, int c) {
  return (r << 6) | ((((c >> 2) ^ (r & 15)) << 2) | (c & 3));
}

// acc += a4[e] * M[k0 + e][c0 .. c0+3] for e = 0..3 (M in the mat_idx layout).
__device__ __forceinline__ void fma4_row(float4& acc, float4 a4, const float* M, int k0, int c0) {
  const float ak[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float4 t4 = *reinterpret_cast<const float4*>(&M[mat_idx(k0 + e, c0)]);
    acc.x = __fmaf_rn(ak[e], t4.x, acc.x);
    acc.y = __fmaf_rn(ak[e], t4.y, acc.y);
    acc.z = __fmaf_rn(ak[e], t4.z, acc.z);
    acc.w = __fmaf_rn(ak[e], t4.w, acc.w);
  }
}

// acc += t4[e] * X[m0 + e][c0 .. c0+3] for e = 0..3 (X a [16][16] scratch block).
__device__ __forceinline__ void fma4_scratch(float4& acc, float4 t4, const float* X, int m0, int c0) {
  const float tk[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float4 x4 = *reinterpret_cast<const float4*>(&X[(m0 + e) * 16 + c0]);
    acc.x = __fmaf_rn(tk[e], x4.x, acc.x);
    acc.y = __fmaf_rn(tk[e], x4.y, acc.y);
    acc.z = __fmaf_rn(tk[e], x4.z, acc.z);
    acc.w = __fmaf_rn(tk[e], x4.w, acc.w);
  }
}

// T = (I + A)^-1 for a strictly lower 64 x 64 A (mat_idx layout): the four
// 16 x 16 diagonal blocks by forward substitution (one thread per block
// column), then the two 32 x 32 diagonal halves, [[T_a, 0], [T_c, T_b]] with
// T_c = -T_b A_c T_a, then the lower-left 32 x 32 block the same way; each
// thread forms 4 adjacent outputs from 16-byte loads. Xs: 4 x 256 floats of
// scratch. All threads of the CTA call this.
__device__ __forceinline__ void solve_unit_lower64(const float* Am, float* Tm, float* Xs, int tid) {
  if (tid < 64) {
    // the block's row r + 1 is loaded (four 16-byte loads) while row r is
    // solved, so no multiply-add waits on its own load
    const int b = tid >> 4, cc = tid & 15, R0 = 16 * b;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) x[r] = (r == cc) ? 1.0f : 0.0f;
    float4 nxt[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      nxt[q] = *reinterpret_cast<const float4*>(&Am[mat_idx(R0 + 1, R0 + 4 * q)]);
#pragma unroll
    for (int r = 1; r < 16; ++r) {
      float a[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[4 * q] = nxt[q].x; a[4 * q + 1] = nxt[q].y; a[4 * q + 2] = nxt[q].z; a[4 * q + 3] = nxt[q].w;
      }
      if (r + 1 < 16) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          nxt[q] = *reinterpret_cast<const float4*>(&Am[mat_idx(R0 + r + 1, R0 + 4 * q)]);
      }
      float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
      for (int k = 0; k < r; k += 2) {
        acc0 = __fmaf_rn(a[k], x[k], acc0);
        if (k + 1 < r) acc1 = __fmaf_rn(a[k + 1], x[k + 1], acc1);
      }
      if (r > cc) x[r] = -__fadd_rn(acc0, acc1);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) Tm[mat_idx(R0 + r, R0 + cc)] = x[r];
  } else {
    // blocks above the diagonal are zero
    for (int idx = tid - 64; idx < 6 * 256; idx += kChunkThreads - 64) {
      const int blk = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
      const int bi = (blk < 3) ? 0 : (blk < 5 ? 1 : 2);
      const int bj = (blk < 3) ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      Tm[mat_idx(16 * bi + r, 16 * bj + cc)] = 0.0f;
    }
  }
  __syncthreads();
  // Round A: the blocks next to the diagonal inside each 32 x 32 half,
  // T_10 = -T_11 (A_10 T_00) and T_32 = -T_33 (A_32 T_22); thread ->
  // (half, row r, columns 4q .. 4q+3).
  if (tid < 128) {
    const int hf = tid >> 6, bi = 2 * hf + 1, bj = 2 * hf, r = (tid >> 2) & 15, q = tid & 3;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int kb = 16 * bj + 4 * it;
      const float4 a4 = *reinterpret_cast<const float4*>(&Am[mat_idx(16 * bi + r, kb)]);
      fma4_row(acc, a4, Tm, kb, 16 * bj + 4 * q);
    }
    *reinterpret_cast<float4*>(&Xs[(hf << 8) + r * 16 + 4 * q]) = acc;
  }
  __syncthreads();
  if (tid < 128) {
    const int hf = tid >> 6, bi = 2 * hf + 1, bj = 2 * hf, r = (tid >> 2) & 15, q = tid & 3;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int m0 = 0; m0 < 16; m0 += 4) {
      const float4 t4 = *reinterpret_cast<const float4*>(&Tm[mat_idx(16 * bi + r, 16 * bi + m0)]);
      fma4_scratch(acc, t4, Xs + (hf << 8), m0, 4 * q);
    }
    *reinterpret_cast<float4*>(&Tm[mat_idx(16 * bi + r, 16 * bj + 4 * q)]) =
        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  __syncthreads();
  // Round B: the lower-left 32 x 32 block, T_21 = -T_22 (A_21 T_11) in
  // 16 x 16 blocks (i, j), i in {2, 3}, j in {0, 1}; thread -> (block,
  // row r, columns 4q .. 4q+3), one block per pair of warps.
  {
    const int blk = tid >> 6, i = 2 + (blk >> 1), j = blk & 1, r = (tid >> 2) & 15, q = tid & 3;
    // X_ij = sum_{k=16j}^{31} A_ik T_kj (16 or 32 terms), two partial sums
    float4 acc0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), acc1 = acc0;
    const int nit = 8 - 4 * j;
#pragma unroll
    for (int it = 0; it < 8; it += 2) {
      if (it < nit) {
        const int kb0 = 16 * j + 4 * it, kb1 = kb0 + 4;
        const float4 a0 = *reinterpret_cast<const float4*>(&Am[mat_idx(16 * i + r, kb0)]);
        const float4 a1 = *reinterpret_cast<const float4*>(&Am[mat_idx(16 * i + r, kb1)]);
        fma4_row(acc0, a0, Tm, kb0, 16 * j + 4 * q);
        fma4_row(acc1, a1, Tm, kb1, 16 * j + 4 * q);
      }
    }
    *reinterpret_cast<float4*>(&Xs[(blk << 8) + r * 16 + 4 * q]) =
        make_float4(__fadd_rn(acc0.x, acc1.x), __fadd_rn(acc0.y, acc1.y),
                    __fadd_rn(acc0.z, acc1.z), __fadd_rn(acc0.w, acc1.w));
  }
  __syncthreads();
  {
    // T_ij = -sum_{kb=2}^{i} T_{i,kb} X_{kb,j} (T_22, T_32, T_33; X_{kb,j} is
    // scratch block ((kb - 2) << 1) | j)
    const int blk = tid >> 6, i = 2 + (blk >> 1), j = blk & 1, r = (tid >> 2) & 15, q = tid & 3;
    float4 acc0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), acc1 = acc0;
#pragma unroll
    for (int kb = 2; kb < 4; ++kb) {
      if (kb <= i) {
        const float* xb = Xs + ((((kb - 2) << 1) | j) << 8);
#pragma unroll
        for (int m0 = 0; m0 < 16; m0 += 8) {
          const float4 t0 = *reinterpret_cast<const float4*>(&Tm[mat_idx(16 * i + r, 16 * kb + m0)]);
          const float4 t1 = *reinterpret_cast<const float4*>(&Tm[mat_idx(16 * i + r, 16 * kb + m0 + 4)]);
          fma4_scratch(acc0, t0, xb, m0, 4 * q);
          fma4_scratch(acc1, t1, xb, m0 + 4, 4 * q);
        }
      }
    }
    *reinterpret_cast<float4*>(&Tm[mat_idx(16 * i + r, 16 * j + 4 * q)]) =
        make_float4(-__fadd_rn(acc0.x, acc1.x), -__fadd_rn(acc0.y, acc1.y),
                    -__fadd_rn(acc0.z, acc1.z), -__fadd_rn(acc0.w, acc1.w));
  }
  __syncthreads();
}

}  // namespace gdn
