// Exhaustive check of the conv's SiLU quotient step (gdn::silu_negquot in
// common.cuh): for every float t in [0, 1], with d = fl(1 + t) formed as the
// conv forms it, the step's -t/d must equal the IEEE quotient bit for bit.
// (At t = 0 the two zeros may differ in sign; the SiLU then forms
// c - a q = fma(a, -q, c) with c >= +0, which is the same for either zero,
// so zeros of either sign count as equal.) Prints the number of differences
// and the first few t (bit patterns).
#include <cstdio>
#include <cstdint>

#include "common.cuh"

__device__ unsigned long long g_diff;
__device__ unsigned int g_first[8];
__device__ unsigned int g_nfirst;

__global__ void check(uint32_t hi) {
  const uint32_t stride = gridDim.x * blockDim.x;
  // pairs (b, b + 1): the step takes two values at once
  for (uint32_t b = 2 * (blockIdx.x * blockDim.x + threadIdx.x); b <= hi; b += 2 * stride) {
    const uint32_t b1 = (b + 1 <= hi) ? b + 1 : b;
    const float2 t = make_float2(__uint_as_float(b), __uint_as_float(b1));
    const float2 nt = make_float2(-t.x, -t.y);
    const float2 nd = __fadd2_rn(nt, make_float2(-1.0f, -1.0f));
    const float2 q = gdn::silu_negquot(nt, nd);
    const float ref[2] = {__fdiv_rn(nt.x, -nd.x), __fdiv_rn(nt.y, -nd.y)};
    const float got[2] = {q.x, q.y};
    const uint32_t bb[2] = {b, b1};
    for (int e = 0; e < 2; ++e)
      if (__float_as_uint(got[e]) != __float_as_uint(ref[e]) &&
          !(got[e] == 0.0f && ref[e] == 0.0f)) {
        atomicAdd(&g_diff, 1ull);
        const unsigned int i = atomicAdd(&g_nfirst, 1u);
        if (i < 8) g_first[i] = bb[e];
      }
  }
}

int main() {
  const uint32_t hi = 0x3f800000u;   // 1.0f; b = 0 is t = +0
  check<<<152 * 8, 256>>>(hi);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    printf("cuda error\n");
    return 2;
  }
  unsigned long long diff = 0;
  unsigned int first[8] = {}, nfirst = 0;
  cudaMemcpyFromSymbol(&diff, g_diff, sizeof diff);
  cudaMemcpyFromSymbol(first, g_first, sizeof first);
  cudaMemcpyFromSymbol(&nfirst, g_nfirst, sizeof nfirst);
  printf("values %u differences %llu", hi + 1, diff);
  for (unsigned int i = 0; i < (nfirst < 8 ? nfirst : 8); ++i) printf(" %08x", first[i]);
  printf("\n");
  return 0;
}
