// The router's selection of one token, shared by the top-k kernel (router.cu) and the fused
// decode front of moe_forward (ffn.cu), so both give the same bits: the k largest fp32 logits
// (ties to the lower expert index), listed by descending logit, and the gate weights
// softmax(l_chosen) = exp(l_j - l_max) / sum over the k chosen.
#pragma once

#include <stdint.h>

namespace moe {

// (value desc, index asc): is (la, ea) ranked before (lb, eb)?
__device__ __forceinline__ bool ranks_before(float la, int ea, float lb, int eb) {
  return la > lb || (la == lb && ea < eb);
}

// One warp, one token: lt holds the token's E logits (E <= 1024); lane j of the warp ends up
// with choice j (j < k): k rounds of warp arg-max (lane j holds experts j, j+32, ...), then the
// weights. Lanes j < k write idx_out[j] and w_out[j] (global or shared memory).
__device__ __forceinline__ void warp_topk_token(const float* lt, int E, int k,
                                                int32_t* idx_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  float l[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) l[m] = (lane + 32 * m < E) ? lt[lane + 32 * m] : -INFINITY;
  uint32_t taken = 0;
  float my_l = -INFINITY;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bl = -INFINITY;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      const int e = lane + 32 * m;
      if (e < E && !((taken >> m) & 1u) && ranks_before(l[m], e, bl, be)) {
        bl = l[m];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float ol = __shfl_xor_sync(0xffffffffu, bl, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ranks_before(ol, oe, bl, be)) {
        bl = ol;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_l = bl;
      my_e = be;
    }
  }
  const float lmax = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = lane < k ? expf(my_l - lmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    idx_out[lane] = my_e;
    w_out[lane] = ex / sum;
  }
}

}  // namespace moe
