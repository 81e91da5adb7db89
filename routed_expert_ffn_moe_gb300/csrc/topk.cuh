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

// Order-preserving 32-bit key of a logit: keys compare as the values do (-0 as +0), so the
// ranking (value desc, index asc) is (key desc, index asc). NaN keys below every number.
__device__ __forceinline__ uint32_t logit_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (v != v) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The logit of a key (exact for every number; -0 comes back as +0).
__device__ __forceinline__ float key_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// The gate weights of a token's k choices, lane j holding choice j's key: softmax over the k
// chosen logits, exp(l_j - l_max) / sum (l_max = choice 0's). Lanes j < k write their choice.
__device__ __forceinline__ void write_choice(int lane, int k, uint32_t my_key, int my_e,
                                             int32_t* idx_out, float* w_out) {
  const float my_l = lane < k ? key_logit(my_key) : -INFINITY;
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

// One warp, one token: lt holds the token's E logits (E <= 1024); lane j of the warp ends up
// with choice j (j < k), then the weights. Lane j holds experts j, j+32, ...; each of the k
// rounds takes the warp's best (the largest key by one warp max-reduction, the lowest expert
// index among equal keys by a min-reduction) and the lane that gave it moves to its next best.
// Up to 256 experts a lane holds 8, sorted once (a 19-comparator network on 64-bit (key,
// expert) words), so its next best is the next entry; above that it looks for its next best
// among its (up to 32) remaining ones.
// Lanes j < k write idx_out[j] and w_out[j] (global or shared memory).
__device__ __forceinline__ void warp_topk_token(const float* lt, int E, int k,
                                                int32_t* idx_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  uint32_t my_key = 0;
  int my_e = 0x7FFFFFFF;
  if (E <= 256) {
    // v[m] = key << 32 | ~expert (0 for no expert): one 64-bit order, key desc then expert asc.
    // The 8 loads go out together (indexes clamped into the row), then the branch-free network.
    float l[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) l[m] = lt[min(lane + 32 * m, E - 1)];
    uint64_t v[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const uint32_t e = (uint32_t)(lane + 32 * m);
      v[m] = e < (uint32_t)E ? ((uint64_t)logit_key(l[m]) << 32) | (uint64_t)(~e) : 0ull;
    }
    auto cx = [&](int a, int b) {
      const uint64_t hi = v[a] > v[b] ? v[a] : v[b];
      const uint64_t lo = v[a] > v[b] ? v[b] : v[a];
      v[a] = hi;
      v[b] = lo;
    };
    cx(0, 2); cx(1, 3); cx(4, 6); cx(5, 7);
    cx(0, 4); cx(1, 5); cx(2, 6); cx(3, 7);
    cx(0, 1); cx(2, 3); cx(4, 5); cx(6, 7);
    cx(2, 4); cx(3, 5);
    cx(1, 4); cx(3, 6);
    cx(1, 2); cx(3, 4); cx(5, 6);
    for (int j = 0; j < k; ++j) {
      const bool has = v[0] != 0ull;
      const uint32_t hk = (uint32_t)(v[0] >> 32);
      const uint32_t top = __reduce_max_sync(0xffffffffu, has ? hk : 0u);
      const uint32_t cand = (has && hk == top) ? ~(uint32_t)v[0] : 0xFFFFFFFFu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
      if (lane == j) {
        my_key = top;
        my_e = win < (uint32_t)E ? (int)win : 0x7FFFFFFF;
      }
      const bool mine = win < (uint32_t)E && (int)(win & 31u) == lane;
#pragma unroll
      for (int m = 0; m < 7; ++m) v[m] = mine ? v[m + 1] : v[m];
      v[7] = mine ? 0ull : v[7];
    }
  } else {
    uint32_t key[32];
    uint32_t avail = 0;  // bit m: expert lane + 32 m exists and is not taken
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      const bool in = lane + 32 * m < E;
      key[m] = in ? logit_key(lt[lane + 32 * m]) : 0u;
      avail |= in ? (1u << m) : 0u;
    }
    // this lane's best: largest key, the lowest m among equal keys
    uint32_t bk = 0;
    int bm = -1;
#pragma unroll
    for (int m = 0; m < 32; ++m)
      if (((avail >> m) & 1u) && (bm < 0 || key[m] > bk)) {
        bk = key[m];
        bm = m;
      }
    for (int j = 0; j < k; ++j) {
      const uint32_t top = __reduce_max_sync(0xffffffffu, bm >= 0 ? bk : 0u);
      const uint32_t cand = (bm >= 0 && bk == top) ? (uint32_t)(lane + 32 * bm) : 0xFFFFFFFFu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
      if (lane == j) {
        my_key = top;
        my_e = win < (uint32_t)E ? (int)win : 0x7FFFFFFF;
      }
      if (win < (uint32_t)E && (int)(win & 31u) == lane) {
        avail &= ~(1u << (win >> 5));
        bk = 0;
        bm = -1;
#pragma unroll
        for (int m = 0; m < 32; ++m)
          if (((avail >> m) & 1u) && (bm < 0 || key[m] > bk)) {
            bk = key[m];
            bm = m;
          }
      }
    }
  }
  write_choice(lane, k, my_key, my_e, idx_out, w_out);
}

}  // namespace moe
