// Combine: y[t] = shared output of t + sum_j g[t,j] * (output of t's j-th expert), fp32
// accumulation in that order, one rounding to bf16. The pages: the combine step sends expert
// outputs back, restores token order and sums them with the routing weights
// ("第 6 章 超節點", 6.2.6 and 6.4.1); on one GPU it is a gather from the slot-ordered outputs.
#include "internal.h"

namespace moe {
namespace {

// One thread per 4 consecutive output features of one token: 16-byte loads of every term.
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ y_perm,
                                                 const int32_t* __restrict__ inv_slot,
                                                 const float* __restrict__ topk_w, int T, int k,
                                                 int d, int n_shared, uint16_t* __restrict__ y,
                                                 int* status) {
  // small batches (a few blocks, latency-bound): warm L2 and this SM's address translations for
  // what the block reads after the wait
  if (T * k <= 256) {
    prefetch_l2_span(inv_slot, (size_t)T * k * 4);
    prefetch_l2_span(topk_w, (size_t)T * k * 4);
    prefetch_l2_pages(y_perm, (size_t)T * (k + n_shared) * d * 4);
  }
  pdl_wait_then_release();
  const int d4 = d >> 2;
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long)T * d4) return;
  const int t = (int)(i / d4);
  const int c = (int)(i % d4) * 4;
  const long routed = (long)T * k;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (n_shared) acc = __ldg(reinterpret_cast<const float4*>(y_perm + (routed + t) * d + c));
  for (int j = 0; j < k; ++j) {
    const int s = __ldg(inv_slot + (long)t * k + j);
    const float g = __ldg(topk_w + (long)t * k + j);
    if (s < 0 || s >= routed) {
      record_error(status, MOE_ERR_DEVICE_BOUNDS);
      continue;
    }
    const float4 v = __ldg(reinterpret_cast<const float4*>(y_perm + (long)s * d + c));
    acc.x = __fmaf_rn(g, v.x, acc.x);
    acc.y = __fmaf_rn(g, v.y, acc.y);
    acc.z = __fmaf_rn(g, v.z, acc.z);
    acc.w = __fmaf_rn(g, v.w, acc.w);
  }
  uint2 out;
  out.x = (uint32_t)f32_to_bf16_rn(acc.x) | ((uint32_t)f32_to_bf16_rn(acc.y) << 16);
  out.y = (uint32_t)f32_to_bf16_rn(acc.z) | ((uint32_t)f32_to_bf16_rn(acc.w) << 16);
  *reinterpret_cast<uint2*>(y + (long)t * d + c) = out;
}

}  // namespace

cudaError_t launch_combine(const moe_shape& s, const float* y_perm, const int32_t* inv_slot,
                           const float* topk_w, uint16_t* y, int* status, cudaStream_t st) {
  const long n = (long)s.T * (s.d / 4);
  if (n == 0) return cudaSuccess;
  const cudaError_t e = launch_pdl(k_combine, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st,
                                   y_perm, inv_slot, topk_w, s.T, s.k, s.d, s.n_shared, y, status);
  count_launches(1);
  return e;
}

}  // namespace moe
