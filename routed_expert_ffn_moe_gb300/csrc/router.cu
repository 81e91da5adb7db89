// Router: logits in a fixed fp32 order, top-k selection, gate weights.
//
// The pages: the router scores every routed expert for each token and keeps the top-k, its
// compute is small and its product is the sparse metadata for dispatch ("DeepSeek-V4-Pro on
// NVIDIA H200", 0.2.2 step D4); V4 uses learned soft routing ("CANN DeepSeek-V4推理优化", MoE
// 专家模型规格). Ascend fuses the gate into one "GatingTopK" kernel (same page, 融合Kernel);
// here the logits GEMM and the selection are two kernels so the selection can see all E
// logits of a token at once.
#include <mutex>

#include "internal.h"

namespace moe {
namespace {

// One warp computes TT tokens x TE experts. Lane j owns the 8-element chunks j, j+32, ... of
// the hidden dimension and accumulates them element by element with fused multiply-add; the
// 32 lane sums are then combined by an xor butterfly. This is the library's defined order for
// the logit, so the top-k choice is reproducible bit for bit.
template <int TT, int TE, int UNROLL = 4>
__global__ void __launch_bounds__(128) k_router_logits(const uint16_t* __restrict__ x,
                                                       const uint16_t* __restrict__ wg,
                                                       const float* __restrict__ bias, int T,
                                                       int d, int E, float* __restrict__ logits) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int n_et = (E + TE - 1) / TE;
  const int t0 = (warp / n_et) * TT, e0 = (warp % n_et) * TE;
  if (t0 >= T) return;
  float acc[TT][TE];
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int e = 0; e < TE; ++e) acc[t][e] = 0.f;
  const int chunks = d >> 3;
  const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll UNROLL
  for (int c = lane; c < chunks; c += 32) {
    uint4 xv[TT], wv[TE];
#pragma unroll
    for (int t = 0; t < TT; ++t)
      xv[t] = (t0 + t < T) ? ldg_u4(x + (size_t)(t0 + t) * d + 8 * c) : zero;
#pragma unroll
    for (int e = 0; e < TE; ++e)
      wv[e] = (e0 + e < E) ? ldg_u4(wg + (size_t)(e0 + e) * d + 8 * c) : zero;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float xf[TT], wf[TE];
#pragma unroll
      for (int t = 0; t < TT; ++t) xf[t] = bf16x8_elem(xv[t], i);
#pragma unroll
      for (int e = 0; e < TE; ++e) wf[e] = bf16x8_elem(wv[e], i);
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int e = 0; e < TE; ++e) acc[t][e] = __fmaf_rn(xf[t], wf[e], acc[t][e]);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
      for (int e = 0; e < TE; ++e)
        acc[t][e] = __fadd_rn(acc[t][e], __shfl_xor_sync(0xffffffffu, acc[t][e], off));
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int e = 0; e < TE; ++e)
      if (((t * TE + e) & 31) == lane && t0 + t < T && e0 + e < E) {
        const float l = bias ? __fadd_rn(acc[t][e], bias[e0 + e]) : acc[t][e];
        logits[(size_t)(t0 + t) * E + e0 + e] = l;
      }
}

// Same per-logit order as k_router_logits, for batches of 64+ tokens: a warp owns TT tokens x
// TE experts and issues the fused multiply-adds of expert pairs as one packed two-lane FMA
// (__ffma2_rn: two independent fp32 fmas, each rounded to nearest). Every accumulator still sees
// exactly the sequence of the defined order, so the logits are bit-identical.
template <int TT, int TE>
__global__ void __launch_bounds__(256) k_router_logits_x2(const uint16_t* __restrict__ x,
                                                          const uint16_t* __restrict__ wg,
                                                          const float* __restrict__ bias, int T,
                                                          int d, int E,
                                                          float* __restrict__ logits) {
  pdl_wait_then_release();
  static_assert(TE % 2 == 0, "experts are paired");
  // A block of 8 warps covers 4 token tiles x 2 expert tiles, so both operands are reused
  // through L1 by the warps that share them.
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int n_et = (E + TE - 1) / TE;
  const int n_eb = (n_et + 1) / 2;
  const int bt = blockIdx.x / n_eb, be = blockIdx.x - bt * n_eb;
  const int et = 2 * be + (w & 1);
  const int t0 = (4 * bt + (w >> 1)) * TT, e0 = et * TE;
  if (t0 >= T || et >= n_et) return;
  float2 acc[TT][TE / 2];
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int q = 0; q < TE / 2; ++q) acc[t][q] = make_float2(0.f, 0.f);
  const int chunks = d >> 3;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int c = lane; c < chunks; c += 32) {
    uint4 xv[TT], wv[TE];
#pragma unroll
    for (int t = 0; t < TT; ++t)
      xv[t] = (t0 + t < T) ? ldg_u4(x + (size_t)(t0 + t) * d + 8 * c) : zero;
#pragma unroll
    for (int e = 0; e < TE; ++e)
      wv[e] = (e0 + e < E) ? ldg_u4(wg + (size_t)(e0 + e) * d + 8 * c) : zero;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 w2[TE / 2];
#pragma unroll
      for (int q = 0; q < TE / 2; ++q)
        w2[q] = make_float2(bf16x8_elem(wv[2 * q], i), bf16x8_elem(wv[2 * q + 1], i));
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float xf = bf16x8_elem(xv[t], i);
        const float2 x2 = make_float2(xf, xf);
#pragma unroll
        for (int q = 0; q < TE / 2; ++q) acc[t][q] = __ffma2_rn(x2, w2[q], acc[t][q]);
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
      for (int q = 0; q < TE / 2; ++q) {
        acc[t][q].x = __fadd_rn(acc[t][q].x, __shfl_xor_sync(0xffffffffu, acc[t][q].x, off));
        acc[t][q].y = __fadd_rn(acc[t][q].y, __shfl_xor_sync(0xffffffffu, acc[t][q].y, off));
      }
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int e = 0; e < TE; ++e)
      if (((t * TE + e) & 31) == lane && t0 + t < T && e0 + e < E) {
        const float a = (e & 1) ? acc[t][e >> 1].y : acc[t][e >> 1].x;
        logits[(size_t)(t0 + t) * E + e0 + e] = bias ? __fadd_rn(a, bias[e0 + e]) : a;
      }
}

// (value desc, index asc): is (la, ea) ranked before (lb, eb)?
__device__ __forceinline__ bool ranks_before(float la, int ea, float lb, int eb) {
  return la > lb || (la == lb && ea < eb);
}

// One warp per token: k rounds of warp-wide arg-max over the E logits (lane j holds experts
// j, j+32, ...), then the gate weights softmax(l_chosen) = exp(l_j - l_max) / sum.
__global__ void __launch_bounds__(256) k_router_topk(const float* __restrict__ logits, int T,
                                                     int E, int k, int32_t* __restrict__ topk_idx,
                                                     float* __restrict__ topk_w) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* lt = logits + (size_t)t * E;
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
    topk_idx[(size_t)t * k + lane] = my_e;
    topk_w[(size_t)t * k + lane] = ex / sum;
  }
}

// Hash routing: one warp per token. Lane j < k takes expert tid2eid[token_ids[t]][j] and its
// logit; the gate weights are exp(l_j - l_max) / sum over those k, computed as k_router_topk
// computes them for the soft choice (so a table holding the soft choices gives the same bits).
// A token id or table entry out of range is recorded in the status word and replaced by 0.
__global__ void __launch_bounds__(256) k_router_hash(const float* __restrict__ logits,
                                                     const int32_t* __restrict__ token_ids,
                                                     const int32_t* __restrict__ tid2eid,
                                                     int vocab, int T, int E, int k,
                                                     int32_t* __restrict__ topk_idx,
                                                     float* __restrict__ topk_w, int* status) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  int tid = __ldg(token_ids + t);
  if (tid < 0 || tid >= vocab) {
    if (lane == 0) record_error(status, MOE_ERR_DEVICE_BOUNDS);
    tid = 0;
  }
  int e = 0;
  float l = -INFINITY;
  if (lane < k) {
    e = __ldg(tid2eid + (size_t)tid * k + lane);
    if (e < 0 || e >= E) {
      record_error(status, MOE_ERR_DEVICE_BOUNDS);
      e = 0;
    }
    l = logits[(size_t)t * E + e];
  }
  float lmax = l;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
  const float ex = lane < k ? expf(l - lmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = e;
    topk_w[(size_t)t * k + lane] = ex / sum;
  }
}

template <int TT, int TE, int UNROLL = 4>
cudaError_t launch_logits(const uint16_t* x, const uint16_t* wg, const float* bias, int T, int d,
                          int E, float* logits, cudaStream_t st) {
  const long warps = (long)((T + TT - 1) / TT) * ((E + TE - 1) / TE);
  const long blocks = (warps + 3) / 4;
  if constexpr (TT == 1) {
    return launch_pdl(k_router_logits<TT, TE, UNROLL>, dim3((unsigned)blocks), dim3(128), 0, st, x, wg,
                      bias, T, d, E, logits);
  } else {
    const long n_tt = (T + TT - 1) / TT, n_eb = ((E + TE - 1) / TE + 1) / 2;
    return launch_pdl(k_router_logits_x2<TT, TE>, dim3((unsigned)(((n_tt + 3) / 4) * n_eb)),
                      dim3(256), 0, st, x, wg, bias, T, d, E, logits);
  }
  return cudaGetLastError();
}

// Tile shape by batch: few tokens -> few experts per warp (more warps in flight for the
// latency-bound case); 64+ tokens -> register-tiled packed-FMA kernel.
cudaError_t launch_logits_for(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                              const float* bias, float* logits, cudaStream_t st) {
  // At these batch sizes the logits are latency-bound: one or two experts a warp (more warps in
  // flight) and eight chunk loads in flight a lane (measured: FP8 T=1 layer 127.7 -> 124.2 us,
  // MXFP4 T=8 272.9 -> 266.3 us).
  if (s.T <= 8) return launch_logits<1, 1, 8>(x, wg, bias, s.T, s.d, s.E, logits, st);
  if (s.T <= 32) return launch_logits<1, 2, 8>(x, wg, bias, s.T, s.d, s.E, logits, st);
  if (s.T < 64) return launch_logits<1, 8>(x, wg, bias, s.T, s.d, s.E, logits, st);
  return launch_logits<4, 8>(x, wg, bias, s.T, s.d, s.E, logits, st);
}

}  // namespace

// ---- router without a caller-provided workspace ------------------------------------------
// The logits scratch of moe_route_noalloc lives in this fixed device array, one copy per GPU
// that loads the library, held until the process exits. Every call shares it: each call
// overwrites the first T*E entries before reading them (nothing in it must start at zero), and
// calls that overlap on the GPU race on it.
constexpr size_t kNoAllocLogits = size_t(1) << 20;  // fp32 logits: 4 MiB
static __device__ __align__(256) float g_noalloc_logits[kNoAllocLogits];

size_t route_noalloc_max_logits() { return kNoAllocLogits; }

// Device address of the array for the current device, looked up once per device (the first
// call on a device does this set-up).
static cudaError_t noalloc_logits_ptr(float** out) {
  static std::mutex mu;
  static float* ptrs[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_logits);
    if (e != cudaSuccess) return e;
    ptrs[dev] = static_cast<float*>(p);
  }
  *out = ptrs[dev];
  return cudaSuccess;
}

cudaError_t launch_route_noalloc(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                 const float* bias, int32_t* topk_idx, float* topk_w,
                                 cudaStream_t st) {
  float* logits = nullptr;
  cudaError_t e = noalloc_logits_ptr(&logits);
  if (e != cudaSuccess || s.T == 0) return e;
  e = launch_logits_for(s, x, wg, bias, logits, st);
  if (e != cudaSuccess) return e;
  count_launches(2);
  return launch_pdl(k_router_topk, dim3((unsigned)((s.T + 7) / 8)), dim3(256), 0, st, logits, s.T,
                    s.E, s.k, topk_idx, topk_w);
}

cudaError_t launch_route(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                         const float* bias, int32_t* topk_idx, float* topk_w, char* ws,
                         const WsLayout& L, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  float* logits = reinterpret_cast<float*>(ws + L.logits);
  cudaError_t e = launch_logits_for(s, x, wg, bias, logits, st);
  if (e != cudaSuccess) return e;
  count_launches(2);
  return launch_pdl(k_router_topk, dim3((unsigned)((s.T + 7) / 8)), dim3(256), 0, st, logits, s.T,
                    s.E, s.k, topk_idx, topk_w);
}

cudaError_t launch_route_hash(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                              const float* bias, const int32_t* token_ids,
                              const int32_t* tid2eid, int vocab, int32_t* topk_idx,
                              float* topk_w, char* ws, const WsLayout& L, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  float* logits = reinterpret_cast<float*>(ws + L.logits);
  cudaError_t e = launch_logits_for(s, x, wg, bias, logits, st);
  if (e != cudaSuccess) return e;
  count_launches(2);
  return launch_pdl(k_router_hash, dim3((unsigned)((s.T + 7) / 8)), dim3(256), 0, st, logits,
                    token_ids, tid2eid, vocab, s.T, s.E, s.k, topk_idx, topk_w,
                    reinterpret_cast<int*>(ws + L.status));
}

}  // namespace moe
