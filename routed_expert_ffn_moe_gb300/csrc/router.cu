// Router: logits in a fixed fp32 order, top-k selection, gate weights.
//
// The pages: the router scores every routed expert for each token and keeps the top-k, its
// compute is small and its product is the sparse metadata for dispatch ("DeepSeek-V4-Pro on
// NVIDIA H200", 0.2.2 step D4); V4 uses learned soft routing ("CANN DeepSeek-V4推理优化", MoE
// 专家模型规格). Ascend fuses the gate into one "GatingTopK" kernel (same page, 融合Kernel);
// here the logits GEMM and the selection are two kernels so the selection can see all E
// logits of a token at once. Batches of 1024+ tokens form approximate logits on the tensor
// cores and recompute only the candidates' logits in the fixed order (same bits; see the
// section below); hash routing forms only the k hashed logits of each token.
#include <cstdlib>

#include "ffn.h"
#include "internal.h"
#include "topk.cuh"

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
                                                       int d, int E, float* __restrict__ logits,
                                                       int* clear) {
  pdl_wait_then_release();
  if (clear && blockIdx.x == 0 && threadIdx.x == 0) *clear = 0;
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

// Batches of at most kSmallT tokens: the same per-logit order, one warp per expert. The block
// first copies the T token rows into shared memory; each lane then issues the loads of up to 32
// of its 8-element chunks of wg_e at once (one round trip to HBM instead of one per few chunks)
// and runs its fused multiply-add chain over them in the defined order against the token rows
// in shared memory.
constexpr int kSmallT = 4;
constexpr int kSmallBatch = 32;  // chunks of wg_e in flight per lane

__global__ void __launch_bounds__(128) k_router_logits_small(const uint16_t* __restrict__ x,
                                                             const uint16_t* __restrict__ wg,
                                                             const float* __restrict__ bias,
                                                             int T, int d, int E,
                                                             float* __restrict__ logits,
                                                             int* clear) {
  extern __shared__ uint4 xs[];  // [T][d / 8]
  const int lane = threadIdx.x & 31;
  const int chunks = d >> 3;
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const uint4* we = reinterpret_cast<const uint4*>(wg + (size_t)min(e, E - 1) * d);
  const int mine = (chunks - lane + 31) / 32;  // chunks lane, lane + 32, ... below `chunks`
  // The router row is a constant input: its first batch of chunks is requested before the wait
  // for x (which the previous kernel may write).
  uint4 w[kSmallBatch];
#pragma unroll
  for (int i = 0; i < kSmallBatch; ++i)
    if (i < mine) w[i] = __ldg(we + lane + 32 * i);
  pdl_wait_then_release();
  if (clear && blockIdx.x == 0 && threadIdx.x == 0) *clear = 0;
  for (int i = threadIdx.x; i < T * chunks; i += blockDim.x)
    xs[i] = ldg_u4(reinterpret_cast<const uint4*>(x) + i);
  __syncthreads();
  if (e >= E) return;
  float acc[kSmallT];
#pragma unroll
  for (int t = 0; t < kSmallT; ++t) acc[t] = 0.f;
  for (int b0 = 0; b0 < mine; b0 += kSmallBatch) {
    if (b0 > 0) {
#pragma unroll
      for (int i = 0; i < kSmallBatch; ++i)
        if (b0 + i < mine) w[i] = __ldg(we + lane + 32 * (b0 + i));
    }
#pragma unroll
    for (int i = 0; i < kSmallBatch; ++i) {
      if (b0 + i >= mine) break;
      const int c = lane + 32 * (b0 + i);
#pragma unroll
      for (int t = 0; t < kSmallT; ++t) {
        if (t >= T) break;
        const uint4 xv = xs[t * chunks + c];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          acc[t] = __fmaf_rn(bf16x8_elem(xv, j), bf16x8_elem(w[i], j), acc[t]);
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
    for (int t = 0; t < kSmallT; ++t)
      acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xffffffffu, acc[t], off));
  if (lane < T) {
    float a = acc[0];
#pragma unroll
    for (int t = 1; t < kSmallT; ++t)
      if (lane == t) a = acc[t];
    logits[(size_t)lane * E + e] = bias ? __fadd_rn(a, bias[e]) : a;
  }
}

// One warp per token: k rounds of warp-wide arg-max over the E logits (lane j holds experts
// j, j+32, ...), then the gate weights softmax(l_chosen) = exp(l_j - l_max) / sum.
__global__ void __launch_bounds__(256) k_router_topk(const float* __restrict__ logits, int T,
                                                     int E, int k, int32_t* __restrict__ topk_idx,
                                                     float* __restrict__ topk_w) {
  pdl_wait_then_release();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  warp_topk_token(logits + (size_t)t * E, E, k, topk_idx + (size_t)t * k, topk_w + (size_t)t * k);
}

// ---- large batches: approximate logits on the tensor cores, exact logits of the candidates --
//
// The logits GEMM of a large batch runs on the tensor cores (bf16 products, fp32 accumulation
// in the MMA's own order), so each approximate logit a[t,e] may differ from the defined logit
// l[t,e] by a rounding error. Both are taken to lie within eps[t,e] = 2^-12 |x_t| |wg_e|
// (+ 2^-22 |a|, for the bias addition) of each other: sum |x_i w_i| <= |x||w| (Cauchy-Schwarz),
// and each of the two fp32 sums, the defined one and the MMA's, errs by at most about
// n 2^-24 sum |x_i w_i| for its n roundings (n <= ~1100 at d = 16384: 2^-13.9), so together at
// most 2^-12.9 |x||w|, provided the MMA's internal additions round no worse than fp32 (its
// accumulation order and precision are not documented, hence the check below). The errors
// measured on the GPU are near 2^-21 |x||w|.
//
// With lo = a - eps and hi = a + eps (rounded outward) and theta the k-th largest lo, at least k
// experts have l >= theta, so every expert of the top-k has hi >= theta, and an expert with
// hi < theta has l < theta <= the k-th largest l: it is neither chosen nor tied with a chosen
// one. The candidates {hi >= theta} get their defined logits recomputed in the defined order,
// and the selection and the gate weights run on those exactly as k_router_topk runs on all E,
// so the result is identical bit for bit. Each recomputed logit is checked against its bound;
// if one misses it, the token's logits are all recomputed (and counted in the status word): a
// bound that failed would show on the candidates, the logits nearest the choice.

// The bound coefficient. MOE_ROUTER_TC_BOUND overrides it; a negative value makes every token
// take the full recomputation (a test runs that path this way).
constexpr float kBoundC = 0x1p-12f;
constexpr float kNormUp = 1.0f + 0x1p-10f;  // covers the rounding of the fp32 norms

// Block 0 writes the one-matrix tile plan of the logits GEMM (expert offsets {0, T}, tile prefix
// {0, tiles}) and clears the router's status words; every warp then takes experts e and writes
// |wg_e| (rounded up).
__global__ void __launch_bounds__(256) k_router_prep(const uint16_t* __restrict__ wg, int T, int d,
                                                     int E, int tiles, int32_t* __restrict__ plan,
                                                     float* __restrict__ wnorm, int* status) {
  pdl_wait_then_release();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    plan[0] = 0;
    plan[1] = T;
    plan[2] = 0;
    plan[3] = tiles;
    status[kStatusRouterFull] = 0;
    status[kStatusRouterBoundUse] = 0;
  }
  const int lane = threadIdx.x & 31;
  const int chunks = d >> 3;
  for (int e = blockIdx.x * 8 + (threadIdx.x >> 5); e < E; e += gridDim.x * 8) {
    const uint16_t* we = wg + (size_t)e * d;
    float ss = 0.f;
    for (int c = lane; c < chunks; c += 32) {
      const uint4 v = ldg_u4(we + 8 * c);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float f = bf16x8_elem(v, i);
        ss = fmaf(f, f, ss);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) wnorm[e] = sqrtf(ss) * kNormUp;
  }
}

// NC defined logits of token row xt at once (experts e[0..NC)), in the order of
// k_router_logits: lane j accumulates chunks j, j+32, ... element by element from +0, then the
// xor butterfly. The x chunk is loaded once for the NC experts. Every lane returns the sums.
template <int NC>
__device__ __forceinline__ void defined_logits(const uint16_t* __restrict__ xt,
                                               const uint16_t* __restrict__ wg, const int (&e)[NC],
                                               int d, int lane, float (&out)[NC]) {
  float acc[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j) acc[j] = 0.f;
  const int chunks = d >> 3;
#pragma unroll 4
  for (int c = lane; c < chunks; c += 32) {
    const uint4 xv = ldg_u4(xt + 8 * c);
    uint4 wv[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) wv[j] = ldg_u4(wg + (size_t)e[j] * d + 8 * c);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float xf = bf16x8_elem(xv, i);
#pragma unroll
      for (int j = 0; j < NC; ++j) acc[j] = __fmaf_rn(xf, bf16x8_elem(wv[j], i), acc[j]);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
    for (int j = 0; j < NC; ++j)
      acc[j] = __fadd_rn(acc[j], __shfl_xor_sync(0xffffffffu, acc[j], off));
#pragma unroll
  for (int j = 0; j < NC; ++j) out[j] = acc[j];
}

// Hash routing: one warp per token. Lane j < k takes expert e_j = tid2eid[token_ids[t]][j]; the
// warp forms those k logits itself, in the defined order (defined_logits, four experts per
// pass over x), and no other logit. The gate weights are exp(l_j - l_max) / sum over the k,
// computed as k_router_topk computes them for the soft choice (so a table holding the soft
// choices gives the same bits). A token id or table entry out of range is recorded in the
// status word and replaced by 0.
__global__ void __launch_bounds__(256) k_router_hash(const uint16_t* __restrict__ x,
                                                     const uint16_t* __restrict__ wg,
                                                     const float* __restrict__ bias,
                                                     const int32_t* __restrict__ token_ids,
                                                     const int32_t* __restrict__ tid2eid,
                                                     int vocab, int T, int d, int E, int k,
                                                     int32_t* __restrict__ topk_idx,
                                                     float* __restrict__ topk_w, int* status) {
  constexpr int kGroup = 4;
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
  if (lane < k) {
    e = __ldg(tid2eid + (size_t)tid * k + lane);
    if (e < 0 || e >= E) {
      record_error(status, MOE_ERR_DEVICE_BOUNDS);
      e = 0;
    }
  }
  const uint16_t* xt = x + (size_t)t * d;
  float l = -INFINITY;
  for (int g = 0; g < k; g += kGroup) {
    int eg[kGroup];
#pragma unroll
    for (int j = 0; j < kGroup; ++j) eg[j] = __shfl_sync(0xffffffffu, e, min(g + j, k - 1));
    float sdef[kGroup];
    defined_logits<kGroup>(xt, wg, eg, d, lane, sdef);
#pragma unroll
    for (int j = 0; j < kGroup; ++j)
      if (g + j < k && lane == g + j) l = bias ? __fadd_rn(sdef[j], bias[eg[j]]) : sdef[j];
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

// One warp per token; lane j holds experts j + 32m, m < MAXM (E <= 32 MAXM). approx holds the
// tensor-core logits without the bias. Up to 256 experts, two blocks share an SM.
template <int MAXM>
__global__ void __launch_bounds__(256, MAXM <= 8 ? 2 : 1) k_router_select(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wg, const float* __restrict__ bias,
    const float* __restrict__ approx, const float* __restrict__ wnorm, int T, int d, int E, int k,
    float bound_c, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int* status) {
  constexpr int kGroup = 4;  // candidates whose defined logits are formed together
  __shared__ int cand[8][32 * MAXM];
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + w;
  if (t >= T) return;
  const uint16_t* xt = x + (size_t)t * d;

  // |x_t|, rounded up
  float ss = 0.f;
  for (int c = lane; c < (d >> 3); c += 32) {
    const uint4 v = ldg_u4(xt + 8 * c);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float f = bf16x8_elem(v, i);
      ss = fmaf(f, f, ss);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float nx = sqrtf(ss) * kNormUp;

  // approximate logits with the bias, their bounds, and the outward-rounded intervals
  float ah[MAXM], eps[MAXM], lo[MAXM];
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    const int e = lane + 32 * m;
    if (e < E) {
      const float a = approx[(size_t)t * E + e];
      ah[m] = bias ? __fadd_rn(a, bias[e]) : a;
      eps[m] = __fadd_ru(__fmul_ru(__fmul_ru(fmaxf(bound_c, 0.f), nx), wnorm[e]),
                         __fmul_ru(0x1p-22f, fabsf(ah[m]))) + 0x1p-126f;
      lo[m] = __fsub_rd(ah[m], eps[m]);
    } else {
      ah[m] = eps[m] = 0.f;
      lo[m] = -INFINITY;
    }
  }
  // theta: the k-th largest lower bound (k rounds of a warp arg-max)
  float theta = -INFINITY;
  {
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
      float bl = -INFINITY;
      int bm = -1;
#pragma unroll
      for (int m = 0; m < MAXM; ++m)
        if (!((taken >> m) & 1u) && lane + 32 * m < E && (bm < 0 || lo[m] > bl)) {
          bl = lo[m];
          bm = m;
        }
      int be = bm < 0 ? 0x7FFFFFFF : lane + 32 * bm;
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
      theta = bl;
    }
  }

  // candidates: hi >= theta, listed in expert order
  uint32_t mine = 0;
#pragma unroll
  for (int m = 0; m < MAXM; ++m)
    if (lane + 32 * m < E && __fadd_ru(ah[m], eps[m]) >= theta) mine |= 1u << m;
  int n = 0;
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    const uint32_t b = __ballot_sync(0xffffffffu, (mine >> m) & 1u);
    if ((mine >> m) & 1u) cand[w][n + __popc(b & ((1u << lane) - 1u))] = lane + 32 * m;
    n += __popc(b);
  }
  __syncwarp();

  // their defined logits (kept by the lane that holds the expert), each checked against its
  // bound
  float lx[MAXM];
#pragma unroll
  for (int m = 0; m < MAXM; ++m) lx[m] = -INFINITY;
  float use = 0.f;
  bool miss = bound_c < 0.f;
  for (int g = 0; g < n; g += kGroup) {
    int e[kGroup];
#pragma unroll
    for (int j = 0; j < kGroup; ++j) e[j] = cand[w][min(g + j, n - 1)];
    float sdef[kGroup];
    defined_logits<kGroup>(xt, wg, e, d, lane, sdef);
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if (g + j >= n) break;
      const float l = bias ? __fadd_rn(sdef[j], bias[e[j]]) : sdef[j];
      const int src = e[j] & 31, mj = e[j] >> 5;
      float a_j = 0.f, eps_j = 1.f;
#pragma unroll
      for (int m = 0; m < MAXM; ++m)
        if (m == mj) {
          a_j = ah[m];
          eps_j = eps[m];
          if (lane == src) lx[m] = l;
        }
      a_j = __shfl_sync(0xffffffffu, a_j, src);
      eps_j = __shfl_sync(0xffffffffu, eps_j, src);
      const float r = fabsf(l - a_j) / eps_j;
      use = fmaxf(use, r);
      miss |= !(r <= 1.f);
    }
  }
  if (miss) {
    // a recomputed logit missed its bound: form every logit of this token in the defined order
    for (int g = 0; g < E; g += kGroup) {
      int e[kGroup];
#pragma unroll
      for (int j = 0; j < kGroup; ++j) e[j] = min(g + j, E - 1);
      float sdef[kGroup];
      defined_logits<kGroup>(xt, wg, e, d, lane, sdef);
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        const float l = bias ? __fadd_rn(sdef[j], bias[e[j]]) : sdef[j];
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
          if (g + j < E && e[j] == lane + 32 * m) lx[m] = l;
      }
    }
    mine = 0;
#pragma unroll
    for (int m = 0; m < MAXM; ++m)
      if (lane + 32 * m < E) mine |= 1u << m;
    if (lane == 0) atomicAdd(status + kStatusRouterFull, 1);
  }
  if (lane == 0) atomicMax(status + kStatusRouterBoundUse, __float_as_int(use));

  // top-k over the defined logits of the candidates, then the gate weights, as k_router_topk
  const float (&l)[MAXM] = lx;
  uint32_t taken = 0;
  float my_l = -INFINITY;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bl = -INFINITY;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      const int e = lane + 32 * m;
      if (((mine >> m) & 1u) && !((taken >> m) & 1u) && ranks_before(l[m], e, bl, be)) {
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

template <int TT, int TE, int UNROLL = 4>
cudaError_t launch_logits(const uint16_t* x, const uint16_t* wg, const float* bias, int T, int d,
                          int E, float* logits, cudaStream_t st, int* clear = nullptr) {
  const long warps = (long)((T + TT - 1) / TT) * ((E + TE - 1) / TE);
  const long blocks = (warps + 3) / 4;
  if constexpr (TT == 1) {
    return launch_pdl(k_router_logits<TT, TE, UNROLL>, dim3((unsigned)blocks), dim3(128), 0, st, x, wg,
                      bias, T, d, E, logits, clear);
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
                              const float* bias, float* logits, cudaStream_t st,
                              int* clear = nullptr) {
  // At these batch sizes the logits are latency-bound: one or two experts a warp (more warps in
  // flight) and eight chunk loads in flight a lane (measured: FP8 T=1 layer 127.7 -> 124.2 us,
  // MXFP4 T=8 272.9 -> 266.3 us).
  if (s.T <= kSmallT) {
    const size_t smem = (size_t)s.T * s.d * 2;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k_router_logits_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return cudaGetLastError();
    return launch_pdl(k_router_logits_small, dim3((unsigned)((s.E + 3) / 4)), dim3(128), smem, st,
                      x, wg, bias, s.T, s.d, s.E, logits, clear);
  }
  if (s.T <= 8) return launch_logits<1, 1, 8>(x, wg, bias, s.T, s.d, s.E, logits, st, clear);
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

// Device address of the array in the current device's context. It is looked up on every call
// (cudaGetSymbolAddress allocates nothing and costs a table lookup), so the address stays right
// after a cudaDeviceReset or under another context on the same device, where the module is
// loaded again at a new address. On a device's first call the lookup also loads the library's
// device code, which is why that first call should come before any stream capture.
static cudaError_t noalloc_logits_ptr(float** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_logits);
  if (e != cudaSuccess) return e;
  *out = static_cast<float*>(p);
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

// Batches from this many tokens take the tensor-core router (MOE_ROUTER_TC_MIN_TOKENS
// overrides it); it needs E % 128 == 0 (whole 128-row tiles of wg) and d % 64 == 0.
static long router_tc_min_tokens() {
  const char* v = getenv("MOE_ROUTER_TC_MIN_TOKENS");
  return v && *v ? atol(v) : 1024;
}

static float router_tc_bound() {
  const char* v = getenv("MOE_ROUTER_TC_BOUND");
  return v && *v ? (float)atof(v) : kBoundC;
}

bool router_uses_tc(const moe_shape& s) {
  return s.E % 128 == 0 && s.d % 64 == 0 && s.E <= 1024 && s.T >= router_tc_min_tokens();
}

cudaError_t launch_router_logits(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                 const float* bias, float* logits, cudaStream_t st,
                                 int* clear_status) {
  count_launches(1);
  return launch_logits_for(s, x, wg, bias, logits, st, clear_status);
}

template <int MAXM>
static cudaError_t launch_select(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                 const float* bias, const float* approx, const float* wnorm,
                                 int32_t* topk_idx, float* topk_w, int* status, cudaStream_t st) {
  return launch_pdl(k_router_select<MAXM>, dim3((unsigned)((s.T + 7) / 8)), dim3(256), 0, st, x,
                    wg, bias, approx, wnorm, s.T, s.d, s.E, s.k, router_tc_bound(), topk_idx,
                    topk_w, status);
}

static cudaError_t launch_route_tc(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                   const float* bias, int32_t* topk_idx, float* topk_w, char* ws,
                                   const WsLayout& L, cudaStream_t st) {
  int32_t* plan = reinterpret_cast<int32_t*>(ws + L.rtc);
  float* wnorm = reinterpret_cast<float*>(ws + L.rtc + 16);
  float* approx = reinterpret_cast<float*>(ws + L.logits);
  int* status = reinterpret_cast<int*>(ws + L.status);
  // the logits GEMM as the down pass of one expert: "h" = x [T, d], "W_d" = wg [E, d], output
  // rows of E logits, 64-token tiles of 128 experts
  const int tiles = (s.T + tc_tile_tokens(false, true) - 1) / tc_tile_tokens(false, true) *
                    (s.E / tc_tile_rows(false, true, s.E));
  const int nb = (s.E + 7) / 8 < 2 * num_sms() ? (s.E + 7) / 8 : 2 * num_sms();
  cudaError_t e = launch_pdl(k_router_prep, dim3((unsigned)nb), dim3(256), 0, st, wg, s.T, s.d,
                             s.E, tiles, plan, wnorm, status);
  if (e != cudaSuccess) return e;
  count_launches(2);  // prep and select (launch_tc counts its own)
  FfnArgs a{};
  a.T = s.T;
  a.k = 1;
  a.E = 1;
  a.n_shared = 0;
  a.d = s.E;
  a.f = s.d;
  a.wdtype = MOE_W_BF16;
  a.offsets = plan;
  a.w2 = wg;
  a.h = const_cast<uint16_t*>(x);  // read only: the down pass loads its rows through TMA
  a.y_perm = approx;
  a.status = status;
  e = launch_tc(a, plan + 2, false, true, st);
  if (e != cudaSuccess) return e;
  if (s.E <= 256)
    return launch_select<8>(s, x, wg, bias, approx, wnorm, topk_idx, topk_w, status, st);
  if (s.E <= 512)
    return launch_select<16>(s, x, wg, bias, approx, wnorm, topk_idx, topk_w, status, st);
  return launch_select<32>(s, x, wg, bias, approx, wnorm, topk_idx, topk_w, status, st);
}

cudaError_t launch_route(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                         const float* bias, int32_t* topk_idx, float* topk_w, char* ws,
                         const WsLayout& L, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  if (router_uses_tc(s)) return launch_route_tc(s, x, wg, bias, topk_idx, topk_w, ws, L, st);
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
  count_launches(1);
  return launch_pdl(k_router_hash, dim3((unsigned)((s.T + 7) / 8)), dim3(256), 0, st, x, wg, bias,
                    token_ids, tid2eid, vocab, s.T, s.d, s.E, s.k, topk_idx, topk_w,
                    reinterpret_cast<int*>(ws + L.status));
}

}  // namespace moe
