// Expert FFN orchestration: a device-side work plan from the expert segment sizes, then the
// gate/up pass and the down pass, each split between the tensor-core grouped GEMM (experts with
// at least tc_min tokens) and the weight-streaming GEMV (experts with fewer).
//
// Expert segment sizes exist only on the device (they come from the router), so the host never
// waits for them: a one-block plan kernel turns expert_offsets into per-expert prefix sums of
// work items for each kernel, and the persistent FFN kernels walk those lists.
#include <climits>
#include <cstdlib>
#include <mutex>

#include "ffn.h"
#include "topk.cuh"

namespace moe {
namespace {

struct PlanArgs {
  int E, n_shared, tc_min;
  int group, items_up, items_dn;   // weight-streaming: tokens per item, items per group
  int nt_up, nt_dn, mt_up, mt_dn;  // tensor-core: tokens per tile, weight tiles per expert
  int stride;
  // Split prefill (split != 0): experts with at most cold_max tokens form a second tile list
  // (nt_c-token tiles, mt_up_c / mt_dn_c weight tiles per expert) run on their own CTAs.
  int split, cold_max, nt_c, mt_up_c, mt_dn_c, nsm;
  // per pass (0 gate/up, 1 down), in SM-microseconds: streaming one cold expert's weights,
  // tensor work per token of a hot expert, and the least a hot expert costs
  float cold_cost[2], hot_cost_tok[2], hot_cost_min[2];
};

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

// plan[row][e]: exclusive prefix over experts of the work of each kernel; entry E1 = total.
// With a split, row kPlanSplit holds the number of CTAs for the cold list and for the rest,
// chosen so that both lists take about the same time by a simple cost model.
__device__ __forceinline__ void plan_block(const int32_t* offsets, const PlanArgs& a,
                                           int32_t* __restrict__ plan) {
  __shared__ float red[32];
  const int E1 = a.E + a.n_shared;
  constexpr int R = kPlanTcDnCold + 1;
  int run[R] = {};
  float cold[2] = {0.f, 0.f}, hot[2] = {0.f, 0.f};
  for (int b = 0; b < E1; b += blockDim.x) {
    const int e = b + threadIdx.x;
    int n[R] = {};
    if (e < E1) {
      const int cnt = offsets[e + 1] - offsets[e];
      if (a.split && cnt > 0 && cnt <= a.cold_max) {
        n[kPlanTcUpCold] = (cnt + a.nt_c - 1) / a.nt_c * a.mt_up_c;
        n[kPlanTcDnCold] = (cnt + a.nt_c - 1) / a.nt_c * a.mt_dn_c;
        cold[0] += a.cold_cost[0];
        cold[1] += a.cold_cost[1];
      } else if (cnt >= a.tc_min) {
        n[kPlanTcUp] = (cnt + a.nt_up - 1) / a.nt_up * a.mt_up;
        n[kPlanTcDown] = (cnt + a.nt_dn - 1) / a.nt_dn * a.mt_dn;
        hot[0] += fmaxf(a.hot_cost_min[0], a.hot_cost_tok[0] * (float)cnt);
        hot[1] += fmaxf(a.hot_cost_min[1], a.hot_cost_tok[1] * (float)cnt);
      } else if (cnt > 0) {
        const int groups = (cnt + a.group - 1) / a.group;
        n[kPlanGemvUp] = groups * a.items_up;
        n[kPlanGemvDown] = groups * a.items_dn;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      int tot;
      const int pre = block_exclusive_scan(n[r], &tot);
      if (e < E1) plan[r * a.stride + e] = run[r] + pre;
      run[r] += tot;
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    cold[i] = block_sum(cold[i], red);
    hot[i] = block_sum(hot[i], red);
  }
  if (threadIdx.x == 0) {
    for (int r = 0; r < R; ++r) plan[r * a.stride + E1] = run[r];
    for (int i = 0; i < 2; ++i) {
      int xc = 0;  // CTAs for the cold list, an even number (the other list runs in pairs)
      if (a.split && cold[i] > 0.f) {
        xc = hot[i] > 0.f ? 2 * __float2int_rn(0.5f * a.nsm * cold[i] / (cold[i] + hot[i]))
                          : a.nsm;
        xc = min(max(xc, 2), hot[i] > 0.f ? a.nsm - 2 : a.nsm);
      }
      plan[kPlanSplit * a.stride + 2 * i] = xc;
      plan[kPlanSplit * a.stride + 2 * i + 1] = a.nsm - xc;
    }
  }
}

// Thread i copies 16-byte chunks 4i .. 4i+3 of the slot rows (d is a multiple of 128, so the four
// chunks lie in one row): four loads in flight per thread.
constexpr int kGatherChunks = 4;

__device__ __forceinline__ void gather_row_chunks(long i, const uint16_t* __restrict__ x,
                                                  const int32_t* perm_token, int T,
                                                  long routed, int d,
                                                  uint16_t* __restrict__ x_perm, int* status) {
  const int d8 = d >> 3;
  const long c0 = i * kGatherChunks;
  if (c0 >= routed * d8) return;
  const long s = c0 / d8;
  const int c = (int)(c0 - s * d8);
  int t = perm_token[s];  // global or shared memory
  if (t < 0 || t >= T) {
    record_error(status, MOE_ERR_DEVICE_BOUNDS);
    t = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + (long)t * d) + c;
  uint4* dst = reinterpret_cast<uint4*>(x_perm + s * d) + c;
  uint4 v[kGatherChunks];
#pragma unroll
  for (int j = 0; j < kGatherChunks; ++j) v[j] = __ldg(src + j);
#pragma unroll
  for (int j = 0; j < kGatherChunks; ++j) dst[j] = v[j];
}

// MXFP4 weights: thread i encodes 32-element block i of the slot rows as two E4M3 terms
// (mx_common.cuh). Slot s < routed holds token perm_token[s]; slot routed + t (the shared
// expert's segment) holds token t. Rows at or beyond nq are not this launch's.
__device__ __forceinline__ void gather_encode_block(long i, const uint16_t* __restrict__ x,
                                                    const int32_t* perm_token, int T,
                                                    long routed, long nq, int d,
                                                    const mx::Planes& xq, int* status) {
  const int nb = d >> 5;
  const long s = i / nb;
  if (s >= nq) return;
  const int b = (int)(i - s * nb);
  int t = s < routed ? perm_token[s] : (int)(s - routed);
  if (t < 0 || t >= T) {
    record_error(status, MOE_ERR_DEVICE_BOUNDS);
    t = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + (long)t * d) + 4 * b;
  uint4 w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) w[j] = __ldg(src + j);
  float v[32];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t u[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      v[8 * j + 2 * m] = __uint_as_float(u[m] << 16);
      v[8 * j + 2 * m + 1] = __uint_as_float(u[m] & 0xFFFF0000u);
    }
  }
  uint32_t hi[8], lo[8], sa, sb;
  mx::encode32(v, hi, lo, sa, sb);
  uint4* dh = reinterpret_cast<uint4*>(xq.hi + s * d + 32 * b);
  uint4* dl = reinterpret_cast<uint4*>(xq.lo + s * d + 32 * b);
  dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
  dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  xq.s_hi[s * nb + b] = (uint8_t)sa;
  xq.s_lo[s * nb + b] = (uint8_t)sb;
}

// E4M3 and MXFP4 weights, prefill tiles: thread i writes 32-element block i of the slot rows (the same
// rows as above) as f16, round to nearest, saturating at +-65504 (exact for bf16 values in f16's
// normal range).
__device__ __forceinline__ void gather_f16_block(long i, const uint16_t* __restrict__ x,
                                                 const int32_t* perm_token, int T,
                                                 long routed, long nq, int d,
                                                 uint16_t* __restrict__ out, int* status) {
  const int nb = d >> 5;
  const long s = i / nb;
  if (s >= nq) return;
  const int b = (int)(i - s * nb);
  int t = s < routed ? perm_token[s] : (int)(s - routed);
  if (t < 0 || t >= T) {
    record_error(status, MOE_ERR_DEVICE_BOUNDS);
    t = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + (long)t * d) + 4 * b;
  uint4* dst = reinterpret_cast<uint4*>(out + s * d) + 4 * b;
  uint4 w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) w[j] = __ldg(src + j);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t u[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
    for (int m = 0; m < 4; ++m)
      asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
          : "=r"(u[m])
          : "f"(__uint_as_float(u[m] & 0xFFFF0000u)), "f"(__uint_as_float(u[m] << 16)));
    dst[j] = make_uint4(u[0], u[1], u[2], u[3]);
  }
}

// What the gather writes for the tensor-core passes.
enum GatherMode : int {
  kGatherBf16 = 0,  // bf16 and FP8 weights: x rows of the routed slots, bf16
  kGatherMxTerms = 1,  // MXFP4 decode tiles: the slot rows as two E4M3 terms (xq)
  kGatherF16 = 2,  // E4M3 and MXFP4 prefill tiles: the slot rows as f16 (x_perm)
};

// One warp copies slot row s (bf16, or converted to f16 as gather_f16_block does): the row's
// token from one load, then 8 of the row's 16-byte chunks in flight a lane at a time (lane j
// takes chunks j, j+32, ...). Slot s < routed holds token perm_token[s]; slot routed + t (the
// shared expert's segment) holds token t.
__device__ __forceinline__ void gather_row_warp(long s, const uint16_t* __restrict__ x,
                                                const int32_t* __restrict__ perm_token, int T,
                                                long routed, int d, uint16_t* __restrict__ out,
                                                bool to_f16, int* status) {
  const int lane = threadIdx.x & 31;
  int t = s < routed ? perm_token[s] : (int)(s - routed);
  if (t < 0 || t >= T) {
    if (lane == 0) record_error(status, MOE_ERR_DEVICE_BOUNDS);
    t = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + (long)t * d);
  uint4* dst = reinterpret_cast<uint4*>(out + s * d);
  const int n = d >> 3;
  for (int c0 = lane; c0 < n; c0 += 32 * 8) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (c0 + 32 * j < n) v[j] = __ldg(src + c0 + 32 * j);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (c0 + 32 * j >= n) break;
      if (to_f16) {
        uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int m = 0; m < 4; ++m)
          asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
              : "=r"(u[m])
              : "f"(__uint_as_float(u[m] & 0xFFFF0000u)), "f"(__uint_as_float(u[m] << 16)));
        v[j] = make_uint4(u[0], u[1], u[2], u[3]);
      }
      dst[c0 + 32 * j] = v[j];
    }
  }
}

// Blocks of the gather: the MXFP4 term encoding takes a thread per 32-element block, the row
// copies a warp per row (8 rows a block of 256 threads).
long gather_blocks(int mode, long nq, int d) {
  if (nq <= 0) return 0;
  return mode == kGatherMxTerms ? (nq * (d / 32) + 255) / 256 : (nq + 7) / 8;
}

// One launch for both: block 0 builds the plan from the expert offsets while the other blocks
// gather the token rows the tensor-core passes read as contiguous TMA rows (GatherMode). Neither
// needs the other.
__global__ void __launch_bounds__(256) k_plan_gather(const int32_t* __restrict__ offsets,
                                                     PlanArgs a, int32_t* __restrict__ plan,
                                                     const uint16_t* __restrict__ x,
                                                     const int32_t* __restrict__ perm_token, int T,
                                                     long routed, int d,
                                                     uint16_t* __restrict__ x_perm, int* status,
                                                     mx::Planes xq, long nq, int mode) {
  pdl_wait_then_release();
  if (blockIdx.x == 0) {
    plan_block(offsets, a, plan);
    return;
  }
  if (mode == kGatherMxTerms) {
    const long i = (long)(blockIdx.x - 1) * blockDim.x + threadIdx.x;
    gather_encode_block(i, x, perm_token, T, routed, nq, d, xq, status);
    return;
  }
  const long s = (long)(blockIdx.x - 1) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (s < nq) gather_row_warp(s, x, perm_token, T, routed, d, x_perm, mode == kGatherF16, status);
}

// Decode batches of at most 8 tokens (one permutation chunk), moe_forward only: after the
// router logits, one launch does what k_router_topk, k_perm_small and k_plan_gather do. Every
// block selects the top k of every token (warp_topk_token, the router's own selection, a warp
// per token) and sorts the T*k (token, choice) pairs in shared memory as k_perm_small sorts one
// chunk (one 32-bit mask of tokens per expert, an exclusive scan of the mask popcounts in
// expert order, a pair's slot = its expert's offset + the number of its expert's tokens before
// it), with a thread per pair and the slot offsets and both tile prefixes in one scan; this is
// repeated in every block so that no block waits for another. (At 32 tokens the repeated
// selection made the front no faster than the three kernels it replaces: V4-Pro decode 1576 us
// with it at 256 threads, 1559 us at 512, 1555 us without.) Block 0 then writes the routing,
// the permutation and the tensor-core passes' tile prefixes; the other blocks gather their
// share of the rows (GatherMode) with the permutation held in their own shared memory.
constexpr int kFrontMaxT = 8;

__global__ void __launch_bounds__(256) k_route_front(
    const float* __restrict__ logits, int T, int E, int k, int n_shared,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm_token, int32_t* __restrict__ inv_slot, PlanArgs a,
    int32_t* __restrict__ plan, const uint16_t* __restrict__ x, long routed, int d,
    uint16_t* __restrict__ x_perm, int* status, mx::Planes xq, long nq, int mode,
    int4* __restrict__ tile1, int n_ctas) {
  extern __shared__ uint32_t fm[];
  const int E1 = a.E + a.n_shared;
  uint32_t* sel = fm;                                               // [E] token masks
  int32_t* off_s = reinterpret_cast<int32_t*>(fm + E);              // [E + 2]
  int32_t* idx_s = off_s + (E + 2);                                 // [T * k]
  float* w_s = reinterpret_cast<float*>(idx_s + T * k);             // [T * k]
  int32_t* perm_s = reinterpret_cast<int32_t*>(w_s + T * k);        // [T * k]
  int32_t* inv_s = perm_s + T * k;                                  // [T * k]
  const int warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) sel[e] = 0;
  prefetch_l2_span(logits, (size_t)T * E * 4);
  if (blockIdx.x > 0) prefetch_l2_span(x, (size_t)T * d * 2);
  pdl_wait_then_release();
  for (int t = warp; t < T; t += (int)(blockDim.x >> 5))
    warp_topk_token(logits + (size_t)t * E, E, k, idx_s + t * k, w_s + t * k);
  __syncthreads();
  // The token masks of the one chunk, a thread per (token, choice) pair. A pair whose expert is
  // out of range or repeats an earlier choice of its token is dropped (and reported).
  const int pairs = T * k;
  for (int i = threadIdx.x; i < pairs; i += blockDim.x) {
    const int t = i / k, j = i - t * k;
    const int32_t* row = idx_s + t * k;
    const int e = row[j];
    bool ok = (unsigned)e < (unsigned)E;
    for (int j2 = 0; j2 < j && ok; ++j2) ok = row[j2] != e;
    if (ok)
      atomicOr(&sel[e], 1u << t);
    else if (blockIdx.x == 0)
      record_error(status, MOE_ERR_DEVICE_BOUNDS);
  }
  __syncthreads();
  // One scan over the experts (the shared one last, T tokens): the slot offsets and, in block
  // 0, the tile prefixes of the gate/up and the down pass (as plan_block writes them; every
  // expert on the tensor cores, no split). Each thread takes a run of consecutive experts.
  {
    const int per = (E1 + (int)blockDim.x - 1) / (int)blockDim.x;
    const int e0 = min(E1, (int)threadIdx.x * per), e1 = min(E1, e0 + per);
    // plan units of an expert with cnt tokens (one token tile unless cnt exceeds it)
    auto units = [](int cnt, int nt, int mt) {
      return cnt <= 0 ? 0 : (cnt <= nt ? 1 : (cnt + nt - 1) / nt) * mt;
    };
    int3 sum = make_int3(0, 0, 0);
    for (int e = e0; e < e1; ++e) {
      const int cnt = e < E ? __popc(sel[e]) : T;
      sum.x += e < E ? cnt : 0;
      sum.y += units(cnt, a.nt_up, a.mt_up);
      sum.z += units(cnt, a.nt_dn, a.mt_dn);
    }
    int3 tot;
    int3 run = block_exclusive_scan3(sum, &tot);
    for (int e = e0; e < e1; ++e) {
      const int cnt = e < E ? __popc(sel[e]) : T;
      if (e < E) off_s[e] = run.x;
      if (blockIdx.x == 0) {
        plan[kPlanTcUp * a.stride + e] = run.y;
        plan[kPlanTcDown * a.stride + e] = run.z;
        // the gate/up CTAs' first tiles (one token tile an expert: weight tile = tile - prefix)
        const int more = tot.y > n_ctas ? 1 << 16 : 0;
        const int u = units(cnt, a.nt_up, a.mt_up);
        for (int j = 0; tile1 && j < u && run.y + j < n_ctas; ++j)
          tile1[run.y + j] = make_int4(e, j, e < E ? run.x : T * k, cnt | more);
      }
      run.x += e < E ? cnt : 0;
      run.y += units(cnt, a.nt_up, a.mt_up);
      run.z += units(cnt, a.nt_dn, a.mt_dn);
    }
    if (threadIdx.x == 0) {
      off_s[E] = T * k;
      off_s[E + 1] = T * k + n_shared * T;
      if (blockIdx.x == 0) {
        plan[kPlanTcUp * a.stride + E1] = tot.y;
        plan[kPlanTcDown * a.stride + E1] = tot.z;
      }
    }
    if (blockIdx.x == 0 && tile1)  // CTAs without a tile
      for (int c = tot.y + (int)threadIdx.x; c < n_ctas; c += blockDim.x)
        tile1[c] = make_int4(-1, 0, 0, tot.y > n_ctas ? 1 << 16 : 0);
  }
  __syncthreads();
  // slots: expert offset + the pair's rank among its expert's tokens (token order)
  for (int i = threadIdx.x; i < pairs; i += blockDim.x) {
    const int t = i / k, j = i - t * k;
    const int32_t* row = idx_s + t * k;
    const int e = row[j];
    bool ok = (unsigned)e < (unsigned)E;
    for (int j2 = 0; j2 < j && ok; ++j2) ok = row[j2] != e;
    if (!ok) {
      inv_s[i] = -1;
      continue;
    }
    const int slot = off_s[e] + __popc(sel[e] & ((1u << t) - 1u));
    perm_s[slot] = t;
    inv_s[i] = slot;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < pairs; i += blockDim.x) {
      topk_idx[i] = idx_s[i];
      topk_w[i] = w_s[i];
      perm_token[i] = perm_s[i];
      inv_slot[i] = inv_s[i];
    }
    for (int e = threadIdx.x; e < E + 2; e += blockDim.x) offsets[e] = off_s[e];
    return;
  }
  const long i = (long)(blockIdx.x - 1) * blockDim.x + threadIdx.x;
  if (mode == kGatherMxTerms)
    gather_encode_block(i, x, perm_s, T, routed, nq, d, xq, status);
  else if (mode == kGatherF16)
    gather_f16_block(i, x, perm_s, T, routed, nq, d, x_perm, status);
  else
    gather_row_chunks(i, x, perm_s, T, routed, d, x_perm, status);
}

size_t front_smem_bytes(int T, int E, int k) {
  return 4 * ((size_t)E + (E + 2) + 4 * (size_t)T * k);
}

// Phase events are recorded as external events while the stream is being captured into a CUDA
// graph (so every replay records them) and as plain events otherwise.
cudaError_t record_phase(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cap);
  return cudaEventRecordWithFlags(ev, st,
                                  cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                       : cudaEventRecordDefault);
}

// Token count from which an expert runs on the tensor cores (default 1: all of them).
int tc_min_tokens() {
  const char* v = getenv("MOE_TC_MIN_TOKENS");
  if (!v || !*v) return 1;
  const long n = strtol(v, nullptr, 10);
  return n < 1 ? 1 : (n > INT_MAX ? INT_MAX : (int)n);
}

// Second stream and fork/join events of the split prefill, one set per device, created on first
// use (host objects; no device memory). The record/wait sequence of one call is made under a
// lock so that calls from several host threads do not interleave their event records.
struct SplitStreams {
  cudaStream_t aux = nullptr;   // split prefill: the other tile list
  cudaStream_t aux2 = nullptr;  // moe_forward: the shared expert
  cudaEvent_t ev[6] = {};
  cudaEvent_t cut[3] = {};      // split prefill: records that end programmatic launch overlap
};
std::recursive_mutex g_split_mu;
SplitStreams g_split[64];

cudaError_t split_streams(SplitStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  SplitStreams& s = g_split[dev];
  if (!s.aux) {
    if ((e = cudaStreamCreateWithFlags(&s.aux, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&s.aux2, cudaStreamNonBlocking)) != cudaSuccess) return e;
    for (auto& ev : s.ev)
      if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (auto& ev : s.cut)
      if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &s;
  return cudaSuccess;
}

// `st` waits for everything enqueued so far on `from`.
cudaError_t join(cudaStream_t st, cudaStream_t from, cudaEvent_t ev) {
  cudaError_t e = cudaEventRecord(ev, from);
  return e == cudaSuccess ? cudaStreamWaitEvent(st, ev, 0) : e;
}

// Tensor-core tile shape of both passes: tokens per tile and plan units (weight tiles, or
// cluster pairs of them) per expert.
struct TileShape {
  int nt_up, nt_dn, mt_up, mt_dn;
};

TileShape tile_shape(const moe_shape& s, bool fp8, bool decode, long routed) {
  TileShape t;
  if (s.wdtype == MOE_W_MXFP4_E8M0_B32 && decode) {
    t.nt_up = t.nt_dn = tc_mx_tile_tokens(decode, routed, s.E);
    t.mt_up = s.f / 128;
    t.mt_dn = s.d / tc_mx_down_rows(decode, s.d);
    return t;
  }
  if (s.wdtype == MOE_W_MXFP4_E8M0_B32) fp8 = true;  // the FP8 prefill tiles, f16 operands
  t.nt_up = fp8 ? tc_fp8_tile_tokens(true, decode, routed, s.E) : tc_tile_tokens(true, decode);
  t.nt_dn = fp8 ? tc_fp8_tile_tokens(false, decode, routed, s.E) : tc_tile_tokens(false, decode);
  if (!fp8) {
    t.mt_up = tc_plan_mtiles(true, decode, s.d, s.f);
    t.mt_dn = tc_plan_mtiles(false, decode, s.d, s.f);
  } else if (!decode) {
    t.mt_up = tc_fp8_wide_plan_mtiles(true, s.d, s.f);
    t.mt_dn = tc_fp8_wide_plan_mtiles(false, s.d, s.f);
  } else {
    t.mt_up = s.f / 128;
    t.mt_dn = s.d / tc_fp8_decode_down_rows(s.d);
  }
  return t;
}

// The shared expert's own tile lists, for moe_forward: its segment starts at slot T*k and holds
// the T tokens in order, so the lists depend on the shape alone. rows[0] and rows[1]: prefixes
// over the E+1 experts for the gate/up and the down pass (zero work for the routed experts);
// rows[2]: the expert offsets the tile decoder reads (entries E and E+1). With MXFP4 weights
// the other blocks write the shared segment's rows (token t at slot T*k + t) in the form the
// passes read (GatherMode: E4M3 terms or f16).
__global__ void k_shared_plan(int T, int k, int E, TileShape ts, int32_t* __restrict__ rows,
                              const uint16_t* __restrict__ x, int d, mx::Planes xq,
                              uint16_t* __restrict__ x16, int mode, int* status) {
  pdl_wait_then_release();
  if (blockIdx.x > 0) {
    const long routed = (long)T * k;
    const long i = (long)(blockIdx.x - 1) * blockDim.x + threadIdx.x + routed * (d >> 5);
    if (mode == kGatherMxTerms)
      gather_encode_block(i, x, nullptr, T, routed, routed + T, d, xq, status);
    else
      gather_f16_block(i, x, nullptr, T, routed, routed + T, d, x16, status);
    return;
  }
  const int n = E + 2;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const bool last = e == E + 1;
    rows[e] = last ? (T + ts.nt_up - 1) / ts.nt_up * ts.mt_up : 0;
    rows[n + e] = last ? (T + ts.nt_dn - 1) / ts.nt_dn * ts.mt_dn : 0;
    rows[2 * n + e] = e == E ? T * k : last ? T * k + T : 0;
  }
}


// Everything the FFN passes of one call need: their arguments, the plan kernel's arguments and
// what the gather writes.
struct FfnCall {
  FfnArgs a;
  PlanArgs pa;
  int32_t* plan;
  int stride, tc_min, mode;
  bool fp8, mxq, decode, use_tc, use_gemv, split;
  long routed, nq, gather_n;
};

FfnCall make_ffn_call(const moe_shape& s, const uint16_t* x, const int32_t* perm_token,
                      const int32_t* offsets, const void* w13, const void* s13, const void* w2,
                      const void* s2, float* y_perm, char* ws, const WsLayout& L,
                      bool with_shared) {
  FfnCall c{};
  FfnArgs& a = c.a;
  // without the shared expert (moe_forward runs it on its own stream) the tile lists end at E
  a.T = s.T; a.d = s.d; a.E = s.E; a.k = s.k; a.f = s.f; a.n_shared = with_shared ? s.n_shared : 0;
  a.wdtype = s.wdtype;
  a.x = x; a.perm_token = perm_token; a.offsets = offsets;
  a.w13 = w13; a.s13 = s13; a.w2 = w2; a.s2 = s2;
  a.h = reinterpret_cast<uint16_t*>(ws + L.h);
  a.x_perm = reinterpret_cast<uint16_t*>(ws + L.x_perm);
  a.y_perm = y_perm;
  a.status = reinterpret_cast<int*>(ws + L.status);
  c.mxq = s.wdtype == MOE_W_MXFP4_E8M0_B32;
  const long all_slots = (long)s.T * s.k + (long)s.n_shared * s.T;
  if (c.mxq) {
    a.xq = mx::planes_at(ws + L.xq, all_slots, s.d);
    a.hq = mx::planes_at(ws + L.hq, all_slots, s.f);
  }
  c.plan = reinterpret_cast<int32_t*>(ws + L.plan);

  // Experts with at least tc_min tokens go to the tensor-core GEMM, the rest to the
  // weight-streaming GEMV. Both stream each weight byte once; the tensor-core kernel does so at
  // full HBM rate from one token up, so by default it takes every expert. MOE_TC_MIN_TOKENS
  // moves the split (a tuning and testing knob; results agree within rounding either way).
  // MXFP4 weights run on the tensor cores only (the block-scaled MMA is their format's path).
  c.tc_min = c.mxq ? 1 : tc_min_tokens();
  c.fp8 = s.wdtype == MOE_W_FP8_E4M3_B128;
  c.routed = (long)s.T * s.k;
  c.decode = c.routed <= 32L * s.E;  // at most ~32 tokens per routed expert on average
  c.use_tc = c.tc_min < INT_MAX;
  c.use_gemv = c.tc_min > 1;
  PlanArgs& pa = c.pa;
  pa.E = s.E; pa.n_shared = a.n_shared;
  pa.tc_min = c.tc_min;
  pa.group = gemv_group_tokens();
  pa.items_up = gemv_items_per_group(true, s.d, s.f);
  pa.items_dn = gemv_items_per_group(false, s.d, s.f);
  const TileShape ts = tile_shape(s, c.fp8, c.decode, c.routed);
  pa.nt_up = ts.nt_up;
  pa.nt_dn = ts.nt_dn;
  pa.mt_up = ts.mt_up;
  pa.mt_dn = ts.mt_dn;
  pa.stride = s.E + 2;
  c.stride = pa.stride;
  // Split prefill (bf16 weights, all experts on the tensor cores): experts with at most one
  // decode tile of tokens stream their weights through the decode tiles on part of the SMs
  // while the others run the prefill tiles on the rest, on a second stream, so that the
  // HBM-bound and the tensor-bound experts overlap instead of taking turns on every SM.
  c.split = s.wdtype == MOE_W_BF16 && !c.decode && c.use_tc && !c.use_gemv && c.routed > 0;
  if (c.split) {
    // Rates on GB300 (one SM), fitted to split sweeps of the skewed prefill layer: decode tiles
    // stream weights at ~68 GB/s in the gate/up pass and ~45 GB/s in the down pass (shorter
    // tiles); prefill tiles run ~7.4 TFLOP/s (gate/up) and ~8.2 TFLOP/s (down). Only the ratio
    // of the two sides matters for the split.
    const double bytes = s.d * (double)s.f * 2.0;       // one bf16 weight matrix of an expert
    const double bw_up = 68e3, bw_dn = 45e3;            // bytes per microsecond
    const double tc_up = 7.4e6, tc_dn = 8.2e6;          // FLOP per microsecond
    pa.split = 1;
    pa.nt_c = tc_cold_tile_tokens();
    pa.cold_max = pa.nt_c;
    pa.mt_up_c = tc_plan_mtiles(true, true, s.d, s.f);
    pa.mt_dn_c = tc_plan_mtiles(false, true, s.d, s.f);
    pa.nsm = num_sms() & ~1;
    pa.cold_cost[0] = (float)(2.0 * bytes / bw_up);
    pa.cold_cost[1] = (float)(bytes / bw_dn);
    pa.hot_cost_min[0] = pa.cold_cost[0];
    pa.hot_cost_min[1] = pa.cold_cost[1];
    pa.hot_cost_tok[0] = (float)(4.0 * s.d * s.f / tc_up);
    pa.hot_cost_tok[1] = (float)(2.0 * s.d * s.f / tc_dn);
  }
  // What the gather writes: bf16 rows of the routed slots (bf16 weights, E4M3 decode tiles), or
  // every slot's row, the shared segment's included, as f16 (E4M3 and MXFP4 prefill tiles) or
  // as two E4M3 terms (MXFP4 decode tiles).
  const bool f16_rows = !c.decode && (c.mxq || c.fp8);
  c.nq = c.routed + (c.mxq || f16_rows ? (long)a.n_shared * s.T : 0);
  c.gather_n = (c.use_tc && c.nq > 0) ? c.nq * (s.d / 8) / kGatherChunks : 0;
  c.mode = f16_rows ? kGatherF16 : c.mxq ? kGatherMxTerms : kGatherBf16;
  return c;
}

// The gate/up and down passes of a call whose plan (and gather) are in place.
cudaError_t launch_passes(const moe_shape& s, const FfnCall& c, cudaStream_t st) {
  const FfnArgs& a = c.a;
  const int32_t* plan = c.plan;
  const int stride = c.stride;
  const PhaseEvents ev = profile_phase_events();
  if (ev.begin && !c.split) record_phase(ev.begin, st);
  cudaError_t e = cudaSuccess;

  // Upper bound on the weight-streaming work: every slot in its own group plus one partial
  // group per expert (the device-side totals are usually far smaller).
  const long slots = c.routed + (long)s.n_shared * s.T;
  const long max_groups = (slots + c.pa.group - 1) / c.pa.group + s.E + s.n_shared;
  const auto cap = [](long v) { return (int)(v < (1L << 30) ? v : (1L << 30)); };
  const int max_up = c.use_gemv ? cap(max_groups * c.pa.items_up) : 0;
  const int max_dn = c.use_gemv ? cap(max_groups * c.pa.items_dn) : 0;
  const auto tc = [&](bool gateup, const int32_t* prefix) {
    return c.mxq ? launch_tc_mx(a, prefix, gateup, c.decode, st)
           : c.fp8 ? launch_tc_fp8(a, prefix, gateup, c.decode, st)
                   : launch_tc(a, prefix, gateup, c.decode, st);
  };

  if (c.split) {
    SplitStreams* ss = nullptr;
    if ((e = split_streams(&ss)) != cudaSuccess) return e;
    const int32_t* act = plan + kPlanSplit * stride;
    std::lock_guard<std::recursive_mutex> lk(g_split_mu);
    cudaStream_t aux = ss->aux;
    // An event recorded on `st` between two kernels makes the second wait for the first to
    // complete instead of launching early under programmatic serialisation. The split passes
    // want that at each pass boundary: launched early, the next pass's CTAs hold SMs (a
    // persistent CTA each) that the other list's CTAs of the running pass are waiting for
    // (measured, skewed prefill: 6.05 ms without these records, 4.81 ms with them).
    const auto cut = [&](cudaEvent_t prof, int i) {
      return record_phase(prof ? prof : ss->cut[i], st);
    };
    if ((e = cut(ev.begin, 0)) != cudaSuccess) return e;
    if ((e = join(aux, st, ss->ev[0])) != cudaSuccess) return e;
    if ((e = launch_tc(a, plan + kPlanTcUpCold * stride, true, true, st, act, true)) != cudaSuccess)
      return e;
    if ((e = launch_tc(a, plan + kPlanTcUp * stride, true, false, aux, act + 1)) != cudaSuccess)
      return e;
    if ((e = join(st, aux, ss->ev[1])) != cudaSuccess) return e;
    if ((e = cut(ev.mid, 1)) != cudaSuccess) return e;
    if ((e = join(aux, st, ss->ev[2])) != cudaSuccess) return e;
    if ((e = launch_tc(a, plan + kPlanTcDnCold * stride, false, true, st, act + 2, true)) !=
        cudaSuccess)
      return e;
    if ((e = launch_tc(a, plan + kPlanTcDown * stride, false, false, aux, act + 3)) != cudaSuccess)
      return e;
    if ((e = join(st, aux, ss->ev[3])) != cudaSuccess) return e;
    return cut(ev.end, 2);
  }

  if (c.use_tc) e = tc(true, plan + kPlanTcUp * stride);
  if (e == cudaSuccess)
    e = launch_gemv(a, plan + kPlanGemvUp * stride, plan + kPlanGemvDown * stride, true, max_up, st);
  if (e != cudaSuccess) return e;
  if (ev.mid) record_phase(ev.mid, st);
  if (c.use_tc) e = tc(false, plan + kPlanTcDown * stride);
  if (e == cudaSuccess)
    e = launch_gemv(a, plan + kPlanGemvUp * stride, plan + kPlanGemvDown * stride, false, max_dn, st);
  if (ev.end) record_phase(ev.end, st);
  return e;
}

}  // namespace

cudaError_t launch_expert_ffn(const moe_shape& s, const uint16_t* x, const int32_t* perm_token,
                              const int32_t* offsets, const void* w13, const void* s13,
                              const void* w2, const void* s2, float* y_perm, char* ws,
                              const WsLayout& L, cudaStream_t st, bool with_shared) {
  if (s.T == 0) return cudaSuccess;
  const FfnCall c = make_ffn_call(s, x, perm_token, offsets, w13, s13, w2, s2, y_perm, ws, L,
                                  with_shared);
  const long gb = c.gather_n > 0 ? gather_blocks(c.mode, c.nq, s.d) : 0;
  cudaError_t e = launch_pdl(k_plan_gather, dim3((unsigned)(1 + gb)),
                             dim3(256), 0, st, offsets, c.pa, c.plan, x, perm_token, s.T,
                             c.routed, s.d, c.a.x_perm, c.a.status, c.a.xq, c.nq, c.mode);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return launch_passes(s, c, st);
}

// moe_forward on a decode batch of at most 8 tokens with the fp32 router and every expert on the
// tensor cores: logits, then k_route_front (top-k, permutation, plan and gather in one launch),
// then the FFN passes and the combine. The outputs are the same bits as the four calls.
static bool front_applies(const moe_shape& s) {
  if (s.T < 1 || s.T > kFrontMaxT || tc_min_tokens() != 1) return false;
  if ((long)s.T * s.k > 32L * s.E) return false;  // the FFN runs its decode tiles
  return front_smem_bytes(s.T, s.E, s.k) <= 48 * 1024;
}

static cudaError_t launch_forward_front(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                        const float* bias, const void* w13, const void* s13,
                                        const void* w2, const void* s2, int32_t* topk_idx,
                                        float* topk_w, int32_t* offsets, int32_t* perm_token,
                                        int32_t* inv_slot, float* y_perm, uint16_t* y, char* ws,
                                        const WsLayout& L, cudaStream_t st) {
  int* status = reinterpret_cast<int*>(ws + L.status);
  float* logits = reinterpret_cast<float*>(ws + L.logits);
  // the call's first kernel clears the status word (no memset node: it would end the
  // programmatic launch overlap with the previous call's last kernel)
  cudaError_t e = launch_router_logits(s, x, wg, bias, logits, st, status);
  if (e != cudaSuccess) return e;
  FfnCall c = make_ffn_call(s, x, perm_token, offsets, w13, s13, w2, s2, y_perm, ws, L, true);
  // E4M3 and MXFP4 decode tiles: the front also hands each gate/up CTA its first tile
  int4* tile1 = nullptr;
  if (c.decode && (c.fp8 || c.mxq) && c.pa.nt_up >= s.T && num_sms() <= kTile1Max) {
    tile1 = reinterpret_cast<int4*>(ws + L.tile1);
    c.a.tile1 = tile1;
  }
  e = launch_pdl(k_route_front, dim3((unsigned)(1 + (c.gather_n + 255) / 256)), dim3(256),
                 front_smem_bytes(s.T, s.E, s.k), st, logits, s.T, s.E, s.k, s.n_shared, topk_idx,
                 topk_w, offsets, perm_token, inv_slot, c.pa, c.plan, x, c.routed, s.d,
                 c.a.x_perm, status, c.a.xq, c.nq, c.mode, tile1, num_sms());
  count_launches(1);
  if (e != cudaSuccess) return e;
  if ((e = launch_passes(s, c, st)) != cudaSuccess) return e;
  return launch_combine(s, y_perm, inv_slot, topk_w, y, status, st);
}

// moe_forward: the shared expert's FFN needs neither the routing nor the permutation, so it runs
// on the second stream from the start of the call while `st` routes, permutes, gathers and runs
// the routed experts; the combine waits for both. With no shared expert, or with the
// weight-streaming GEMV in use, the four steps simply run in order.
cudaError_t launch_forward(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                           const float* bias, const void* w13, const void* s13, const void* w2,
                           const void* s2, int32_t* topk_idx, float* topk_w, int32_t* offsets,
                           int32_t* perm_token, int32_t* inv_slot, float* y_perm, uint16_t* y,
                           char* ws, const WsLayout& L, cudaStream_t st) {
  int* status = reinterpret_cast<int*>(ws + L.status);
  cudaError_t e;
  // Prefill-sized batches only: in decode the shared expert's few tiles hold SMs that the routed
  // experts' persistent tiles then wait for (measured: FP8 T=1 128.6 -> 169.4 us with the
  // overlap; T=16384 14.41 -> 14.06 ms, skewed prefill 5.33 -> 5.24 ms).
  const bool prefill = (long)s.T * s.k > 32L * s.E;
  const bool overlap = s.n_shared == 1 && s.T > 0 && prefill && tc_min_tokens() == 1;
  if (!overlap && front_applies(s) && !router_uses_tc(s))
    return launch_forward_front(s, x, wg, bias, w13, s13, w2, s2, topk_idx, topk_w, offsets,
                                perm_token, inv_slot, y_perm, y, ws, L, st);
  // A layer starts here: clear the device status word.
  if ((e = cudaMemsetAsync(status, 0, sizeof(int), st)) != cudaSuccess) return e;
  if (!overlap) {
    if ((e = launch_route(s, x, wg, bias, topk_idx, topk_w, ws, L, st)) != cudaSuccess) return e;
    if ((e = launch_permute(s, topk_idx, offsets, perm_token, inv_slot, ws, L, st)) != cudaSuccess)
      return e;
    if ((e = launch_expert_ffn(s, x, perm_token, offsets, w13, s13, w2, s2, y_perm, ws, L, st)) !=
        cudaSuccess)
      return e;
    return launch_combine(s, y_perm, inv_slot, topk_w, y, status, st);
  }
  SplitStreams* ss = nullptr;
  if ((e = split_streams(&ss)) != cudaSuccess) return e;
  std::lock_guard<std::recursive_mutex> lk(g_split_mu);
  cudaStream_t aux = ss->aux2;
  if ((e = join(aux, st, ss->ev[4])) != cudaSuccess) return e;

  // shared expert on `aux`: its tile lists, then gate/up and down
  const bool fp8 = s.wdtype == MOE_W_FP8_E4M3_B128;
  const long routed = (long)s.T * s.k;
  const bool decode = routed <= 32L * s.E;
  const TileShape ts = tile_shape(s, fp8, decode, routed);
  int32_t* rows = reinterpret_cast<int32_t*>(ws + L.shared);
  const int n = s.E + 2;
  FfnArgs a{};
  a.T = s.T; a.d = s.d; a.E = s.E; a.k = s.k; a.f = s.f; a.n_shared = 1; a.wdtype = s.wdtype;
  a.x = x; a.perm_token = perm_token; a.offsets = rows + 2 * n;
  a.w13 = w13; a.s13 = s13; a.w2 = w2; a.s2 = s2;
  a.h = reinterpret_cast<uint16_t*>(ws + L.h);
  a.x_perm = reinterpret_cast<uint16_t*>(ws + L.x_perm);
  a.y_perm = y_perm;
  a.status = status;
  const bool mxq = s.wdtype == MOE_W_MXFP4_E8M0_B32;
  if (mxq) {
    const long all_slots = routed + s.T;
    a.xq = mx::planes_at(ws + L.xq, all_slots, s.d);
    a.hq = mx::planes_at(ws + L.hq, all_slots, s.f);
  }
  // MXFP4, and E4M3 on the prefill tiles: the shared segment's rows are encoded here (two E4M3
  // terms or f16), the routed ones by the routed path's gather
  const long enc = (mxq || (fp8 && !decode)) ? (long)s.T * (s.d / 32) : 0;
  const int mode = (mxq && decode) ? kGatherMxTerms : kGatherF16;
  if ((e = launch_pdl(k_shared_plan, dim3((unsigned)(1 + (enc + 255) / 256)), dim3(256), 0, aux,
                      s.T, s.k, s.E, ts, rows, x, s.d, a.xq, a.x_perm, mode, status)) !=
      cudaSuccess)
    return e;
  count_launches(1);
  for (int pass = 0; pass < 2; ++pass) {
    const bool gateup = pass == 0;
    e = mxq ? launch_tc_mx(a, rows + pass * n, gateup, decode, aux)
        : fp8 ? launch_tc_fp8(a, rows + pass * n, gateup, decode, aux)
              : launch_tc(a, rows + pass * n, gateup, decode, aux);
    if (e != cudaSuccess) return e;
  }
  if ((e = cudaEventRecord(ss->ev[5], aux)) != cudaSuccess) return e;

  // routed experts on `st`
  if ((e = launch_route(s, x, wg, bias, topk_idx, topk_w, ws, L, st)) != cudaSuccess) return e;
  if ((e = launch_permute(s, topk_idx, offsets, perm_token, inv_slot, ws, L, st)) != cudaSuccess)
    return e;
  if ((e = launch_expert_ffn(s, x, perm_token, offsets, w13, s13, w2, s2, y_perm, ws, L, st,
                             false)) != cudaSuccess)
    return e;
  if ((e = cudaStreamWaitEvent(st, ss->ev[5], 0)) != cudaSuccess) return e;
  return launch_combine(s, y_perm, inv_slot, topk_w, y, status, st);
}

}  // namespace moe
