// Expert FFN orchestration: a device-side work plan from the expert segment sizes, then the
// gate/up pass and the down pass, each split between the tensor-core grouped GEMM (experts with
// at least tc_min tokens) and the weight-streaming GEMV (experts with fewer).
//
// Expert segment sizes exist only on the device (they come from the router), so the host never
// waits for them: a one-block plan kernel turns expert_offsets into per-expert prefix sums of
// work items for each kernel, and the persistent FFN kernels walk those lists.
#include <climits>
#include <cstdlib>

#include "ffn.h"

namespace moe {
namespace {

struct PlanArgs {
  int E, n_shared, tc_min;
  int group, items_up, items_dn;   // weight-streaming: tokens per item, items per group
  int nt_up, nt_dn, mt_up, mt_dn;  // tensor-core: tokens per tile, weight tiles per expert
  int stride;
};

// plan[row][e]: exclusive prefix over experts of the work of each kernel; entry E1 = total.
__global__ void __launch_bounds__(1024) k_ffn_plan(const int32_t* __restrict__ offsets,
                                                   PlanArgs a, int32_t* __restrict__ plan) {
  pdl_wait_then_release();
  const int E1 = a.E + a.n_shared;
  int run[4] = {0, 0, 0, 0};
  for (int b = 0; b < E1; b += blockDim.x) {
    const int e = b + threadIdx.x;
    int n[4] = {0, 0, 0, 0};
    if (e < E1) {
      const int cnt = offsets[e + 1] - offsets[e];
      if (cnt >= a.tc_min) {
        n[kPlanTcUp] = (cnt + a.nt_up - 1) / a.nt_up * a.mt_up;
        n[kPlanTcDown] = (cnt + a.nt_dn - 1) / a.nt_dn * a.mt_dn;
      } else if (cnt > 0) {
        const int groups = (cnt + a.group - 1) / a.group;
        n[kPlanGemvUp] = groups * a.items_up;
        n[kPlanGemvDown] = groups * a.items_dn;
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      int tot;
      const int pre = block_exclusive_scan(n[r], &tot);
      if (e < E1) plan[r * a.stride + e] = run[r] + pre;
      run[r] += tot;
    }
  }
  if (threadIdx.x == 0)
    for (int r = 0; r < 4; ++r) plan[r * a.stride + E1] = run[r];
}

// x_perm[s] = x[perm_token[s]] for every routed slot: the tensor-core path's token tiles are
// contiguous rows for TMA.
__global__ void __launch_bounds__(256) k_gather_rows(const uint16_t* __restrict__ x,
                                                     const int32_t* __restrict__ perm_token,
                                                     int T, long routed, int d,
                                                     uint16_t* __restrict__ x_perm, int* status) {
  pdl_wait_then_release();
  const int d8 = d >> 3;
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= routed * d8) return;
  const long s = i / d8;
  const int c = (int)(i - s * d8);
  int t = __ldg(perm_token + s);
  if (t < 0 || t >= T) {
    record_error(status, MOE_ERR_DEVICE_BOUNDS);
    t = 0;
  }
  reinterpret_cast<uint4*>(x_perm + s * d)[c] =
      __ldg(reinterpret_cast<const uint4*>(x + (long)t * d) + c);
}

// Phase events are recorded as external events while the stream is being captured into a CUDA
// graph (so every replay records them) and as plain events otherwise.
void record_phase(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cap);
  cudaEventRecordWithFlags(ev, st,
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

}  // namespace

cudaError_t launch_expert_ffn(const moe_shape& s, const uint16_t* x, const int32_t* perm_token,
                              const int32_t* offsets, const void* w13, const float* s13,
                              const void* w2, const float* s2, float* y_perm, char* ws,
                              const WsLayout& L, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  FfnArgs a{};
  a.T = s.T; a.d = s.d; a.E = s.E; a.k = s.k; a.f = s.f; a.n_shared = s.n_shared;
  a.wdtype = s.wdtype;
  a.x = x; a.perm_token = perm_token; a.offsets = offsets;
  a.w13 = w13; a.s13 = s13; a.w2 = w2; a.s2 = s2;
  a.h = reinterpret_cast<uint16_t*>(ws + L.h);
  a.x_perm = reinterpret_cast<uint16_t*>(ws + L.x_perm);
  a.y_perm = y_perm;
  a.status = reinterpret_cast<int*>(ws + L.status);
  int32_t* plan = reinterpret_cast<int32_t*>(ws + L.plan);

  // Experts with at least tc_min tokens go to the tensor-core GEMM, the rest to the
  // weight-streaming GEMV. Both stream each weight byte once; the tensor-core kernel does so at
  // full HBM rate from one token up, so by default it takes every expert. MOE_TC_MIN_TOKENS
  // moves the split (a tuning and testing knob; results agree within rounding either way).
  const int tc_min = tc_min_tokens();
  const bool fp8 = s.wdtype == MOE_W_FP8_E4M3_B128;
  const long routed = (long)s.T * s.k;
  const bool decode = routed <= 32L * s.E;  // at most ~32 tokens per routed expert on average
  const bool use_tc = tc_min < INT_MAX;
  const bool use_gemv = tc_min > 1;
  PlanArgs pa{};
  pa.E = s.E; pa.n_shared = s.n_shared;
  pa.tc_min = tc_min;
  pa.group = gemv_group_tokens();
  pa.items_up = gemv_items_per_group(true, s.d, s.f);
  pa.items_dn = gemv_items_per_group(false, s.d, s.f);
  pa.nt_up = fp8 ? tc_fp8_tile_tokens(true, decode, routed, s.E) : tc_tile_tokens(true, decode);
  pa.nt_dn = fp8 ? tc_fp8_tile_tokens(false, decode, routed, s.E) : tc_tile_tokens(false, decode);
  pa.mt_up = s.f / 128;
  pa.mt_dn = s.d / tc_tile_rows(false, decode, s.d);
  if (!fp8) {
    pa.mt_up = tc_plan_mtiles(true, decode, s.d, s.f);
    pa.mt_dn = tc_plan_mtiles(false, decode, s.d, s.f);
  } else if (!decode) {
    pa.mt_up = tc_fp8_wide_plan_mtiles(true, s.d, s.f);
    pa.mt_dn = tc_fp8_wide_plan_mtiles(false, s.d, s.f);
  }
  pa.stride = s.E + 2;
  const int stride = pa.stride;

  const PhaseEvents ev = profile_phase_events();
  cudaError_t e = launch_pdl(k_ffn_plan, dim3(1), dim3(1024), 0, st, offsets, pa, plan);
  count_launches(1);
  if (e != cudaSuccess) return e;
  if (use_tc && routed > 0) {
    const long n = routed * (s.d / 8);
    e = launch_pdl(k_gather_rows, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, x,
                   perm_token, s.T, routed, s.d, a.x_perm, a.status);
    count_launches(1);
    if (e != cudaSuccess) return e;
  }
  if (ev.begin) record_phase(ev.begin, st);

  // Upper bound on the weight-streaming work: every slot in its own group plus one partial
  // group per expert (the device-side totals are usually far smaller).
  const long slots = routed + (long)s.n_shared * s.T;
  const long max_groups = (slots + pa.group - 1) / pa.group + s.E + s.n_shared;
  const auto cap = [](long v) { return (int)(v < (1L << 30) ? v : (1L << 30)); };
  const int max_up = use_gemv ? cap(max_groups * pa.items_up) : 0;
  const int max_dn = use_gemv ? cap(max_groups * pa.items_dn) : 0;
  const auto tc = [&](bool gateup, const int32_t* prefix) {
    return fp8 ? launch_tc_fp8(a, prefix, gateup, decode, st)
               : launch_tc(a, prefix, gateup, decode, st);
  };

  if (use_tc) e = tc(true, plan + kPlanTcUp * stride);
  if (e == cudaSuccess)
    e = launch_gemv(a, plan + kPlanGemvUp * stride, plan + kPlanGemvDown * stride, true, max_up, st);
  if (e != cudaSuccess) return e;
  if (ev.mid) record_phase(ev.mid, st);
  if (use_tc) e = tc(false, plan + kPlanTcDown * stride);
  if (e == cudaSuccess)
    e = launch_gemv(a, plan + kPlanGemvUp * stride, plan + kPlanGemvDown * stride, false, max_dn, st);
  if (ev.end) record_phase(ev.end, st);
  return e;
}

}  // namespace moe
