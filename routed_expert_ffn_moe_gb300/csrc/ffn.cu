// Expert FFN orchestration: a device-side work plan from the expert segment sizes, then the
// gate/up pass and the down pass.
//
// Expert segment sizes exist only on the device (they come from the router), so the host never
// waits for them: a one-block plan kernel turns expert_offsets into per-expert prefix sums of
// work items, and the persistent FFN kernels walk those items.
#include "ffn.h"

namespace moe {
namespace {

// plan[kPlanGemvUp][e] / plan[kPlanGemvDown][e]: exclusive prefix over experts of the number of
// weight-streaming work items; entry E1 is the total.
__global__ void __launch_bounds__(1024) k_ffn_plan(const int32_t* __restrict__ offsets, int E,
                                                   int n_shared, int items_up, int items_down,
                                                   int group, int32_t* __restrict__ plan,
                                                   int plan_stride) {
  const int E1 = E + n_shared;
  int run_up = 0, run_dn = 0;
  for (int b = 0; b < E1; b += blockDim.x) {
    const int e = b + threadIdx.x;
    int n_up = 0, n_dn = 0;
    if (e < E1) {
      const int cnt = offsets[e + 1] - offsets[e];
      const int groups = cnt > 0 ? (cnt + group - 1) / group : 0;
      n_up = groups * items_up;
      n_dn = groups * items_down;
    }
    int tot_up, tot_dn;
    const int p_up = block_exclusive_scan(n_up, &tot_up);
    const int p_dn = block_exclusive_scan(n_dn, &tot_dn);
    if (e < E1) {
      plan[kPlanGemvUp * plan_stride + e] = run_up + p_up;
      plan[kPlanGemvDown * plan_stride + e] = run_dn + p_dn;
    }
    run_up += tot_up;
    run_dn += tot_dn;
  }
  if (threadIdx.x == 0) {
    plan[kPlanGemvUp * plan_stride + E1] = run_up;
    plan[kPlanGemvDown * plan_stride + E1] = run_dn;
  }
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
  const int stride = s.E + 2;
  const int group = gemv_group_tokens();
  const int items_up = gemv_items_per_group(true, s.d, s.f);
  const int items_dn = gemv_items_per_group(false, s.d, s.f);
  const PhaseEvents ev = profile_phase_events();
  k_ffn_plan<<<1, 1024, 0, st>>>(offsets, s.E, s.n_shared, items_up, items_dn, group, plan, stride);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ev.begin) cudaEventRecord(ev.begin, st);
  // Upper bound on the number of groups: every slot in its own group plus one partial group
  // per expert.
  const long slots = (long)s.T * s.k + (long)s.n_shared * s.T;
  const long max_groups = (slots + group - 1) / group + s.E + s.n_shared;
  const long max_up = max_groups * items_up, max_dn = max_groups * items_dn;
  e = launch_gemv(a, plan + kPlanGemvUp * stride, plan + kPlanGemvDown * stride, true,
                  (int)(max_up < (1L << 30) ? max_up : (1L << 30)), st);
  if (e != cudaSuccess) return e;
  if (ev.mid) cudaEventRecord(ev.mid, st);
  e = launch_gemv(a, plan + kPlanGemvUp * stride, plan + kPlanGemvDown * stride, false,
                  (int)(max_dn < (1L << 30) ? max_dn : (1L << 30)), st);
  if (ev.end) cudaEventRecord(ev.end, st);
  return e;
}

}  // namespace moe
