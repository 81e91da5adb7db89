// Internal interface of the MoE library: workspace layout, launch entry points of each kernel
// family, and small device helpers shared by the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---- workspace -----------------------------------------------------------------------------
// One scratch buffer serves the four calls of a layer:
//   status   int32[64]            device error code (first error wins) + details
//   logits   f32 [T, E]           router logits
//   hist     i32 [E, nchunk]      per (expert, 32-token chunk) counts
//   base     i32 [E, nchunk]      exclusive scan of hist: first slot of each (expert, chunk)
//   plan     i32 [kPlanRows, E+2] per-expert work prefixes of the FFN kernels + counters
//   x_perm   bf16 [T*k, d]        token rows gathered in slot order (tensor-core path input;
//                                 f16 and [T*k + S*T, d] for E4M3 and MXFP4 weights)
//   h        bf16 [T*k + S*T, f]  SiLU(gate) * up for every slot (f16 on the prefill tiles of
//                                 E4M3 and MXFP4 weights)
//   shared   i32 [3, E+2]         moe_forward: the shared expert's own tile lists and offsets
//   rtc      i32 [4] + f32 [E]    tensor-core router: its one-matrix tile plan, then |wg[e]|
// Status words after the error code: [1] tokens whose logits the tensor-core router had to
// recompute in full (a bound check failed), [2] the largest share of its error bound that a
// candidate logit used (fp32 bits); both written by that router only.
constexpr int kChunkTokens = 32;
constexpr int kStatusRouterFull = 1, kStatusRouterBoundUse = 2;
constexpr int kPlanRows = 8;

// Most CTAs a small-batch gate/up pass may be launched with (its per-CTA tile descriptors).
constexpr int kTile1Max = 1024;

struct WsLayout {
  size_t status, logits, hist, base, plan, x_perm, h, shared, xq, hq, rtc, tile1, total;
  int nchunk;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(const moe_shape& s) {
  WsLayout L{};
  const size_t T = (size_t)s.T, E = (size_t)s.E, k = (size_t)s.k;
  L.nchunk = (int)((T + kChunkTokens - 1) / kChunkTokens);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + bytes, 256); return at; };
  L.status = take(256);
  L.logits = take(T * E * 4);
  L.hist = take(E * (size_t)L.nchunk * 4);
  L.base = take(E * (size_t)L.nchunk * 4);
  L.plan = take((size_t)kPlanRows * (E + 2) * 4 + 256);
  const size_t slots = T * k + (size_t)s.n_shared * T;
  const bool mxfp4 = s.wdtype == MOE_W_MXFP4_E8M0_B32;
  const bool fp8 = s.wdtype == MOE_W_FP8_E4M3_B128;
  // bf16 weights, and E4M3 weights on the decode tiles: gathered bf16 token rows and bf16 h.
  // E4M3 and MXFP4 weights on the prefill tiles: f16 x (every slot, the shared segment
  // included) and f16 h. MXFP4 decode tiles: both as two E4M3 terms with their scales (xq, hq).
  L.x_perm = take((mxfp4 || fp8 ? slots : T * k) * (size_t)s.d * 2);
  L.h = take(slots * (size_t)s.f * 2);
  L.shared = take(3 * (E + 2) * 4);
  L.xq = take(mxfp4 ? slots * (2 * (size_t)s.d + 2 * (size_t)(s.d / 32)) : 0);
  L.hq = take(mxfp4 ? slots * (2 * (size_t)s.f + 2 * (size_t)(s.f / 32)) : 0);
  L.rtc = take(16 + E * 4);
  L.tile1 = take(kTile1Max * 16);  // small-batch gate/up: each CTA's first tile
  L.total = off;
  return L;
}

// plan rows (each E+2 int32 entries, see ffn kernels)
enum PlanRow {
  kPlanGemvUp = 0, kPlanGemvDown = 1, kPlanTcUp = 2, kPlanTcDown = 3,
  kPlanTcUpCold = 4, kPlanTcDnCold = 5,  // split prefill: the cold experts' tile lists
  kPlanSplit = 6                         // split prefill: [CTAs for cold, CTAs for the rest]
};

// ---- launchers (each returns cudaGetLastError() of its launches) ---------------------------
cudaError_t launch_route(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                         const float* bias, int32_t* topk_idx, float* topk_w, char* ws,
                         const WsLayout& L, cudaStream_t st);
// hash routing: logits as in launch_route, experts from a token-id table (router.cu)
cudaError_t launch_route_hash(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                              const float* bias, const int32_t* token_ids,
                              const int32_t* tid2eid, int vocab, int32_t* topk_idx,
                              float* topk_w, char* ws, const WsLayout& L, cudaStream_t st);
// the fp32 router's logits alone, in the defined order (router.cu); with clear_status (batches
// of at most 8 tokens), the kernel also zeroes that word after its wait, as the first kernel of
// a call. Whether a batch takes the tensor-core router instead.
cudaError_t launch_router_logits(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                 const float* bias, float* logits, cudaStream_t st,
                                 int* clear_status = nullptr);
bool router_uses_tc(const moe_shape& s);
cudaError_t launch_permute(const moe_shape& s, const int32_t* topk_idx, int32_t* offsets,
                           int32_t* perm_token, int32_t* inv_slot, char* ws, const WsLayout& L,
                           cudaStream_t st);
cudaError_t launch_expert_ffn(const moe_shape& s, const uint16_t* x, const int32_t* perm_token,
                              const int32_t* offsets, const void* w13, const void* s13,
                              const void* w2, const void* s2, float* y_perm, char* ws,
                              const WsLayout& L, cudaStream_t st, bool with_shared = true);
// the whole layer, the shared expert's FFN on a second stream (ffn.cu)
cudaError_t launch_forward(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                           const float* bias, const void* w13, const void* s13, const void* w2,
                           const void* s2, int32_t* topk_idx, float* topk_w, int32_t* offsets,
                           int32_t* perm_token, int32_t* inv_slot, float* y_perm, uint16_t* y,
                           char* ws, const WsLayout& L, cudaStream_t st);
cudaError_t launch_combine(const moe_shape& s, const float* y_perm, const int32_t* inv_slot,
                           const float* topk_w, uint16_t* y, int* status, cudaStream_t st);

int num_sms();

// router with its logits scratch in a fixed device array (router.cu)
size_t route_noalloc_max_logits();
cudaError_t launch_route_noalloc(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                 const float* bias, int32_t* topk_idx, float* topk_w,
                                 cudaStream_t st);

// a wait that nothing completes, bounded by limit_ns (selftest.cu); records the timeout status
cudaError_t launch_selftest_bounded_wait(int* status, uint64_t limit_ns, cudaStream_t st);

// profiling hooks (capi.cu): kernel launch counter and per-call phase events
void count_launches(int n);
struct PhaseEvents {
  cudaEvent_t begin = nullptr, mid = nullptr, end = nullptr;
};
PhaseEvents profile_phase_events();  // all null unless a profiling session is on

// ---- programmatic dependent launch -------------------------------------------------------
// Every kernel of the layer is launched so that it may start while the kernel before it in the
// stream is still finishing. Each kernel first does the set-up that touches no global memory
// (shared-memory barriers, TMEM allocation, tensor-map prefetch), then pdl_wait(), which returns
// once the previous kernel has completed and its writes are visible, and only then reads its
// inputs. A kernel launched without the attribute passes pdl_wait() at once.
#ifdef __CUDACC__
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// The same launch with blocks grouped into clusters of `cluster` consecutive blocks along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t st, unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Wait for the previous kernel in the stream (all its writes visible), then let the next
// kernel's blocks be scheduled as this grid's blocks are placed.
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// ---- device helpers ------------------------------------------------------------------------
#ifdef __CUDACC__
// Hint: bring the 128-byte line holding p into L2. Issued before griddepcontrol.wait for data
// the previous kernel may still be writing, it only warms the address translation and L2 (the
// point of coherence): every value is still read after the wait.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// prefetch_l2 over [p, p + bytes), the block's threads taking one line each in turn
__device__ __forceinline__ void prefetch_l2_span(const void* p, size_t bytes) {
  const char* c = static_cast<const char*>(p);
  for (size_t o = (size_t)threadIdx.x * 128; o < bytes; o += (size_t)blockDim.x * 128)
    prefetch_l2(c + o);
}

// One line every 64 KB of [p, p + bytes): the address translations of a larger buffer.
__device__ __forceinline__ void prefetch_l2_pages(const void* p, size_t bytes) {
  const char* c = static_cast<const char*>(p);
  for (size_t o = (size_t)threadIdx.x << 16; o < bytes; o += (size_t)blockDim.x << 16)
    prefetch_l2(c + o);
}

__device__ __forceinline__ void record_error(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// element i (0..7) of eight packed bf16 values, as fp32 (exact)
__device__ __forceinline__ float bf16x8_elem(const uint4& v, int i) {
  const uint32_t w = i < 2 ? v.x : i < 4 ? v.y : i < 6 ? v.z : v.w;
  return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

__device__ __forceinline__ uint4 ldg_u4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// streamed once: do not keep in L1
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
  // round to nearest even via the hardware conversion
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

// fp32 -> f16, round to nearest even, magnitudes beyond the largest finite f16 saturate to it.
__device__ __forceinline__ uint16_t f32_to_f16_satfinite(float v) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(0.f), "f"(v));
  return (uint16_t)(r & 0xFFFFu);
}

// Exclusive scan of one int per thread over a block of up to 1024 threads; returns the
// thread's exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_tot[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    int w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_tot[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int warp_prefix = wid ? warp_tot[wid - 1] : 0;
  *total = warp_tot[((blockDim.x + 31) >> 5) - 1];
  __syncthreads();
  return warp_prefix + incl - v;
}

// Three exclusive scans in one pass (each component as block_exclusive_scan would give it).
__device__ __forceinline__ int3 block_exclusive_scan3(int3 v, int3* total) {
  __shared__ int3 warp_tot3[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int3 incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nx = __shfl_up_sync(0xffffffffu, incl.x, o);
    const int ny = __shfl_up_sync(0xffffffffu, incl.y, o);
    const int nz = __shfl_up_sync(0xffffffffu, incl.z, o);
    if (lane >= o) {
      incl.x += nx;
      incl.y += ny;
      incl.z += nz;
    }
  }
  if (lane == 31) warp_tot3[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    int3 w = lane < nw ? warp_tot3[lane] : make_int3(0, 0, 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nx = __shfl_up_sync(0xffffffffu, w.x, o);
      const int ny = __shfl_up_sync(0xffffffffu, w.y, o);
      const int nz = __shfl_up_sync(0xffffffffu, w.z, o);
      if (lane >= o) {
        w.x += nx;
        w.y += ny;
        w.z += nz;
      }
    }
    warp_tot3[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int3 wp = wid ? warp_tot3[wid - 1] : make_int3(0, 0, 0);
  *total = warp_tot3[((blockDim.x + 31) >> 5) - 1];
  __syncthreads();
  return make_int3(wp.x + incl.x - v.x, wp.y + incl.y - v.y, wp.z + incl.z - v.z);
}
#endif

}  // namespace moe
