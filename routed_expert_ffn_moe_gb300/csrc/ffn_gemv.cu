// Expert FFN, weight-streaming path: for experts that received only a few tokens.
//
// The pages: in small-batch decode each expert gets few tokens, its GEMMs are thin and the
// expert weights must still stream from HBM, so the layer is bandwidth-bound
// ("DeepSeek-V4-Pro on NVIDIA H200", 0.1.2 and 0.2.2 step D6; "DeepSeek-V3/R1 推理系统完全拆解",
// 问题一; "第 6 章 超節點", 6.1.2: 90.1 us of weight reads vs 0.31 us of math at batch 1).
// So this path is a GEMV: each weight row is read once with 16-byte streaming loads and dotted
// with every token of the expert's group (up to kGroup tokens, staged in shared memory).
// SiLU(gate) * up is fused into the gate/up pass; FP8 block scales are applied per 16-element
// chunk (a chunk never crosses a 128-column block).
#include <cuda_fp8.h>

#include "ffn.h"

namespace moe {
namespace {

constexpr int kGroup = 4;        // tokens per work item
constexpr int kRowsPerItem = 64; // output rows per work item (8 warps x 8 rows)
constexpr int kWarps = 8;

// Converts 16 bytes of weights to fp32: 8 bf16 or 16 E4M3 values.
template <bool FP8>
__device__ __forceinline__ void weights_to_f32(const uint4& v, float* out) {
  if constexpr (FP8) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[q] & 0xFFFFu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[q] >> 16), __NV_E4M3);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      out[4 * q + 0] = a.x;
      out[4 * q + 1] = a.y;
      out[4 * q + 2] = b.x;
      out[4 * q + 3] = b.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = bf16x8_elem(v, i);
  }
}

// GATEUP: input rows are tokens x[t] (width d); expert rows r (gate) and f + r (up) of w13;
//         output h[slot][r] = bf16(SiLU(gate) * up).
// !GATEUP: input rows are h[slot] (width f); expert rows r and r + 1 of w2;
//         output y_perm[slot][r], y_perm[slot][r + 1] (fp32).
template <bool FP8, bool GATEUP>
__global__ void __launch_bounds__(256) k_gemv(FfnArgs a, const int32_t* __restrict__ prefix) {
  pdl_wait_then_release();
  constexpr int CH = FP8 ? 16 : 8;  // weight elements per 16-byte chunk
  extern __shared__ uint4 xs_u4[];  // [kGroup][K] bf16
  const int K = GATEUP ? a.d : a.f;          // input width
  const int N = GATEUP ? a.f : a.d;          // output rows per expert
  const int E1 = a.E + a.n_shared;
  const long routed = (long)a.T * a.k;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int total = prefix[E1];
  const int per_group = N / kRowsPerItem;
  const int kch = K / 8;                     // 16-byte chunks of one bf16 input row
  const int nch = K / CH;                    // 16-byte chunks of one weight row
  const size_t wrow_bytes = (size_t)K * (FP8 ? 1 : 2);
  const size_t wexp_rows = GATEUP ? 2 * (size_t)a.f : (size_t)a.d;
  const int sblk_cols = K / 128;
  const char* Wb = reinterpret_cast<const char*>(GATEUP ? a.w13 : a.w2);
  const float* Sb = static_cast<const float*>(GATEUP ? a.s13 : a.s2);

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int lo = 0, hi = E1;  // largest e with prefix[e] <= item
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= item) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int local = item - prefix[e];
    const int grp = local / per_group, rb = local % per_group;
    const int seg0 = a.offsets[e];
    const int cnt = a.offsets[e + 1] - seg0;
    const int tok0 = grp * kGroup;
    const int ntok = min(kGroup, cnt - tok0);

    __syncthreads();  // previous item's readers are done with xs
    for (int i = threadIdx.x; i < ntok * kch; i += blockDim.x) {
      const int tt = i / kch, c = i - tt * kch;
      const long slot = seg0 + tok0 + tt;
      const uint16_t* src;
      if (GATEUP) {
        long t = slot < routed ? a.perm_token[slot] : slot - routed;
        if (t < 0 || t >= a.T) {
          record_error(a.status, MOE_ERR_DEVICE_BOUNDS);
          t = 0;
        }
        src = a.x + t * a.d;
      } else {
        src = a.h + slot * a.f;
      }
      xs_u4[tt * kch + c] = ldg_u4(src + 8 * c);
    }
    __syncthreads();

    const char* We = Wb + (size_t)e * wexp_rows * wrow_bytes;
    const float* Se = FP8 ? Sb + (size_t)e * (wexp_rows / 128) * sblk_cols : nullptr;
    const int rows_per_warp = kRowsPerItem / kWarps;
    for (int rr = 0; rr < rows_per_warp; rr += (GATEUP ? 1 : 2)) {
      const int r = rb * kRowsPerItem + wid * rows_per_warp + rr;
      const int row0 = r;
      const int row1 = GATEUP ? a.f + r : r + 1;
      const char* w0 = We + (size_t)row0 * wrow_bytes;
      const char* w1 = We + (size_t)row1 * wrow_bytes;
      float acc0[kGroup], acc1[kGroup];
#pragma unroll
      for (int tt = 0; tt < kGroup; ++tt) acc0[tt] = acc1[tt] = 0.f;
#pragma unroll 4
      for (int c = lane; c < nch; c += 32) {
        const uint4 v0 = ld_stream_u4(w0 + (size_t)c * 16);
        const uint4 v1 = ld_stream_u4(w1 + (size_t)c * 16);
        float f0[CH], f1[CH];
        weights_to_f32<FP8>(v0, f0);
        weights_to_f32<FP8>(v1, f1);
        float s0 = 1.f, s1 = 1.f;
        if constexpr (FP8) {
          const int kb = (c * CH) >> 7;
          s0 = __ldg(Se + (size_t)(row0 >> 7) * sblk_cols + kb);
          s1 = __ldg(Se + (size_t)(row1 >> 7) * sblk_cols + kb);
        }
#pragma unroll
        for (int tt = 0; tt < kGroup; ++tt) {
          if (tt < ntok) {
            float xv[CH];
#pragma unroll
            for (int q = 0; q < CH / 8; ++q) {
              const uint4 xc = xs_u4[tt * kch + c * (CH / 8) + q];
#pragma unroll
              for (int i = 0; i < 8; ++i) xv[8 * q + i] = bf16x8_elem(xc, i);
            }
            if constexpr (FP8) {
              float p0 = 0.f, p1 = 0.f;
#pragma unroll
              for (int i = 0; i < CH; ++i) {
                p0 = __fmaf_rn(f0[i], xv[i], p0);
                p1 = __fmaf_rn(f1[i], xv[i], p1);
              }
              acc0[tt] = __fmaf_rn(s0, p0, acc0[tt]);
              acc1[tt] = __fmaf_rn(s1, p1, acc1[tt]);
            } else {
#pragma unroll
              for (int i = 0; i < CH; ++i) {
                acc0[tt] = __fmaf_rn(f0[i], xv[i], acc0[tt]);
                acc1[tt] = __fmaf_rn(f1[i], xv[i], acc1[tt]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
        for (int tt = 0; tt < kGroup; ++tt) {
          acc0[tt] += __shfl_xor_sync(0xffffffffu, acc0[tt], off);
          acc1[tt] += __shfl_xor_sync(0xffffffffu, acc1[tt], off);
        }
#pragma unroll
      for (int tt = 0; tt < kGroup; ++tt) {
        if (lane == tt && tt < ntok) {
          const long slot = seg0 + tok0 + tt;
          if (GATEUP) {
            const float g = acc0[tt], u = acc1[tt];
            const float silu = g / (1.0f + __expf(-g));
            a.h[slot * a.f + r] = f32_to_bf16_rn(silu * u);
          } else {
            a.y_perm[slot * a.d + r] = acc0[tt];
            a.y_perm[slot * a.d + r + 1] = acc1[tt];
          }
        }
      }
    }
  }
}

template <bool FP8, bool GATEUP>
cudaError_t launch_one(const FfnArgs& a, const int32_t* prefix, int grid, cudaStream_t st) {
  const int K = GATEUP ? a.d : a.f;
  const size_t smem = (size_t)kGroup * K * 2;
  cudaError_t e = cudaFuncSetAttribute(k_gemv<FP8, GATEUP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_gemv<FP8, GATEUP><<<grid, 32 * kWarps, smem, st>>>(a, prefix);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

int gemv_items_per_group(bool gateup, int d, int f) {
  return (gateup ? f : d) / kRowsPerItem;
}
int gemv_group_tokens() { return kGroup; }

cudaError_t launch_gemv(const FfnArgs& a, const int32_t* prefix_up, const int32_t* prefix_down,
                        bool gateup, int max_items, cudaStream_t st) {
  if (max_items <= 0) return cudaSuccess;
  const int K = gateup ? a.d : a.f;
  const int per_sm = K * kGroup * 2 <= 64 * 1024 ? 3 : 1;
  int grid = num_sms() * per_sm;
  if (grid > max_items) grid = max_items;
  const bool fp8 = a.wdtype == MOE_W_FP8_E4M3_B128;
  if (gateup)
    return fp8 ? launch_one<true, true>(a, prefix_up, grid, st)
               : launch_one<false, true>(a, prefix_up, grid, st);
  return fp8 ? launch_one<true, false>(a, prefix_down, grid, st)
             : launch_one<false, false>(a, prefix_down, grid, st);
}

}  // namespace moe
