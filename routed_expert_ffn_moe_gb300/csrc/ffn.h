// Internal interface of the expert-FFN kernels (weight-streaming and tensor-core paths).
#pragma once

#include "internal.h"
#include "mx_common.cuh"

namespace moe {

struct FfnArgs {
  int T, d, E, k, f, n_shared, wdtype;
  const uint16_t* x;           // [T, d] bf16
  const int32_t* perm_token;   // [T*k]
  const int32_t* offsets;      // [E+2]
  const void* w13;             // [E+S, 2f, d]
  const void* s13;             // FP8 (fp32) or MXFP4 (E8M0) scales, or null
  const void* w2;              // [E+S, d, f]
  const void* s2;
  uint16_t* h;                 // [slots, f] bf16 (workspace)
  uint16_t* x_perm;            // [T*k, d] bf16 (workspace)
  float* y_perm;               // [slots, d] fp32
  int* status;                 // device error word
  mx::Planes xq, hq;           // MXFP4 weights: x and h as E4M3 terms (workspace), [slots, d|f]
  // small-batch front: each gate/up CTA's first tile {e, m-tile, slot0, ntok | more << 16}
  // (more: the pass has more tiles than CTAs), written by the front; or null
  const int4* tile1;
};

// weight-streaming path (ffn_gemv.cu)
int gemv_items_per_group(bool gateup, int d, int f);
int gemv_group_tokens();
cudaError_t launch_gemv(const FfnArgs& a, const int32_t* prefix_up, const int32_t* prefix_down,
                        bool gateup, int max_items, cudaStream_t st);

// tensor-core path (ffn_tc.cu): bf16 weights
int tc_tile_tokens(bool gateup, bool decode);
int tc_cold_tile_tokens();  // tokens per tile of a split prefill's cold list
int tc_tile_rows(bool gateup, bool decode, int d);  // weight rows per tile
// plan units (weight tiles, or cluster pairs of them) per expert
int tc_plan_mtiles(bool gateup, bool decode, int d, int f);
cudaError_t launch_tc(const FfnArgs& a, const int32_t* prefix, bool gateup, bool decode,
                      cudaStream_t st, const int32_t* active = nullptr, bool cold = false);

// tensor-core path (ffn_tc_fp8.cu): E4M3 weights dequantised into TMEM
int tc_fp8_tile_tokens(bool gateup, bool decode, long routed, int E);
int tc_fp8_decode_down_rows(int d);  // weight rows per down tile of the decode tiles
cudaError_t launch_tc_fp8(const FfnArgs& a, const int32_t* prefix, bool gateup, bool decode,
                          cudaStream_t st);
// tensor-core path (ffn_tc_mxfp4.cu): MXFP4 weights fed to block-scaled MMAs as stored
int tc_mx_tile_tokens(bool decode, long routed, int E);
int tc_mx_down_rows(bool decode, int d);  // weight rows per down tile
cudaError_t launch_tc_mx(const FfnArgs& a, const int32_t* prefix, bool gateup, bool decode,
                         cudaStream_t st);
// wide-tile variant (ffn_tc_fp8_wide.cu): E4M3 weights dequantised to bf16 into TMEM
int tc_fp8_wide_tile_tokens();
// plan units (weight tiles, or cluster pairs of them) per expert in a prefill-tile pass
int tc_fp8_wide_plan_mtiles(bool gateup, int d, int f);
cudaError_t launch_tc_fp8_wide(const FfnArgs& a, const int32_t* prefix, bool gateup,
                               cudaStream_t st);
// the same prefill tiles for MXFP4 weights (dequantised to f16; x and h as f16 rows)
cudaError_t launch_tc_mx_wide(const FfnArgs& a, const int32_t* prefix, bool gateup,
                              cudaStream_t st);

}  // namespace moe
