// Expert FFN, tensor-core path for FP8 E4M3 expert weights, wide-tile variant for large token
// batches (W8A16). Same passages and warp roles as ffn_tc_fp8.cu; the difference is where the
// block scale goes. With 64-128 tokens per tile, scaling the token rows would cost as much as
// converting the weights, so here the weights themselves are dequantised: eight converter warps
// turn each 128x128 E4M3 block into bf16(code * scale) and store it straight into TMEM with
// tcgen05.st (one weight row per TMEM lane), and the MMA (kind::f16, bf16 x bf16 -> fp32) reads
// A from TMEM and the bf16 token tile from shared memory. Each weight is rounded once to bf16
// (relative error <= 2^-9).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "tc_common.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kQK = 128;                          // K per stage = one scale block
constexpr uint32_t kQTileBytes = kBM * kQK;       // 16 KB of E4M3 codes
constexpr int kConvWarps = 8;                     // two per TMEM lane quadrant
constexpr int kThreadsQ = 32 * (6 + kConvWarps);  // producer, MMA, 4 epilogue, converters
constexpr uint32_t kACols = kQK / 2;              // TMEM columns of one 128 x 128 bf16 tile

template <bool GATEUP, int NT, int STAGES, int ASTAGES>
struct SmemQ {
  static constexpr int kA = GATEUP ? 2 : 1;
  static constexpr uint32_t kBHalf = (uint32_t)NT * kBK * 2;   // NT rows x 64 K bf16
  static constexpr uint32_t kStageBytes = kA * kQTileBytes + 2 * kBHalf;
  static constexpr uint32_t kTilesBytes = STAGES * kStageBytes;
  static constexpr uint32_t kBarBytes = 8 * (2 * STAGES + 2 * ASTAGES + 4) + 16;
  static constexpr uint32_t kTotal = kTilesBytes + kBarBytes + 1024;
  static constexpr uint32_t kAccCols = GATEUP ? 2 * NT : NT;
  static constexpr uint32_t kAStageCols = kA * kACols;
  static constexpr uint32_t kUsedCols = 2 * kAccCols + ASTAGES * kAStageCols;
  static constexpr uint32_t kTmemCols =
      kUsedCols <= 32 ? 32 : kUsedCols <= 64 ? 64 : kUsedCols <= 128 ? 128
      : kUsedCols <= 256 ? 256 : 512;
};

// Two E4M3 codes (low byte first) times the block scale, as a bf16 pair (low element first).
__device__ __forceinline__ uint32_t dequant2(uint32_t two, float s) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * s, f.y * s);
  return *reinterpret_cast<const uint32_t*>(&b);
}

template <bool GATEUP, int NT, int STAGES, int ASTAGES>
__global__ void __launch_bounds__(kThreadsQ, 1)
    k_tc_ffn_fp8_wide(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b0,
                 const __grid_constant__ CUtensorMap tm_b1, const TcParams p,
                 const float* __restrict__ scales) {
  using S = SmemQ<GATEUP, NT, STAGES, ASTAGES>;
  static_assert(S::kUsedCols <= 512, "TMEM columns");
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 256, "MMA N");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kTilesBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* a_full = empty + STAGES;
  uint64_t* a_empty = a_full + ASTAGES;
  uint64_t* acc_full = a_empty + ASTAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E1 = p.E + p.n_shared;
  const int total = __ldg(p.prefix + E1);
  const int kblocks = p.K / kQK;
  constexpr uint32_t kConvThreads = 32 * kConvWarps;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConvThreads + 1);  // every converter thread + the MMA commit
    }
    for (int s = 0; s < ASTAGES; ++s) {
      mbar_init(&a_full[s], kConvThreads);
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_b0);
    prefetch_tmap(&tm_b1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint32_t acol0 = 2 * S::kAccCols;  // first TMEM column of the A ring

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        Tile t;
        decode_tile<GATEUP, NT>(p, tile, t);
        const int nbox = (t.ntok + kBoxRows - 1) / kBoxRows;
        const uint32_t bytes = S::kA * kQTileBytes + (uint32_t)nbox * 2 * kBBoxBytes;
        const int wrow = t.e * p.rows_per_expert + t.mt * kBM;
        const CUtensorMap* bmap = (GATEUP && t.shared) ? &tm_b1 : &tm_b0;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          uint8_t* st = smem + stage * S::kStageBytes;
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_2d(st, &tm_w, &full[stage], kb * kQK, wrow, pol_w);
          if (GATEUP) tma_load_2d(st + kQTileBytes, &tm_w, &full[stage], kb * kQK, wrow + p.f, pol_w);
          uint8_t* bt = st + S::kA * kQTileBytes;
          for (int i = 0; i < nbox; ++i)
            for (int hk = 0; hk < 2; ++hk)
              tma_load_2d(bt + hk * S::kBHalf + i * kBBoxBytes, bmap, &full[stage],
                          kb * kQK + hk * kBK, t.brow0 + i * kBoxRows, pol_b);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t issued_phase = (s < (int)stage) ? phase : (phase ^ 1u);
        drain_bar(&full[s], issued_phase, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, astage = 0, aphase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        Tile t;
        decode_tile<GATEUP, NT>(p, tile, t);
        const int npad = (t.ntok + 15) & ~15;
        const uint32_t idesc = idesc_bf16(kBM, npad);
        if (!wait_bar(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc * S::kAccCols;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(&full[stage], phase, abort_flag, p.status) ||
              !wait_bar(&a_full[astage], aphase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = tmem_base + acol0 + astage * S::kAStageCols;
          const uint32_t bst = smem_u32(smem + stage * S::kStageBytes + S::kA * kQTileBytes);
#pragma unroll
          for (int kk = 0; kk < kQK / 16; ++kk) {
            const uint64_t bd = sw128_desc(bst + (kk >> 2) * S::kBHalf) + 2 * (kk & 3);
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            mma_ts(d0, a0 + kk * 8, bd, idesc, accum);
            if (GATEUP) mma_ts(d0 + NT, a0 + kACols + kk * 8, bd, idesc, accum);
          }
          mma_commit(&empty[stage]);    // token rows consumed
          mma_commit(&a_empty[astage]); // dequantised weights consumed
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          if (++astage == ASTAGES) { astage = 0; aphase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else if (warp < 6) {
    // ---------------- epilogue (warps 2..5) ----------------
    run_epilogue<GATEUP, NT, S::kAccCols>(p, total, tmem_base, acc_full, acc_empty, abort_flag);
  } else {
    // ---------------- dequantisers (warps 6..13) ----------------
    const int q = warp & 3;                   // TMEM lane quadrant
    const int hk = (warp - 6) >> 2;           // which 64-wide half of the stage's K
    const int row = q * 32 + lane;            // weight row within the tile = TMEM lane
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    const int kbl = p.K / 128;                // scale blocks along K
    uint32_t stage = 0, phase = 0, astage = 0, aphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      Tile t;
      decode_tile<GATEUP, NT>(p, tile, t);
      const float* sc = scales + (size_t)t.e * (p.rows_per_expert / 128) * kbl;
      const int rb_g = t.mt, rb_u = p.f / 128 + t.mt;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_bar(&full[stage], phase, abort_flag, p.status) ||
            !wait_bar(&a_empty[astage], aphase ^ 1u, abort_flag, p.status)) { ok = false; break; }
        const uint32_t st = smem_u32(smem + stage * S::kStageBytes);
        uint4 raw[S::kA][4];
#pragma unroll
        for (int o = 0; o < S::kA; ++o)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t chunk = (uint32_t)(4 * hk + j) ^ (uint32_t)(row & 7);  // 128B swizzle
            raw[o][j] = lds_u4(st + o * kQTileBytes + row * 128 + (chunk << 4));
          }
        mbar_arrive(&empty[stage]);           // this thread is done with the E4M3 bytes
        float s_o[2];
        s_o[0] = __ldg(sc + rb_g * kbl + kb);
        s_o[1] = GATEUP ? __ldg(sc + rb_u * kbl + kb) : 0.f;
#pragma unroll
        for (int o = 0; o < S::kA; ++o) {
          uint32_t out[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t w[4] = {raw[o][j].x, raw[o][j].y, raw[o][j].z, raw[o][j].w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              out[j * 8 + 2 * m] = dequant2(w[m] & 0xFFFFu, s_o[o]);
              out[j * 8 + 2 * m + 1] = dequant2(w[m] >> 16, s_o[o]);
            }
          }
          tmem_st32(lane_base + acol0 + astage * S::kAStageCols + o * kACols + hk * 32, out);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&a_full[astage]);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        if (++astage == ASTAGES) { astage = 0; aphase ^= 1u; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
}

template <bool GATEUP, int NT, int STAGES, int ASTAGES>
cudaError_t launch_variant(const CUtensorMap& w, const CUtensorMap& b0, const CUtensorMap& b1,
                           const TcParams& p, const float* scales, cudaStream_t st) {
  using S = SmemQ<GATEUP, NT, STAGES, ASTAGES>;
  static_assert(S::kTotal <= 227 * 1024, "shared memory");
  auto kern = k_tc_ffn_fp8_wide<GATEUP, NT, STAGES, ASTAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S::kTotal);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), kThreadsQ, S::kTotal, st>>>(w, b0, b1, p, scales);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_fp8_wide(const FfnArgs& a, const int32_t* prefix, bool gateup,
                               cudaStream_t st) {
  TcParams p{};
  p.T = a.T; p.k = a.k; p.E = a.E; p.n_shared = a.n_shared;
  p.f = a.f; p.d = a.d;
  p.K = gateup ? a.d : a.f;
  p.mtiles = (gateup ? a.f : a.d) / kBM;
  p.rows_per_expert = gateup ? 2 * a.f : a.d;
  p.offsets = a.offsets;
  p.prefix = prefix;
  p.h = a.h;
  p.y_perm = a.y_perm;
  p.status = a.status;
  const uint64_t E1 = (uint64_t)a.E + a.n_shared;
  const uint64_t routed = (uint64_t)a.T * a.k;
  const uint64_t slots = routed + (uint64_t)a.n_shared * a.T;
  CUtensorMap w, b0, b1;
  cudaError_t e;
  if (gateup) {
    e = encode_u8_2d(&w, a.w13, E1 * 2 * a.f, a.d, kBM);
    if (e == cudaSuccess) e = encode_bf16_2d(&b0, a.x_perm, routed ? routed : 1, a.d, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&b1, a.x, a.T, a.d, kBoxRows);
  } else {
    e = encode_u8_2d(&w, a.w2, E1 * a.d, a.f, kBM);
    if (e == cudaSuccess) e = encode_bf16_2d(&b0, a.h, slots, a.f, kBoxRows);
    b1 = b0;
  }
  if (e != cudaSuccess) return e;
  const float* sc = gateup ? a.s13 : a.s2;
  if (gateup) return launch_variant<true, 64, 4, 2>(w, b0, b1, p, sc, st);
  return launch_variant<false, 128, 4, 4>(w, b0, b1, p, sc, st);
}

}  // namespace moe
