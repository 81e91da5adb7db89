// Expert FFN, tensor-core path for FP8 E4M3 expert weights with one fp32 scale per 128x128
// block (W8A16: weights dequantised on chip, activations arrive as bf16).
//
// The pages: FP8/FP4 expert weights cut the bytes streamed from HBM, at the price of "scale
// reading, unpacking and tile alignment" work on chip ("DeepSeek-V4-Pro on NVIDIA H200",
// 0.1.3; "CANN DeepSeek-V4推理优化", 量化策略). Here that work is a warp-specialised stage of
// the grouped GEMM, arranged so the per-weight work is as small as possible.
//
// A tile covers 128 weight rows (one row block) and K in 128-wide stages (one column block), so
// one stage of one weight matrix has a single scale s, and
//     sum_k (q[m,k] * s) * x[n,k]  ==  sum_k q[m,k] * (s * x[n,k]).
// The weights therefore go to the tensor cores as their exact code values, and the scale is
// applied to the (few) token rows instead:
//
//   TMA       E4M3 weight tiles (128 rows x 128 K) and bf16 token tiles -> smem ring
//   convert   2 groups of 4 warps, alternating stages: codes -> f16 (exact; one cvt per two
//             codes) written straight into TMEM
//             with tcgen05.st, one weight row per TMEM lane; token rows -> f16(s * x) written
//             into a smem tile per weight matrix (gate and up have their own scale)
//   MMA       one issuing thread per weight tile (warps 1 and 14):
//             tcgen05.mma.kind::f16 (f16 x f16 -> fp32) with A (codes) read from TMEM and B
//             (scaled tokens) from smem
//   epilogue  as in the bf16 kernel: TMEM accumulators -> SiLU(gate) * up -> bf16 h, or fp32
//
// Numerics: codes are exact in f16; s * x is rounded once to f16 (11-bit significand, better
// than bf16) and saturates at +-65504, so the product of a block scale and an activation must
// stay below that (block scales are amax/448, far below 1 for expert weights).
//
// This variant serves decode-sized tiles (32 or 64 tokens); prefill tiles go to
// ffn_tc_fp8_wide.cu, where dequantising the weights costs less than scaling 128-256 token rows.
#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kQK = 128;                          // K per stage = one scale block
constexpr uint32_t kQTileBytes = kBM * kQK;       // 16 KB of E4M3 codes
constexpr int kConvGroups = 2;                    // groups take alternate stages
constexpr int kConvWarps = 4 * kConvGroups;       // a group = one warp per TMEM lane quadrant
constexpr int kConvThreads = 32 * kConvWarps;
// warps: 0 producer, 1 MMA issuer of weight tile 0, 2..5 epilogue, 6..13 converters, 14 MMA
// issuer of weight tile 1 (two issuing threads issue MMAs faster than one)
constexpr int kIssuer2 = 6 + kConvWarps;
constexpr int kThreadsQ = 32 * (kIssuer2 + 1);
constexpr uint32_t kACols = kQK / 2;              // TMEM columns of one 128 x 128 f16 tile

// KA weight tiles of 128 rows share each token tile: gate and up rows of the same features in
// the gate/up pass; one, or two consecutive, 128-row tiles of W_d in the down pass.
template <bool GATEUP, int NT, int STAGES, int CSTAGES, int KA>
struct SmemQ {
  static constexpr int kA = KA;
  static constexpr uint32_t kBHalf = (uint32_t)NT * kBK * 2;   // NT rows x 64 K of 16-bit
  static constexpr uint32_t kStageBytes = kA * kQTileBytes + 2 * kBHalf;   // TMA ring
  static constexpr uint32_t kCSlotBytes = kA * 2 * kBHalf;                 // scaled token tiles
  static constexpr uint32_t kTilesBytes = STAGES * kStageBytes + CSTAGES * kCSlotBytes;
  static constexpr uint32_t kBarBytes = 8 * (2 * STAGES + 2 * CSTAGES + 4) + 16;
  static constexpr uint32_t kTotal = kTilesBytes + kBarBytes + kTileListBytes + 1024;
  static constexpr uint32_t kAccCols = KA * NT;
  static constexpr uint32_t kAStageCols = kA * kACols;
  static constexpr uint32_t kUsedCols = 2 * kAccCols + CSTAGES * kAStageCols;
  static constexpr uint32_t kTmemCols =
      kUsedCols <= 32 ? 32 : kUsedCols <= 64 ? 64 : kUsedCols <= 128 ? 128
      : kUsedCols <= 256 ? 256 : 512;
};

// Instruction descriptor of kind::f16 with f16 A and B, fp32 accumulator, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Four E4M3 codes (lowest byte first) as two exact f16 pairs: codes 0,1 -> lo, codes 2,3 -> hi.
// The 16-bit halves of the word feed the conversions directly (no masking or shifting).
__device__ __forceinline__ void codes4_to_f16x2(uint32_t four, uint32_t& lo, uint32_t& hi) {
  asm("{\n"
      "  .reg .b16 c01, c23;\n"
      "  mov.b32 {c01, c23}, %2;\n"
      "  cvt.rn.f16x2.e4m3x2 %0, c01;\n"
      "  cvt.rn.f16x2.e4m3x2 %1, c23;\n"
      "}"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
}

// f16 pair (lo, hi) = (round(lo), round(hi)), saturating to the largest finite f16.
__device__ __forceinline__ uint32_t f32x2_to_f16x2_sat(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ void sts_u4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

template <bool GATEUP, int NT, int STAGES, int CSTAGES, int KA>
__global__ void __launch_bounds__(kThreadsQ, 1)
    k_tc_ffn_fp8(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b0,
                 const __grid_constant__ CUtensorMap tm_b1, TcParams p,
                 const float* __restrict__ scales) {
  using S = SmemQ<GATEUP, NT, STAGES, CSTAGES, KA>;
  static_assert(S::kUsedCols <= 512, "TMEM columns");
  static_assert(!GATEUP || KA == 2, "gate/up tiles pair the gate and up rows");
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 256, "MMA N");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* cslots = smem + STAGES * S::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kTilesBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* c_full = empty + STAGES;
  uint64_t* c_empty = c_full + CSTAGES;
  uint64_t* acc_full = c_empty + CSTAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* list_s = reinterpret_cast<int32_t*>(smem + S::kTilesBytes + S::kBarBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E1 = p.E + p.n_shared;
  const int kblocks = p.K / kQK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);               // the stage's converter group (4 warps) has read it
    }
    for (int s = 0; s < CSTAGES; ++s) {
      mbar_init(&c_full[s], 4);              // converted operands written
      mbar_init(&c_empty[s], KA);            // MMA commits (one per issuer): operands consumed
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], KA);           // one commit per issuer
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
  // One stage of a tile: its weight boxes (KA tiles of 128 rows x 128 K), then its token rows
  // (nbox boxes of 16 rows, two 64-wide K halves), all completing on the stage's full barrier.
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_b = policy_evict_last();
  auto stage_bytes = [&](const Tile& t) {
    return S::kA * kQTileBytes + (uint32_t)((t.ntok + kBoxRows - 1) / kBoxRows) * 2 * kBBoxBytes;
  };
  auto load_weights = [&](const Tile& t, int kb, uint32_t stage) {
    uint8_t* st = smem + stage * S::kStageBytes;
    const int wrow = t.e * p.rows_per_expert + t.mt * kBM * (GATEUP ? 1 : KA);
    tma_load_2d(st, &tm_w, &full[stage], kb * kQK, wrow, pol_w);
    if (KA == 2)  // up rows of the same features, or the next 128 rows of W_d
      tma_load_2d(st + kQTileBytes, &tm_w, &full[stage], kb * kQK, wrow + (GATEUP ? p.f : kBM),
                  pol_w);
  };
  auto load_tokens = [&](const Tile& t, int kb, uint32_t stage) {
    uint8_t* bt = smem + stage * S::kStageBytes + S::kA * kQTileBytes;
    const CUtensorMap* bmap = (GATEUP && t.shared) ? &tm_b1 : &tm_b0;
    const int nbox = (t.ntok + kBoxRows - 1) / kBoxRows;
    for (int i = 0; i < nbox; ++i)
      for (int hk = 0; hk < 2; ++hk)
        tma_load_2d(bt + hk * S::kBHalf + i * kBBoxBytes, bmap, &full[stage],
                    kb * kQK + hk * kBK, t.brow0 + i * kBoxRows, pol_b);
  };
  prefetch_l2_span(p.prefix, (size_t)(E1 + 1) * 4);
  prefetch_l2_span(p.offsets, (size_t)(E1 + 1) * 4);
  // The gate/up pass's tile list is written by the previous kernel. The down pass's was written
  // two kernels back and its weights are constant: the list is read and the weights of the
  // first tile's first stages are requested before the wait, which only the token rows (h, from
  // the gate/up pass) need.
  int pre = 0;  // stages whose weights went out before the wait
  if constexpr (!GATEUP) {
    stage_tile_list_early(p, list_s);
    if (threadIdx.x == 0 && (int)blockIdx.x < p.prefix[E1]) {
      Tile t;
      decode_tile<GATEUP, NT>(p, blockIdx.x, t);
      pre = min(STAGES, kblocks);
      for (int kb = 0; kb < pre; ++kb) {
        mbar_arrive_expect_tx(&full[kb], stage_bytes(t));
        load_weights(t, kb, (uint32_t)kb);
      }
    }
  }
  pdl_wait_then_release();
  int total = -1;
  if constexpr (GATEUP) {
    total = enter_one_tile(p);  // small batches: this CTA's tile from the front's descriptor
    if (total < 0) stage_tile_list(p, list_s);
  }
  if (total < 0) total = p.prefix[E1];
  const uint32_t acol0 = 2 * S::kAccCols;  // first TMEM column of the converted-weights ring

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      if (pre > 0) {  // the token rows of the stages requested before the wait
        Tile t;
        decode_tile<GATEUP, NT>(p, blockIdx.x, t);
        for (int kb = 0; kb < pre; ++kb) load_tokens(t, kb, (uint32_t)kb);
        stage = (uint32_t)(pre % STAGES);
        phase = pre == STAGES ? 1u : 0u;
      }
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        Tile t;
        decode_tile<GATEUP, NT>(p, tile, t);
        const uint32_t bytes = stage_bytes(t);
        for (int kb = tile == (int)blockIdx.x ? pre : 0; kb < kblocks; ++kb) {
          if (!wait_bar(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], bytes);
          load_weights(t, kb, stage);
          load_tokens(t, kb, stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t issued_phase = (s < (int)stage) ? phase : (phase ^ 1u);
        drain_bar(&full[s], issued_phase, p.status);
      }
    }
  } else if (warp == 1 || warp == kIssuer2) {
    // ---------------- MMA issuers: warp 1 weight tile 0, warp 14 weight tile 1 ----------------
    const int o = warp == 1 ? 0 : 1;
    if (lane == 0 && o < KA) {
      uint32_t cs = 0, cphase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        Tile t;
        decode_tile<GATEUP, NT>(p, tile, t);
        const int npad = (t.ntok + 15) & ~15;
        const uint32_t idesc = idesc_f16(kBM, npad);
        if (!wait_bar(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc * S::kAccCols + o * NT;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(&c_full[cs], cphase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = tmem_base + acol0 + cs * S::kAStageCols + o * kACols;
          const uint32_t bp = smem_u32(cslots + cs * S::kCSlotBytes) + o * 2 * S::kBHalf;
#pragma unroll
          for (int kk = 0; kk < kQK / 16; ++kk) {
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            const uint32_t boff = (kk >> 2) * S::kBHalf;
            mma_ts(d0, a0 + kk * 8, sw128_desc(bp + boff) + 2 * (kk & 3), idesc, accum);
          }
          mma_commit(&c_empty[cs]);
          if (++cs == CSTAGES) { cs = 0; cphase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else if (warp < 6) {
    // ---------------- epilogue (warps 2..5) ----------------
    run_epilogue<GATEUP, NT, S::kAccCols, KA>(p, total, tmem_base, acc_full, acc_empty,
                                              abort_flag);
  } else if (warp < kIssuer2) {
    // ---------------- converters (warps 6..13) ----------------
    // Group g (4 warps, one per TMEM lane quadrant) converts every stage i with i % 2 == g, the
    // whole 128-wide K of its 32 rows, so two stages are converted at once.
    const int grp = (warp - 6) >> 2;
    const int gt = threadIdx.x - 192 - grp * 128;  // 0..127 within the group
    const int q = warp & 3;                   // TMEM lane quadrant
    const int row = q * 32 + lane;            // weight row within the tile = TMEM lane
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    const int kbl = p.K / 128;                // scale blocks along K
    uint32_t it = 0;                          // global stage counter
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      Tile t;
      decode_tile<GATEUP, NT>(p, tile, t);
      const float* sc = scales + (size_t)t.e * (p.rows_per_expert / 128) * kbl;
      const int rb0 = GATEUP ? t.mt : t.mt * KA;             // scale row block of tile 0
      const float* sc_g = sc + rb0 * kbl;                    // gate (or down) row block
      const float* sc_u = sc + (GATEUP ? p.f / 128 + t.mt : rb0 + 1) * kbl;  // up / next rows
      for (int kb = 0; kb < kblocks; ++kb, ++it) {
        if ((int)(it % kConvGroups) != grp) continue;
        const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
        const uint32_t cs = it % CSTAGES, cphase = (it / CSTAGES) & 1u;
        const float s_g = __ldg(sc_g + kb);
        const float s_u = KA == 2 ? __ldg(sc_u + kb) : 0.f;
        if (!wait_bar(&full[stage], phase, abort_flag, p.status) ||
            !wait_bar(&c_empty[cs], cphase ^ 1u, abort_flag, p.status)) { ok = false; break; }
        const uint32_t st = smem_u32(smem + stage * S::kStageBytes);
        const uint32_t bsrc = st + S::kA * kQTileBytes;
        const uint32_t bdst = smem_u32(cslots + cs * S::kCSlotBytes);
        // weight codes of this thread's row -> exact f16 in TMEM (no scale needed)
#pragma unroll
        for (int o = 0; o < S::kA; ++o)
#pragma unroll
          for (int hk = 0; hk < 2; ++hk) {
            uint4 raw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t chunk = (uint32_t)(4 * hk + j) ^ (uint32_t)(row & 7);  // 128B swizzle
              raw[j] = lds_u4(st + o * kQTileBytes + row * 128 + (chunk << 4));
            }
            uint32_t out[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                codes4_to_f16x2(w[m], out[j * 8 + 2 * m], out[j * 8 + 2 * m + 1]);
              }
            }
            tmem_st32(lane_base + acol0 + cs * S::kAStageCols + o * kACols + hk * 32, out);
          }
        // token rows -> f16(s * x), same 128-byte-swizzled K-major layout as the TMA source.
        // Only the tile's ntok rows: MMA columns are independent, so the padding rows up to the
        // next multiple of 16 only feed output columns the epilogue never reads.
        const int units = S::kA * t.ntok * 16;  // (operand, row, 16-byte chunk)
        for (int u = gt; u < units; u += 128) {
          const int o = u / (t.ntok * 16);
          const int rem = u - o * t.ntok * 16;
          const int n = rem >> 4, c = rem & 15;
          const uint32_t off = (uint32_t)(c >> 3) * S::kBHalf + (uint32_t)n * 128 +
                               ((uint32_t)((c & 7) ^ (n & 7)) << 4);
          const uint4 xv = lds_u4(bsrc + off);
          const float s = o ? s_u : s_g;
          uint4 r;
          r.x = f32x2_to_f16x2_sat(__uint_as_float(xv.x << 16) * s, __uint_as_float(xv.x & 0xFFFF0000u) * s);
          r.y = f32x2_to_f16x2_sat(__uint_as_float(xv.y << 16) * s, __uint_as_float(xv.y & 0xFFFF0000u) * s);
          r.z = f32x2_to_f16x2_sat(__uint_as_float(xv.z << 16) * s, __uint_as_float(xv.z & 0xFFFF0000u) * s);
          r.w = f32x2_to_f16x2_sat(__uint_as_float(xv.w << 16) * s, __uint_as_float(xv.w & 0xFFFF0000u) * s);
          sts_u4(bdst + o * 2 * S::kBHalf + off, r);
        }
        fence_proxy_async_smem();             // scaled token tiles -> visible to the MMA
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[stage]);         // this warp is done reading the TMA stage
          mbar_arrive(&c_full[cs]);
        }
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

template <bool GATEUP, int NT, int STAGES, int CSTAGES, int KA>
cudaError_t launch_variant(const CUtensorMap& w, const CUtensorMap& b0, const CUtensorMap& b1,
                           const TcParams& p, const float* scales, cudaStream_t st) {
  using S = SmemQ<GATEUP, NT, STAGES, CSTAGES, KA>;
  static_assert(S::kTotal <= 227 * 1024, "shared memory");
  auto kern = k_tc_ffn_fp8<GATEUP, NT, STAGES, CSTAGES, KA>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S::kTotal);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return launch_pdl(kern, dim3(num_sms()), dim3(kThreadsQ), S::kTotal, st, w, b0, b1, p, scales);
}

}  // namespace

// Decode tiles: 32 tokens while experts average at most 16 routed tokens, else 64 (so an expert
// near the average still fits one tile and its weights are converted once).
static bool fp8_tile64(long routed, int E) { return routed > 16L * E; }

// Down tiles pair two consecutive 128-row tiles of W_d (32 KB of codes per stage, as in the
// gate/up pass) when d allows it: the per-stage hand-offs then move twice the bytes.
int tc_fp8_decode_down_rows(int d) { return d % 256 == 0 ? 2 * kBM : kBM; }

int tc_fp8_tile_tokens(bool gateup, bool decode, long routed, int E) {
  (void)gateup;
  if (!decode) return tc_fp8_wide_tile_tokens();
  return fp8_tile64(routed, E) ? 64 : 32;
}

cudaError_t launch_tc_fp8(const FfnArgs& a, const int32_t* prefix, bool gateup, bool decode,
                          cudaStream_t st) {
  if (!decode) return launch_tc_fp8_wide(a, prefix, gateup, st);
  TcParams p{};
  p.T = a.T; p.k = a.k; p.E = a.E; p.n_shared = a.n_shared;
  p.f = a.f; p.d = a.d;
  p.K = gateup ? a.d : a.f;
  const bool pair_dn = !gateup && tc_fp8_decode_down_rows(a.d) == 2 * kBM;
  p.mtiles = gateup ? a.f / kBM : a.d / tc_fp8_decode_down_rows(a.d);
  p.rows_per_expert = gateup ? 2 * a.f : a.d;
  p.offsets = a.offsets;
  p.prefix = prefix;
  p.h = a.h;
  p.y_perm = a.y_perm;
  p.status = a.status;
  if (gateup) p.tile1 = a.tile1;
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
  const float* sc = static_cast<const float*>(gateup ? a.s13 : a.s2);
  if (fp8_tile64((long)routed, a.E)) {
    if (gateup) return launch_variant<true, 64, 3, 2, 2>(w, b0, b1, p, sc, st);
    if (pair_dn) return launch_variant<false, 64, 3, 2, 2>(w, b0, b1, p, sc, st);
    return launch_variant<false, 64, 5, 3, 1>(w, b0, b1, p, sc, st);
  }
  if (gateup) return launch_variant<true, 32, 4, 3, 2>(w, b0, b1, p, sc, st);
  if (pair_dn) return launch_variant<false, 32, 4, 3, 2>(w, b0, b1, p, sc, st);
  return launch_variant<false, 32, 6, 4, 1>(w, b0, b1, p, sc, st);
}

}  // namespace moe
