// Expert FFN, tensor-core path: a persistent grouped GEMM on tcgen05 with TMEM accumulators,
// fed by TMA, for bf16 expert weights.
//
// The pages: once an expert receives enough tokens its weights are reused across rows and the
// work becomes a real matrix multiply ("第 6 章 超節點", 6.1.3 and 6.3.2: batch reuse moves the
// limit from weight reads to math; "DeepSeek V3/R1 Inference Efficiency (1)": DeepGEMM's
// grouped expert GEMMs). Y = [SiLU(X W_g) (.) (X W_u)] W_d ("第 6 章 超節點", 6.2.2) is computed in
// two passes, gate/up (with SiLU x up fused into the epilogue) and down.
//
// Shape of one tile (swap-AB): M = 128 rows of one expert's weight matrix (output features),
// N = the expert's tokens in this tile (16..NT, a multiple of 16), K streamed in 64-wide
// stages. Weights are the M side so that a decode expert with a handful of tokens still reads
// each weight byte exactly once per call, at full tile width. Gate/up tiles issue two MMAs per
// K step (gate rows and up rows of the same output features) into two accumulators.
//
// Warp roles (7 warps, one CTA per SM, persistent over a device-built tile list):
//   warp 0     TMA producer (one thread): weight tile + token tile per stage
//   warp 1     TMEM owner and MMA issuer of weight tile 0 (one thread)
//   warps 2-5  epilogue: TMEM -> registers -> SiLU(gate)*up -> bf16 h, or fp32 expert output
//   warp 6     MMA issuer of weight tile 1 (one thread), when the tile pairs two weight tiles
// Accumulators are double-buffered in TMEM so the epilogue of tile i overlaps the mainloop of
// tile i+1. Every wait is bounded: a wait that gives up records MOE_ERR_DEVICE_TIMEOUT and the
// CTA winds down, frees its TMEM and exits.
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

// KA weight tiles of 128 rows share each token tile: gate + up rows of the same features in the
// gate/up pass, one or two consecutive 128-row tiles of W_d in the down pass. ACCB accumulator
// buffers: 2 lets the epilogue of one tile overlap the next tile's mainloop; wide tiles
// (KA * NT = 512 columns) fill TMEM with a single buffer.
template <int NT, int STAGES, int KA, int ACCB, bool PAIR = false>
struct Smem {
  // weight tiles and token rows of one stage (CTA pairs: half of the token tile in each CTA)
  static constexpr uint32_t kBBytes = (uint32_t)(PAIR ? NT / 2 : NT) * kBK * 2;
  static constexpr uint32_t kStageBytes = KA * kATileBytes + kBBytes;
  static constexpr uint32_t kTilesBytes = STAGES * kStageBytes;
  static constexpr uint32_t kBarBytes = 8 * (2 * STAGES + 4) + 16;
  static constexpr uint32_t kTotal = kTilesBytes + kBarBytes + 1024;  // + alignment slack
  static constexpr uint32_t kAccCols = KA * NT;                       // per accumulator buffer
  static constexpr uint32_t kTmemCols = ACCB * kAccCols;
};

// warps: 0 producer, 1 MMA issuer of weight tile 0, 2..5 epilogue, 6 MMA issuer of weight tile 1
// (two issuing threads issue MMAs faster than one)
constexpr int kThreadsB = 32 * 7;

template <bool GATEUP, int NT, int STAGES, int KA, int ACCB, bool PAIR>
__global__ void __launch_bounds__(kThreadsB, 1)
    k_tc_ffn(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b0,
             const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b0w,
             const __grid_constant__ CUtensorMap tm_b1w, const TcParams p) {
  using S = Smem<NT, STAGES, KA, ACCB, PAIR>;
  static_assert(S::kTmemCols <= 512 && (S::kTmemCols & (S::kTmemCols - 1)) == 0, "TMEM cols");
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 256, "MMA N");
  static_assert(!GATEUP || KA == 2, "gate/up tiles pair the gate and up rows");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kTilesBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E1 = p.E + p.n_shared;
  const int kblocks = p.K / kBK;
  // CTA pairs (cta_group::2): both CTAs walk the same list of (expert, m-tile pair, token tile)
  // entries; this CTA takes m-tile 2 * mt + rank and loads its own weight rows and half of the
  // tile's (padded) token rows, the even CTA issues MMAs of M = 256 that read both CTAs'
  // operands, and each CTA's tensor memory receives its own 128 rows. Every load of either CTA
  // completes on the even CTA's stage barrier; the MMA commits free the stage in both.
  int nact = (int)gridDim.x;
  if (p.active) {
    pdl_wait_then_release();  // the count is written by the plan kernel
    nact = __ldg(p.active);   // even with pairs, so both CTAs of a cluster leave together
    if ((int)blockIdx.x >= nact) return;
  }
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  const bool issuer_cta = rank == 0;  // the CTA whose threads issue the MMAs
  const int tile0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int tstep = PAIR ? nact >> 1 : nact;
  const auto decode = [&](int tile, Tile& t) {
    decode_tile<GATEUP, NT>(p, tile, t);
    if (PAIR) t.mt = 2 * t.mt + rank;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);       // the (even CTA's) producer, + TMA bytes
      mbar_init(&empty[s], KA);     // MMA commits: one per issuer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], KA);  // one commit per issuer
      mbar_init(&acc_empty[b], PAIR ? 8 : 4);  // epilogue warps (of both CTAs of a pair)
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_b0);
    prefetch_tmap(&tm_b1);
    prefetch_tmap(&tm_b0w);
    prefetch_tmap(&tm_b1w);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_holder, S::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, S::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // both CTAs' barriers are initialised before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // the tile list (prefix) is written by the previous kernel
  pdl_wait_then_release();
  const int total = __ldg(p.prefix + E1);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // weights: streamed once per call (evict first), unless the expert has several token
      // tiles, whose tiles run at about the same time on other SMs and read them again
      const uint64_t pol_once = policy_evict_first(), pol_again = policy_evict_normal();
      const uint64_t pol_b = policy_evict_last();   // token rows: reused by every weight tile
      const uint32_t full0 = PAIR ? mapa_shared(smem_u32(&full[0]), 0) : 0;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < total; tile += tstep) {
        Tile t;
        decode(tile, t);
        const bool wide = t.ntok == NT;   // full token tile: one TMA box (NT, or NT/2 rows)
        // this CTA's token rows: all of them, or (pairs) half of the padded count
        const int half = PAIR ? ((t.ntok + 15) & ~15) / 2 : t.ntok;
        const int row0 = t.brow0 + rank * half;
        const int nbox = (half + kBoxRows - 1) / kBoxRows;
        const uint32_t bytes =
            KA * kATileBytes + (wide ? S::kBBytes : (uint32_t)nbox * kBBoxBytes);
        // gate/up: 128 features, rows [f0, f0+128) (gate) and [f + f0, ...) (up);
        // down: KA consecutive 128-row tiles of W_d
        const int wrow = t.e * p.rows_per_expert + t.mt * (GATEUP ? kBM : kBM * KA);
        const int wrow1 = GATEUP ? wrow + p.f : wrow + kBM;   // second weight tile
        const bool sh = GATEUP && t.shared;
        const CUtensorMap* bmap = sh ? &tm_b1 : &tm_b0;
        const CUtensorMap* bmapw = sh ? &tm_b1w : &tm_b0w;
        const uint64_t pol_w = t.multi ? pol_again : pol_once;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          uint8_t* st = smem + stage * S::kStageBytes;
          uint8_t* bt = st + KA * kATileBytes;
          if (PAIR) {
            // both CTAs load the same number of bytes, so the even CTA expects twice its own
            if (issuer_cta) mbar_arrive_expect_tx(&full[stage], 2 * bytes);
            const uint32_t bar = full0 + 8u * stage;
            tma_load_2d_pair(st, &tm_w, bar, kb * kBK, wrow, pol_w);
            if (KA == 2) tma_load_2d_pair(st + kATileBytes, &tm_w, bar, kb * kBK, wrow1, pol_w);
            if (wide) {
              tma_load_2d_pair(bt, bmapw, bar, kb * kBK, row0, pol_b);
            } else {
              for (int i = 0; i < nbox; ++i)
                tma_load_2d_pair(bt + i * kBBoxBytes, bmap, bar, kb * kBK, row0 + i * kBoxRows,
                                 pol_b);
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            continue;
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_2d(st, &tm_w, &full[stage], kb * kBK, wrow, pol_w);
          if (KA == 2) tma_load_2d(st + kATileBytes, &tm_w, &full[stage], kb * kBK, wrow1, pol_w);
          if (wide) {
            tma_load_2d(bt, bmapw, &full[stage], kb * kBK, t.brow0, pol_b);
          } else {
            for (int i = 0; i < nbox; ++i)
              tma_load_2d(bt + i * kBBoxBytes, bmap, &full[stage], kb * kBK,
                          t.brow0 + i * kBoxRows, pol_b);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // Every load issued has landed before the CTA may exit (in pairs the even CTA's barrier
      // counts both CTAs' bytes), and in pairs the MMA commits for every issued stage have
      // arrived here.
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t issued_phase = (s < (int)stage) ? phase : (phase ^ 1u);
        if (!PAIR || issuer_cta) drain_bar(&full[s], issued_phase, p.status);
        if (PAIR) drain_bar(&empty[s], issued_phase, p.status);
      }
    }
  } else if (warp == 1 || warp == 6) {
    // ---------------- MMA issuers: warp 1 weight tile 0, warp 6 weight tile 1 ----------------
    const int o = warp == 1 ? 0 : 1;
    if (lane == 0 && o < KA && issuer_cta) {
      uint32_t stage = 0, phase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < total; tile += tstep) {
        Tile t;
        decode(tile, t);
        const int npad = (t.ntok + 15) & ~15;
        const uint32_t idesc = idesc_bf16(PAIR ? 2 * kBM : kBM, npad);
        if (!wait_bar(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc * S::kAccCols + o * NT;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * S::kStageBytes);
          const uint64_t da = sw128_desc(st + o * kATileBytes);
          const uint64_t db = sw128_desc(st + KA * kATileBytes);
          if (PAIR) {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_ss_pair(d0, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
            mma_commit_pair(&empty[stage]);  // frees the stage in both CTAs of the pair
          } else {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16_ss(d0, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
            mma_commit(&empty[stage]);  // frees the stage once these MMAs have read it
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (PAIR)
          mma_commit_pair(&acc_full[acc]);  // accumulators ready for both CTAs' epilogues
        else
          mma_commit(&acc_full[acc]);       // accumulator ready for the epilogue
        if (++acc == ACCB) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else if (warp < 6) {
    // ---------------- epilogue (warps 2..5) ----------------
    run_epilogue<GATEUP, NT, S::kAccCols, KA, ACCB>(p, total, tmem_base, acc_full, acc_empty,
                                                    abort_flag, tile0, tstep, PAIR ? rank : -1, 2,
                                                    PAIR && !issuer_cta);
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, S::kTmemCols);
    else
      tmem_dealloc(tmem_base, S::kTmemCols);
  }
}

template <bool GATEUP, int NT, int STAGES, int KA, int ACCB, bool PAIR = false>
cudaError_t launch_variant(const CUtensorMap& w, const CUtensorMap& b0, const CUtensorMap& b1,
                           const CUtensorMap& b0w, const CUtensorMap& b1w, const TcParams& p,
                           cudaStream_t st) {
  using S = Smem<NT, STAGES, KA, ACCB, PAIR>;
  static_assert(S::kTotal <= 227 * 1024, "shared memory");
  auto kern = k_tc_ffn<GATEUP, NT, STAGES, KA, ACCB, PAIR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S::kTotal);
  if (e != cudaSuccess) return e;
  count_launches(1);
  if (PAIR)
    return launch_pdl_cluster(kern, dim3((unsigned)(num_sms() & ~1)), dim3(kThreadsB), S::kTotal,
                              st, 2u, w, b0, b1, b0w, b1w, p);
  return launch_pdl(kern, dim3(num_sms()), dim3(kThreadsB), S::kTotal, st, w, b0, b1, b0w, b1w, p);
}

// Weight rows per down-pass tile: two 128-row tiles share the token tile in the prefill
// variant when d allows it.
bool down_pairs(int d, bool decode) { return !decode && d % 256 == 0; }

}  // namespace

int tc_tile_tokens(bool gateup, bool decode) {
  (void)gateup;
  return decode ? 64 : 256;
}

// The cold list of a split prefill (experts with few tokens, HBM-bound): 32-token tiles, whose
// smaller token slots leave room for deeper weight rings.
int tc_cold_tile_tokens() { return 32; }

int tc_tile_rows(bool gateup, bool decode, int d) {
  return (!gateup && down_pairs(d, decode)) ? 2 * kBM : kBM;
}

// Prefill tiles with two weight tiles per token tile run on CTA pairs (cta_group::2: consecutive
// m-tiles, half of the token tile in each CTA) when an expert has an even number of such tiles.
static bool tc_clustered(bool gateup, bool decode, int d, int f) {
  if (decode || (!gateup && !down_pairs(d, decode))) return false;
  return ((gateup ? f : d) / tc_tile_rows(gateup, decode, d)) % 2 == 0;
}

int tc_plan_mtiles(bool gateup, bool decode, int d, int f) {
  const int mtiles = (gateup ? f : d) / tc_tile_rows(gateup, decode, d);
  return tc_clustered(gateup, decode, d, f) ? mtiles / 2 : mtiles;
}

cudaError_t launch_tc(const FfnArgs& a, const int32_t* prefix, bool gateup, bool decode,
                      cudaStream_t st, const int32_t* active, bool cold) {
  TcParams p{};
  p.active = active;
  p.T = a.T; p.k = a.k; p.E = a.E; p.n_shared = a.n_shared;
  p.f = a.f; p.d = a.d;
  p.K = gateup ? a.d : a.f;
  p.mtiles = (gateup ? a.f : a.d) / tc_tile_rows(gateup, decode, a.d);
  p.rows_per_expert = gateup ? 2 * a.f : a.d;
  p.offsets = a.offsets;
  p.prefix = prefix;
  p.h = a.h;
  p.y_perm = a.y_perm;
  p.status = a.status;
  const uint64_t E1 = (uint64_t)a.E + a.n_shared;
  const uint64_t routed = (uint64_t)a.T * a.k;
  const uint64_t slots = routed + (uint64_t)a.n_shared * a.T;
  const bool cl = tc_clustered(gateup, decode, a.d, a.f);
  // full token tiles arrive in one box of the kernel's NT rows, or, with pairs, in one half-tile
  // box in each CTA
  const int tile_nt = cold ? tc_cold_tile_tokens() : tc_tile_tokens(gateup, decode);
  const uint32_t nt = (uint32_t)tile_nt / (cl ? 2u : 1u);
  CUtensorMap w, b0, b1, b0w, b1w;
  cudaError_t e;
  if (gateup) {
    e = encode_bf16_2d(&w, a.w13, E1 * 2 * a.f, a.d, kBM);
    if (e == cudaSuccess) e = encode_bf16_2d(&b0, a.x_perm, routed ? routed : 1, a.d, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&b1, a.x, a.T, a.d, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&b0w, a.x_perm, routed ? routed : 1, a.d, nt);
    if (e == cudaSuccess) e = encode_bf16_2d(&b1w, a.x, a.T, a.d, nt);
  } else {
    e = encode_bf16_2d(&w, a.w2, E1 * a.d, a.f, kBM);
    if (e == cudaSuccess) e = encode_bf16_2d(&b0, a.h, slots, a.f, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&b0w, a.h, slots, a.f, nt);
    b1 = b0;
    b1w = b0w;
  }
  if (e != cudaSuccess) return e;
  if (cold)  // 32-token tiles: 6 stages of 36 KB (gate/up), 10 of 20 KB (down)
    return gateup ? launch_variant<true, 32, 6, 2, 2>(w, b0, b1, b0w, b1w, p, st)
                  : launch_variant<false, 32, 10, 1, 2>(w, b0, b1, b0w, b1w, p, st);
  if (gateup)
    return decode ? launch_variant<true, 64, 5, 2, 2>(w, b0, b1, b0w, b1w, p, st)
                  : cl ? launch_variant<true, 256, 4, 2, 1, true>(w, b0, b1, b0w, b1w, p, st)
                       : launch_variant<true, 256, 3, 2, 1>(w, b0, b1, b0w, b1w, p, st);
  if (decode) return launch_variant<false, 64, 8, 1, 2>(w, b0, b1, b0w, b1w, p, st);
  if (cl) return launch_variant<false, 256, 4, 2, 1, true>(w, b0, b1, b0w, b1w, p, st);
  return down_pairs(a.d, decode) ? launch_variant<false, 256, 3, 2, 1>(w, b0, b1, b0w, b1w, p, st)
                                 : launch_variant<false, 256, 4, 1, 2>(w, b0, b1, b0w, b1w, p, st);
}

}  // namespace moe
