// Expert FFN, tensor-core path for MXFP4 expert weights: E2M1 codes (two per byte) with one E8M0
// scale per 32 consecutive elements of a weight row.
//
// The pages: V4-Pro's routed experts are stored in FP4, which halves the bytes streamed from HBM
// again, at the price of unpacking and scale handling on chip ("DeepSeek-V4-Pro on NVIDIA H200",
// 0.1.3); the format is MXFP4 ("CANN DeepSeek-V4推理优化", 量化策略). On sm_103a that price is
// paid by the tensor core itself: tcgen05.mma.kind::mxf8f6f4 with block scaling multiplies rows
// of E2M1 codes by rows of E4M3 codes and applies one E8M0 scale per 32-wide K block of every row
// of either operand, accumulating in fp32. No weight is converted on chip:
//
//   TMA       E2M1 weight tiles (128 rows x 128 K; the 16U4_ALIGN16B tensor map spreads every 8
//             bytes of code pairs over 16 bytes of shared memory, the form the MMA reads) and the
//             token rows' two E4M3 terms (mx_common.cuh) -> shared-memory ring
//   scales    4 warps: the weight rows' and the token rows' scale words -> TMEM; the MMA reads
//             row m's word from TMEM lane m, column (m / 32) of the word group
//   MMA       per 32-wide K block and weight tile: the hi and the lo term rows of the tokens sit
//             one after the other in one B tile, so one MMA of N = 2 x tokens covers both and the
//             epilogue adds the two halves
//   epilogue  gate/up: SiLU(gate) * up, written straight as the down pass's two E4M3 terms;
//             down: the fp32 expert output
//
// One persistent CTA per SM walks the tile list of its pass (an expert's token tile x KA
// consecutive 128-row weight tiles), as the bf16 and FP8 kernels do.
#include "mx_common.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kMxK = 128;                        // K per stage: four 32-wide scale blocks
constexpr uint32_t kWSmem = kBM * kMxK;          // one weight tile in shared memory (16 KB)
constexpr uint32_t kWTx = kBM * kMxK / 2;        // the bytes TMA reads for it (8 KB)
constexpr uint32_t kTBox = kBoxRows * kMxK;      // one 16-row box of E4M3 token codes
// warps: 0 producer, 1 MMA issuer of weight tile 0, 2..5 epilogue, 6..9 scale writers, 10 MMA
// issuer of weight tile 1 (two issuing threads together issue block-scaled MMAs ~1.5x as fast as
// one: measured 40 vs 59 cycles an MMA at N = 32)
constexpr int kThreadsMx = 32 * 11;
constexpr int kSfAhead = 4;                      // K slices the scale words are loaded ahead

struct MxParams {
  const uint8_t* w_scales;    // [rows of the weight map, K/32] E8M0
  const uint8_t* t_scale_hi;  // [slots, K/32] E8M0 of the token rows' hi terms
  const uint8_t* t_scale_lo;  // ... and lo terms
  mx::Planes h;               // gate/up output: h as the down pass's terms, [slots, f]
};

// A ring stage holds SUB consecutive 128-wide K slices (each: KA weight tiles and the token
// tile): the per-stage hand-offs (barrier waits, commit) are paid once per SUB slices.
template <bool GATEUP, int NT, int STAGES, int KA, int ACCB, int SUB>
struct SmemMx {
  static constexpr uint32_t kBTile = (uint32_t)NT * kMxK;  // one term's token tile
  static constexpr uint32_t kSliceBytes = KA * kWSmem + 2 * kBTile;
  static constexpr uint32_t kStageBytes = SUB * kSliceBytes;
  static constexpr uint32_t kTilesBytes = STAGES * kStageBytes;
  static constexpr uint32_t kBarBytes = 8 * (2 * STAGES + 2 * ACCB) + 16;
  // the tile list goes to shared memory where it fits beside the ring
  static constexpr bool kStageList = kTilesBytes + kBarBytes + kTileListBytes + 1024 <= 227 * 1024;
  static constexpr uint32_t kTotal =
      kTilesBytes + kBarBytes + (kStageList ? kTileListBytes : 0) + 1024;
  static constexpr uint32_t kAccN = 2 * NT;  // accumulator columns per weight tile: hi, then lo
  static constexpr uint32_t kAccCols = KA * kAccN;
  // scale words of the token B rows (hi rows, then lo rows): one 4-column group per 128 rows
  static constexpr uint32_t kBSfCols = 2 * NT <= 128 ? 4 : 8;
  // per stage: a 4-column group per (slice, weight tile), then the token groups of each slice
  static constexpr uint32_t kSfCols = SUB * (4 * KA + kBSfCols);
  static constexpr uint32_t kUsedCols = ACCB * kAccCols + STAGES * kSfCols;
  static constexpr uint32_t kTmemCols =
      kUsedCols <= 32 ? 32 : kUsedCols <= 64 ? 64 : kUsedCols <= 128 ? 128
      : kUsedCols <= 256 ? 256 : 512;
};

__device__ __forceinline__ uint32_t ldg_u32(const uint8_t* p) {
  return __ldg(reinterpret_cast<const uint32_t*>(p));
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v)
               : "memory");
}

// Gate/up epilogue (warps 2..5): h = SiLU(gate) * up for the tile's tokens, encoded as two E4M3
// terms per element with one scale byte per term and 32 consecutive features -- exactly the 32
// lanes of one warp, so the block maximum is a warp reduction.
template <int NT, int ACCB, uint32_t ACC_COLS, uint32_t ACC_N>
__device__ __forceinline__ void gateup_epilogue(const TcParams& p, const MxParams& q, int total,
                                                uint32_t tmem_base, uint64_t* acc_full,
                                                uint64_t* acc_empty, volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3;
  const int fb = p.f / 32;
  uint32_t acc = 0, acc_phase = 0;
  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    Tile t;
    decode_tile<true, NT>(p, tile, t);
    const int npad = (t.ntok + 15) & ~15;
    if (!wait_bar(&acc_full[acc], acc_phase, abort_flag, p.status)) break;
    tc_fence_after();
    const uint32_t tbase = tmem_base + ((uint32_t)(qd * 32) << 16) + acc * ACC_COLS;
    const int feat = t.mt * kBM + qd * 32 + lane;   // h column of this lane
    const int blk = t.mt * (kBM / 32) + qd;         // its 32-feature scale block
    for (int c0 = 0; c0 < npad; c0 += 16) {
      uint32_t g[16], u[16], g2[16], u2[16];
      tmem_ld16(tbase + c0, g);
      tmem_ld16(tbase + ACC_N + c0, u);
      tmem_ld16(tbase + npad + c0, g2);  // the lo term's products, npad columns further on
      tmem_ld16(tbase + ACC_N + npad + c0, u2);
      tmem_ld_wait2(g, u);
      tmem_ld_wait2(g2, u2);
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const int n = c0 + j;
        if (n >= t.ntok) break;  // the same n in every lane
        float v[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float gv = __uint_as_float(g[j + i]) + __uint_as_float(g2[j + i]);
          const float uv = __uint_as_float(u[j + i]) + __uint_as_float(u2[j + i]);
          v[i] = n + i < t.ntok ? gv / (1.0f + __expf(-gv)) * uv : 0.f;
        }
        uint32_t hi0, lo0, hi1, lo1, a0, b0, a1, b1;
        mx::encode_warp2(v[0], v[1], hi0, lo0, hi1, lo1, a0, b0, a1, b1);
        const long row = t.slot0 + n;
        q.h.hi[row * p.f + feat] = (uint8_t)hi0;
        q.h.lo[row * p.f + feat] = (uint8_t)lo0;
        if (lane == 0) {
          q.h.s_hi[row * fb + blk] = (uint8_t)a0;
          q.h.s_lo[row * fb + blk] = (uint8_t)b0;
        }
        if (n + 1 < t.ntok) {
          q.h.hi[(row + 1) * p.f + feat] = (uint8_t)hi1;
          q.h.lo[(row + 1) * p.f + feat] = (uint8_t)lo1;
          if (lane == 0) {
            q.h.s_hi[(row + 1) * fb + blk] = (uint8_t)a1;
            q.h.s_lo[(row + 1) * fb + blk] = (uint8_t)b1;
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&acc_empty[acc]);
    if (++acc == ACCB) { acc = 0; acc_phase ^= 1u; }
  }
}

// Down epilogue (warps 2..5): the expert output of token n and weight row r is the sum of the
// hi-term column n and the lo-term column npad + n of the accumulator.
template <int NT, int KA, int ACCB, uint32_t ACC_COLS, uint32_t ACC_N>
__device__ __forceinline__ void down_epilogue(const TcParams& p, int total,
                                                     uint32_t tmem_base, uint64_t* acc_full,
                                                     uint64_t* acc_empty,
                                                     volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3;
  const int row = qd * 32 + lane;
  uint32_t acc = 0, acc_phase = 0;
  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    Tile t;
    decode_tile<false, NT>(p, tile, t);
    const int npad = (t.ntok + 15) & ~15;
    if (!wait_bar(&acc_full[acc], acc_phase, abort_flag, p.status)) break;
    tc_fence_after();
    const uint32_t tbase = tmem_base + ((uint32_t)(qd * 32) << 16) + acc * ACC_COLS;
#pragma unroll
    for (int a = 0; a < KA; ++a) {
      const int orow = t.mt * (kBM * KA) + a * kBM + row;
      for (int c0 = 0; c0 < npad; c0 += 16) {
        uint32_t h[16], l[16];
        tmem_ld16(tbase + a * ACC_N + c0, h);
        tmem_ld16(tbase + a * ACC_N + npad + c0, l);
        tmem_ld_wait2(h, l);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = c0 + j;
          if (n < t.ntok)
            p.y_perm[(size_t)(t.slot0 + n) * p.d + orow] =
                __uint_as_float(h[j]) + __uint_as_float(l[j]);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&acc_empty[acc]);
    if (++acc == ACCB) { acc = 0; acc_phase ^= 1u; }
  }
}

template <bool GATEUP, int NT, int STAGES, int KA, int ACCB, int SUB>
__global__ void __launch_bounds__(kThreadsMx, 1)
    k_tc_ffn_mx(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_hi,
                const __grid_constant__ CUtensorMap tm_lo, TcParams p, const MxParams q) {
  using S = SmemMx<GATEUP, NT, STAGES, KA, ACCB, SUB>;
  static_assert(S::kUsedCols <= 512, "TMEM columns");
  static_assert(2 * NT <= 256, "MMA N");
  static_assert(!GATEUP || KA == 2, "gate/up tiles pair the gate and up rows");
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 128, "token tile");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kTilesBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + ACCB;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + ACCB);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* list_s = reinterpret_cast<int32_t*>(smem + S::kTilesBytes + S::kBarBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E1 = p.E + p.n_shared;
  const int kblocks = p.K / (kMxK * SUB);  // stages per tile
  const int ksb = p.K / 32;                // scale bytes per row

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 5);   // the producer's expect-tx arrival and the four scale writers
      mbar_init(&empty[s], KA);  // MMA commits (one per issuer): tiles and scale words consumed
    }
    for (int b = 0; b < ACCB; ++b) {
      mbar_init(&acc_full[b], KA);  // one commit per issuer
      mbar_init(&acc_empty[b], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_hi);
    prefetch_tmap(&tm_lo);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // One stage of a tile: SUB K slices, each its weight boxes (KA tiles of 128 rows x 128 codes)
  // and its token terms (nbox boxes of 16 hi rows, then as many lo rows), all completing on the
  // stage's full barrier.
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_b = policy_evict_last();
  auto stage_bytes = [&](const Tile& t) {
    return SUB * (KA * kWTx + (uint32_t)((t.ntok + kBoxRows - 1) / kBoxRows) * 2 * kTBox);
  };
  auto load_weights = [&](const Tile& t, int kb, uint32_t stage) {
    const int wrow = t.e * p.rows_per_expert + t.mt * kBM * (GATEUP ? 1 : KA);
#pragma unroll
    for (int sb = 0; sb < SUB; ++sb) {
      uint8_t* sl = smem + stage * S::kStageBytes + sb * S::kSliceBytes;
      const int xk = (kb * SUB + sb) * kMxK;
      tma_load_2d(sl, &tm_w, &full[stage], xk, wrow, pol_w);
      if (KA == 2)  // up rows of the same features, or the next 128 rows of W_d
        tma_load_2d(sl + kWSmem, &tm_w, &full[stage], xk, wrow + (GATEUP ? p.f : kBM), pol_w);
    }
  };
  auto load_tokens = [&](const Tile& t, int kb, uint32_t stage) {
    const int nbox = (t.ntok + kBoxRows - 1) / kBoxRows;
#pragma unroll
    for (int sb = 0; sb < SUB; ++sb) {
      uint8_t* bt = smem + stage * S::kStageBytes + sb * S::kSliceBytes + KA * kWSmem;
      const int xk = (kb * SUB + sb) * kMxK;
      for (int i = 0; i < nbox; ++i) {
        tma_load_2d(bt + i * kTBox, &tm_hi, &full[stage], xk, t.slot0 + i * kBoxRows, pol_b);
        // the lo rows right after the tile's nbox boxes of hi rows
        tma_load_2d(bt + (nbox + i) * kTBox, &tm_lo, &full[stage], xk, t.slot0 + i * kBoxRows,
                    pol_b);
      }
    }
  };
  prefetch_l2_span(p.prefix, (size_t)(E1 + 1) * 4);
  prefetch_l2_span(p.offsets, (size_t)(E1 + 1) * 4);
  // As in the E4M3 decode tiles: the down pass reads its tile list (written two kernels back)
  // and requests its first tile's first weight stages before the wait; the token terms of h come
  // from the gate/up pass, after it.
  int pre = 0;  // stages whose weights went out before the wait
  if constexpr (!GATEUP && S::kStageList) {
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
  pdl_wait_then_release();  // tile list, token terms and (down pass) h come from earlier kernels
  int total = -1;
  if constexpr (GATEUP) {
    total = enter_one_tile(p);  // small batches: this CTA's tile from the front's descriptor
    if (total < 0 && S::kStageList) stage_tile_list(p, list_s);
  }
  if (total < 0) total = p.prefix[E1];
  const uint32_t sf0 = ACCB * S::kAccCols;  // first TMEM column of the scale-word ring

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      if (pre > 0) {  // the token terms of the stages requested before the wait
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
  } else if (warp == 1 || warp == 10) {
    // ---------------- MMA issuers: warp 1 weight tile 0, warp 10 weight tile 1 ----------------
    const int o = warp == 1 ? 0 : 1;
    if (lane == 0 && o < KA) {
      uint32_t stage = 0, phase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        Tile t;
        decode_tile<GATEUP, NT>(p, tile, t);
        const int npad = (t.ntok + 15) & ~15;
        if (!wait_bar(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t dp = tmem_base + acc * S::kAccCols + o * S::kAccN;
        uint32_t idesc[kMxK / 32];
#pragma unroll
        for (int kk = 0; kk < kMxK / 32; ++kk)
          idesc[kk] = idesc_mx_e2m1_e4m3(kBM, 2 * npad, kk, kk);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sfc = tmem_base + sf0 + stage * S::kSfCols;
#pragma unroll
          for (int sb = 0; sb < SUB; ++sb) {
            const uint32_t a0 = smem_u32(smem + stage * S::kStageBytes + sb * S::kSliceBytes);
            const uint64_t ad = sw128_desc(a0 + o * kWSmem);
            const uint64_t bh = sw128_desc(a0 + KA * kWSmem);
            const uint32_t sfa = sfc + 4 * (sb * KA + o);
            const uint32_t sfb = sfc + 4 * KA * SUB + sb * S::kBSfCols;
#pragma unroll
            for (int kk = 0; kk < kMxK / 32; ++kk) {
              mma_mx(dp, ad + 2 * kk, bh + 2 * kk, idesc[kk], sfa, sfb, (kb | sb | kk) ? 1u : 0u);
            }
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
        if (++acc == ACCB) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else if (warp < 6) {
    // ---------------- epilogue (warps 2..5) ----------------
    if (GATEUP)
      gateup_epilogue<NT, ACCB, S::kAccCols, S::kAccN>(p, q, total, tmem_base, acc_full,
                                                       acc_empty, abort_flag);
    else
      down_epilogue<NT, KA, ACCB, S::kAccCols, S::kAccN>(p, total, tmem_base, acc_full,
                                                         acc_empty, abort_flag);
  } else if (warp < 10) {
    // ---------------- scale writers (warps 6..9) ----------------
    // Warp of lane quadrant qd writes, per K slice of a stage: weight row 32*qd + lane's word
    // (its four K-block scales of the slice) at column qd of the slice's group for that weight
    // tile, and the B rows' words in every lane quadrant, B row 32*c + lane in column c of the
    // slice's token groups, which is where the MMA reads them. B row r is token r's hi term
    // (r < npad) and token r - npad's lo term after it. Then it arrives on the stage's full
    // barrier. The words are loaded kSfAhead slices ahead of their store (a register ring).
    const int qd = warp & 3;
    const uint32_t lane_base = tmem_base + ((uint32_t)(qd * 32) << 16);
    const int nslices = kblocks * SUB;
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      Tile t;
      decode_tile<GATEUP, NT>(p, tile, t);
      const int wrow = t.e * p.rows_per_expert + t.mt * kBM * (GATEUP ? 1 : KA);
      const uint8_t* wa = q.w_scales + (size_t)(wrow + qd * 32 + lane) * ksb;
      const size_t wstep = (size_t)(GATEUP ? p.f : kBM) * ksb;  // to the second weight tile
      const int npad = (t.ntok + 15) & ~15;
      uint32_t ra[kSfAhead][2], rb[kSfAhead][8];
      const auto load = [&](uint32_t (&a)[2], uint32_t (&b)[8], int ks) {
        if (ks >= nslices) return;
        a[0] = ldg_u32(wa + 4 * ks);
        a[1] = KA == 2 ? ldg_u32(wa + wstep + 4 * ks) : 0u;
#pragma unroll
        for (int c = 0; c < (int)S::kBSfCols; ++c) {
          int n = 32 * c + lane;  // token of B row 32c + lane
          const bool lo = n >= npad;
          if (lo) n -= npad;
          b[c] = 0x7F7F7F7Fu;
          if (n < t.ntok)
            b[c] = ldg_u32((lo ? q.t_scale_lo : q.t_scale_hi) + (size_t)(t.slot0 + n) * ksb +
                           4 * ks);
        }
      };
#pragma unroll
      for (int j = 0; j < kSfAhead; ++j) load(ra[j], rb[j], j);
      // ks walks the tile's K slices; slice ks is part sb = ks % SUB of stage `it`
      for (int ks0 = 0; ok && ks0 < nslices; ks0 += kSfAhead) {
#pragma unroll
        for (int j = 0; j < kSfAhead; ++j) {
          const int ks = ks0 + j;
          if (ks >= nslices) break;
          const int sb = ks % SUB;
          const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
          if (sb == 0) {
            if (!wait_bar(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
          }
          const uint32_t col = lane_base + sf0 + stage * S::kSfCols;
          tmem_st1(col + 4 * (sb * KA) + qd, ra[j][0]);
          if (KA == 2) tmem_st1(col + 4 * (sb * KA + 1) + qd, ra[j][1]);
          const uint32_t bcol = col + 4 * KA * SUB + sb * S::kBSfCols;
          tmem_st4(bcol, *reinterpret_cast<const uint32_t(*)[4]>(&rb[j][0]));
          if (S::kBSfCols == 8)
            tmem_st4(bcol + 4, *reinterpret_cast<const uint32_t(*)[4]>(&rb[j][4]));
          if (sb == SUB - 1) {
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[stage]);
            ++it;
          }
          load(ra[j], rb[j], ks + kSfAhead);
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

template <bool GATEUP, int NT, int STAGES, int KA, int ACCB, int SUB = 1>
cudaError_t launch_variant(const CUtensorMap& w, const CUtensorMap& hi, const CUtensorMap& lo,
                           const TcParams& p, const MxParams& q, cudaStream_t st) {
  using S = SmemMx<GATEUP, NT, STAGES, KA, ACCB, SUB>;
  static_assert(S::kTotal <= 227 * 1024, "shared memory");
  auto kern = k_tc_ffn_mx<GATEUP, NT, STAGES, KA, ACCB, SUB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S::kTotal);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return launch_pdl(kern, dim3(num_sms()), dim3(kThreadsMx), S::kTotal, st, w, hi, lo, p, q);
}

// Row-major [rows, K] MXFP4 codes (K/2 bytes a row), box of 128 rows x 128 codes, spread into
// shared memory as the MMA reads them (16U4_ALIGN16B: 8 bytes of codes, 8 bytes of gap).
cudaError_t encode_e2m1_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K / 2};
  const cuuint32_t box[2] = {(cuuint32_t)kMxK, (cuuint32_t)kBM};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

// Token tile of the decode batches: 16 tokens while experts average at most 4 routed tokens, 32
// up to 16, 48 up to the decode bound of 32 (few experts then exceed one tile, and 48-token
// tiles leave TMEM room for two accumulators: measured T=1024 1757 -> 1713 us against 64-token
// tiles with one). Prefill batches run the f16 prefill tiles of ffn_tc_fp8_wide.cu.
int tc_mx_tile_tokens(bool decode, long routed, int E) {
  (void)decode;
  return routed > 16L * E ? 48 : routed > 4L * E ? 32 : 16;
}

// Down tiles pair two 128-row tiles of W_d when d allows it (two MMA issuers, one a tile).
int tc_mx_down_rows(bool decode, int d) {
  (void)decode;
  return d % 256 == 0 ? 2 * kBM : kBM;
}

cudaError_t launch_tc_mx(const FfnArgs& a, const int32_t* prefix, bool gateup, bool decode,
                         cudaStream_t st) {
  if (!decode) return launch_tc_mx_wide(a, prefix, gateup, st);
  TcParams p{};
  p.T = a.T; p.k = a.k; p.E = a.E; p.n_shared = a.n_shared;
  p.f = a.f; p.d = a.d;
  p.K = gateup ? a.d : a.f;
  const int dn_rows = tc_mx_down_rows(decode, a.d);
  p.mtiles = gateup ? a.f / kBM : a.d / dn_rows;
  p.rows_per_expert = gateup ? 2 * a.f : a.d;
  p.offsets = a.offsets;
  p.prefix = prefix;
  p.h = nullptr;
  p.y_perm = a.y_perm;
  p.status = a.status;
  if (gateup) p.tile1 = a.tile1;
  const uint64_t E1 = (uint64_t)a.E + a.n_shared;
  const uint64_t routed = (uint64_t)a.T * a.k;
  const uint64_t slots = routed + (uint64_t)a.n_shared * a.T;
  const mx::Planes& tok = gateup ? a.xq : a.hq;
  MxParams q{};
  q.w_scales = static_cast<const uint8_t*>(gateup ? a.s13 : a.s2);
  q.t_scale_hi = tok.s_hi;
  q.t_scale_lo = tok.s_lo;
  q.h = a.hq;
  CUtensorMap w, hi, lo;
  cudaError_t e = gateup ? encode_e2m1_2d(&w, a.w13, E1 * 2 * a.f, a.d)
                         : encode_e2m1_2d(&w, a.w2, E1 * a.d, a.f);
  const uint64_t K = gateup ? a.d : a.f;
  if (e == cudaSuccess) e = encode_u8_2d(&hi, tok.hi, slots ? slots : 1, K, kBoxRows);
  if (e == cudaSuccess) e = encode_u8_2d(&lo, tok.lo, slots ? slots : 1, K, kBoxRows);
  if (e != cudaSuccess) return e;
  const int nt = tc_mx_tile_tokens(decode, (long)routed, a.E);
  if (nt == 48) {
    if (gateup) return launch_variant<true, 48, 5, 2, 2>(w, hi, lo, p, q, st);
    if (dn_rows == 2 * kBM) return launch_variant<false, 48, 5, 2, 2>(w, hi, lo, p, q, st);
    return launch_variant<false, 48, 6, 1, 2>(w, hi, lo, p, q, st);
  }
  // Two 128-wide K slices per stage where K allows (measured: V4-Pro decode 1148 -> 1053 us; the
  // MMA-issuing thread's per-stage waits and commit are paid half as often)
  const bool sub2 = K % 256 == 0;
  if (nt == 16) {
    if (sub2) {
      if (gateup) return launch_variant<true, 16, 3, 2, 2, 2>(w, hi, lo, p, q, st);
      if (dn_rows == 2 * kBM)
        return launch_variant<false, 16, 3, 2, 2, 2>(w, hi, lo, p, q, st);
      return launch_variant<false, 16, 5, 1, 2, 2>(w, hi, lo, p, q, st);
    }
    if (gateup) return launch_variant<true, 16, 6, 2, 2>(w, hi, lo, p, q, st);
    if (dn_rows == 2 * kBM) return launch_variant<false, 16, 6, 2, 2>(w, hi, lo, p, q, st);
    return launch_variant<false, 16, 10, 1, 2>(w, hi, lo, p, q, st);
  }
  if (sub2) {
    if (gateup) return launch_variant<true, 32, 2, 2, 2, 2>(w, hi, lo, p, q, st);
    if (dn_rows == 2 * kBM) return launch_variant<false, 32, 2, 2, 2, 2>(w, hi, lo, p, q, st);
    return launch_variant<false, 32, 4, 1, 2, 2>(w, hi, lo, p, q, st);
  }
  if (gateup) return launch_variant<true, 32, 5, 2, 2>(w, hi, lo, p, q, st);
  if (dn_rows == 2 * kBM) return launch_variant<false, 32, 5, 2, 2>(w, hi, lo, p, q, st);
  return launch_variant<false, 32, 8, 1, 2>(w, hi, lo, p, q, st);
}

}  // namespace moe
