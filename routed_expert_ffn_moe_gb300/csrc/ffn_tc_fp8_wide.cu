// Expert FFN, tensor-core path for FP8 E4M3 expert weights, wide-tile variant for large token
// batches (W8A16). Same passages as ffn_tc_fp8.cu. With up to 256 tokens per tile each weight
// element serves many tokens, so the tile shape follows the bf16 prefill kernel (two 128-row
// weight tiles per 256-token tile, 512 TMEM columns of accumulator) and the dequantisation moves
// to a shared-memory stage of its own:
//
//   TMA (codes)   E4M3 codes (128 rows x 64 K per weight tile, 64-byte swizzle) -> code ring
//   TMA (tokens)  f16 token rows (256 x 64 K, 128-byte swizzle) -> token ring
//   convert       8 warps: f16(code * f16(block scale)) into a third ring in the 128-byte-
//                 swizzle K-major layout the MMA reads: one exact cvt per two codes and one f16x2
//                 multiply (each weight rounded once, 2^-11 relative for products in f16's normal
//                 range, i.e. for block scales above 2^-14: blocks whose largest weight is above
//                 448 * 2^-14 = 0.027; smaller products are f16 subnormals, 2^-24 absolute)
//   MMA           tcgen05.mma.kind::f16, f16 x f16 -> fp32, both operands from smem, one
//                 issuing thread per weight tile (warps 1 and 15)
//   epilogue      TMEM -> SiLU(gate) * up -> f16 h, or the fp32 expert output
//
// The token rows (x gathered in slot order, the shared expert's rows included) and h are f16:
// exact for bf16 x in f16's normal range (|x| between 2^-14 and 65504), h rounded once to f16
// (saturating at +-65504).
//
// MXFP4 weights (MX): the same kernel with E2M1 code pairs (128 rows x 64 codes = 32 bytes a row,
// 32-byte swizzle) and one E8M0 scale per 32 codes of a row. The dequantised weight
// q * 2^(e-127) is exact in f16 (one cvt per two codes, one f16x2 multiply by the power of two)
// for blocks whose scale lies in f16's range (2^-24 .. 2^15; a block's largest weight between
// 2^-19 and 2^16).
//
// The three rings are released independently: a code slot as soon as the converters have read
// it, a token slot and a converted slot when the MMAs that read them complete. The codes are
// the stream that comes from HBM, so they get the deepest ring and a producer thread of their
// own, which runs as far ahead as the code ring allows whatever the token ring is doing.
//
// CTA pairs (cta_group::2, where an expert has an even number of 128-row tiles): the two CTAs of
// a 2-CTA cluster take the consecutive 128-row weight tiles 2j and 2j+1 of the same expert and
// token tile, and one MMA of M = 256 covers both: each CTA converts its own weight rows and
// loads half of the token rows into its own shared memory, the even CTA issues the MMAs (which
// read both CTAs' operands), and each CTA's tensor memory receives its own 128 rows. So every
// SM stages half of each token tile (16 KB a slot instead of 32), which pays for a third
// converted slot and a fourth token slot, and issues half as many MMA instructions. The even
// CTA's barriers gate the MMAs: its token-slot barrier counts both CTAs' TMA bytes (the odd
// CTA's loads complete on it), its converted-slot barrier both CTAs' converters and its
// accumulator-empty barrier both CTAs' epilogues; the MMA commits arrive in both CTAs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_common.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

constexpr uint32_t kCodeTileBytes = kBM * kBK;    // 128 rows x 64 codes = 8 KB
template <bool MX>
constexpr uint32_t code_tile_bytes() { return MX ? kCodeTileBytes / 2 : kCodeTileBytes; }
constexpr int kConvWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kConvWarp0 = 6;                     // converters: warps 6..13
constexpr int kTokWarp = kConvWarp0 + kConvWarps; // token producer: warp 14
constexpr int kIssuer2 = kTokWarp + 1;            // MMA issuer of weight tile 1: warp 15
constexpr int kThreadsW = 32 * (kIssuer2 + 1);

template <int NT, int QS, int BS, int CS, int KA, int ACCB, bool MX, bool PAIR>
struct SmemW {
  static constexpr uint32_t kQSlot = KA * code_tile_bytes<MX>();  // codes of the KA tiles
  // f16 token rows: the whole tile, or (CTA pairs) this CTA's half of it
  static constexpr uint32_t kBSlot = (uint32_t)(PAIR ? NT / 2 : NT) * kBK * 2;
  static constexpr uint32_t kCSlot = KA * kATileBytes;           // converted f16 weight tiles
  static constexpr uint32_t kBOff = QS * kQSlot;
  static constexpr uint32_t kCOff = kBOff + BS * kBSlot;
  static constexpr uint32_t kTilesBytes = kCOff + CS * kCSlot;
  static constexpr uint32_t kBarBytes = 8 * (2 * QS + 2 * BS + 2 * CS + 4) + 16;
  static constexpr uint32_t kTotal = kTilesBytes + kBarBytes + 1024;
  static constexpr uint32_t kAccCols = KA * NT;
  static constexpr uint32_t kTmemCols = ACCB * kAccCols;
};

// Four E4M3 codes (lowest byte first) times the block scale as two f16 pairs (codes 0,1 -> lo,
// codes 2,3 -> hi): each 16-bit half of the word converts exactly to an f16 pair, and one f16x2
// multiply by the scale (an f16 pair) rounds each product once.
__device__ __forceinline__ void dequant4_f16(uint32_t four, uint32_t s2, uint32_t& lo,
                                             uint32_t& hi) {
  asm("{\n"
      "  .reg .b16 c01, c23;\n"
      "  mov.b32 {c01, c23}, %2;\n"
      "  cvt.rn.f16x2.e4m3x2 %0, c01;\n"
      "  cvt.rn.f16x2.e4m3x2 %1, c23;\n"
      "  mul.rn.f16x2 %0, %0, %3;\n"
      "  mul.rn.f16x2 %1, %1, %3;\n"
      "}"
      : "=r"(lo), "=r"(hi)
      : "r"(four), "r"(s2));
}

// fp32 scale -> f16 pair (round to nearest, saturating at the largest finite f16).
__device__ __forceinline__ uint32_t f16x2_of(float v) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(v));
  return r;
}

// 2^(e-127) as an f16 pair, the exponent clamped to f16's range (subnormals down to 2^-24).
__device__ __forceinline__ uint32_t f16x2_pow2(uint32_t e) {
  const int k = min((int)e - 127, 15);
  const uint32_t h = k >= -14 ? (uint32_t)(k + 15) << 10 : (k >= -24 ? 1u << (k + 24) : 0u);
  return h | (h << 16);
}

// Eight E2M1 codes (a word, lowest nibble first) times 2^k as four f16 pairs: each byte converts
// exactly to an f16 pair, and one f16x2 multiply by the power of two scales it (exact in range).
__device__ __forceinline__ void dequant_e2m1x8(uint32_t w, uint32_t s2, uint32_t (&o)[4]) {
  asm("{\n"
      "  .reg .b8 b0, b1, b2, b3;\n"
      "  mov.b32 {b0, b1, b2, b3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "  cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "  cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "  cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      "}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o[i]) : "r"(s2));
}

__device__ __forceinline__ void sts_u4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

template <bool GATEUP, int NT, int QS, int BS, int CS, int KA, int ACCB, bool PAIR, bool MX>
__global__ void __launch_bounds__(kThreadsW, 1)
    k_tc_ffn_fp8_wide(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_b0,
                      const __grid_constant__ CUtensorMap tm_b1,
                      const __grid_constant__ CUtensorMap tm_b0w,
                      const __grid_constant__ CUtensorMap tm_b1w, const TcParams p,
                      const void* __restrict__ scales) {
  using S = SmemW<NT, QS, BS, CS, KA, ACCB, MX, PAIR>;
  static_assert(S::kTmemCols <= 512 && (S::kTmemCols & (S::kTmemCols - 1)) == 0, "TMEM cols");
  static_assert(!GATEUP || KA == 2, "gate/up tiles pair the gate and up rows");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* bring = smem + S::kBOff;
  uint8_t* cring = smem + S::kCOff;
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + S::kTilesBytes);
  uint64_t* q_empty = q_full + QS;
  uint64_t* b_full = q_empty + QS;
  uint64_t* b_empty = b_full + BS;
  uint64_t* c_full = b_empty + BS;
  uint64_t* c_empty = c_full + CS;
  uint64_t* acc_full = c_empty + CS;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E1 = p.E + p.n_shared;
  const int kblocks = p.K / kBK;
  // CTA pairs: both CTAs walk the same list of (expert, pair of m-tiles, token tile) entries;
  // this CTA takes m-tile 2 * mt + rank and rows [rank * n/2, (rank + 1) * n/2) of the tile's n
  // (padded) token rows.
  constexpr int CL = PAIR ? 2 : 1;
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  const bool issuer_cta = rank == 0;  // the CTA whose threads issue the MMAs
  const int tile0 = (int)blockIdx.x / CL;
  const int tstep = (int)gridDim.x / CL;
  const auto decode = [&](int tile, Tile& t) {
    decode_tile<GATEUP, NT>(p, tile, t);
    if (PAIR) t.mt = 2 * t.mt + rank;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < QS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], kConvWarps);   // every converter warp has read its codes
    }
    for (int s = 0; s < BS; ++s) {
      mbar_init(&b_full[s], 1);             // the (even CTA's) token producer, + TMA bytes
      mbar_init(&b_empty[s], KA);           // MMA commits (one per issuer)
    }
    for (int s = 0; s < CS; ++s) {
      mbar_init(&c_full[s], CL * kConvWarps);  // converter warps (of both CTAs of a pair)
      mbar_init(&c_empty[s], KA);           // MMA commits (one per issuer)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], KA);          // one commit per issuer
      mbar_init(&acc_empty[b], 4 * CL);     // epilogue warps (of both CTAs of a pair)
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
    // ---------------- TMA producer: E4M3 codes ----------------
    if (lane == 0) {
      // codes: streamed once per call (evict first), unless the expert has several token
      // tiles, whose tiles run at about the same time on other SMs and read them again
      const uint64_t pol_once = policy_evict_first(), pol_again = policy_evict_normal();
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < total; tile += tstep) {
        Tile t;
        decode(tile, t);
        const uint64_t pol_w = t.multi ? pol_again : pol_once;
        const int wrow = t.e * p.rows_per_expert + t.mt * (GATEUP ? kBM : kBM * KA);
        const int wrow1 = GATEUP ? wrow + p.f : wrow + kBM;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(&q_empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          uint8_t* st = smem + stage * S::kQSlot;
          mbar_arrive_expect_tx(&q_full[stage], S::kQSlot);
          const int xq = MX ? kb * (kBK / 2) : kb * kBK;  // in bytes of the code map
          tma_load_2d(st, &tm_w, &q_full[stage], xq, wrow, pol_w);
          if (KA == 2)
            tma_load_2d(st + code_tile_bytes<MX>(), &tm_w, &q_full[stage], xq, wrow1, pol_w);
          if (++stage == QS) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < QS; ++s)
        drain_bar(&q_full[s], (s < (int)stage) ? phase : (phase ^ 1u), p.status);
    }
  } else if (warp == kTokWarp) {
    // ---------------- TMA producer: f16 token rows ----------------
    if (lane == 0) {
      const uint64_t pol_b = policy_evict_last();
      // pairs: every load of either CTA completes on the even CTA's barrier
      const uint32_t b_full0 = PAIR ? mapa_shared(smem_u32(&b_full[0]), 0) : 0;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = tile0; ok && tile < total; tile += tstep) {
        Tile t;
        decode(tile, t);
        const bool wide = t.ntok == NT;  // one box: NT rows, or NT/2 in pairs
        // this CTA's rows of the tile: all of them, or (pairs) half of the padded count
        const int half = PAIR ? ((t.ntok + 15) & ~15) / 2 : t.ntok;
        const int row0 = t.brow0 + rank * half;
        const int nbox = (half + kBoxRows - 1) / kBoxRows;
        const uint32_t bytes = wide ? S::kBSlot : (uint32_t)nbox * kBBoxBytes;
        const bool sh = GATEUP && t.shared;
        const CUtensorMap* bmap = sh ? &tm_b1 : &tm_b0;
        const CUtensorMap* bmapw = sh ? &tm_b1w : &tm_b0w;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(&b_empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          uint8_t* bt = bring + stage * S::kBSlot;
          if (PAIR) {
            // both halves are the same size, so the even CTA expects twice its own bytes
            if (issuer_cta) mbar_arrive_expect_tx(&b_full[stage], 2 * bytes);
            const uint32_t bar = b_full0 + 8u * stage;
            if (wide) {
              tma_load_2d_pair(bt, bmapw, bar, kb * kBK, row0, pol_b);
            } else {
              for (int i = 0; i < nbox; ++i)
                tma_load_2d_pair(bt + i * kBBoxBytes, bmap, bar, kb * kBK, row0 + i * kBoxRows,
                                 pol_b);
            }
          } else {
            mbar_arrive_expect_tx(&b_full[stage], bytes);
            if (wide) {
              tma_load_2d(bt, bmapw, &b_full[stage], kb * kBK, t.brow0, pol_b);
            } else {
              for (int i = 0; i < nbox; ++i)
                tma_load_2d(bt + i * kBBoxBytes, bmap, &b_full[stage], kb * kBK,
                            t.brow0 + i * kBoxRows, pol_b);
            }
          }
          if (++stage == BS) { stage = 0; phase ^= 1u; }
        }
      }
      // every issued load has landed (in pairs the even CTA's barrier counts both CTAs' bytes)
      if (!PAIR || issuer_cta)
        for (int s = 0; s < BS; ++s)
          drain_bar(&b_full[s], (s < (int)stage) ? phase : (phase ^ 1u), p.status);
      if (PAIR) {
        // the MMA commits for every issued stage have arrived here before the CTA may exit
        for (int s = 0; s < BS; ++s)
          drain_bar(&b_empty[s], (s < (int)stage) ? phase : (phase ^ 1u), p.status);
      }
    }
  } else if (warp == 1 || warp == kIssuer2) {
    // ---------------- MMA issuers: warp 1 weight tile 0, warp 15 weight tile 1 ----------------
    const int o = warp == 1 ? 0 : 1;
    if (lane == 0 && o < KA && issuer_cta) {
      uint32_t bs = 0, bphase = 0, cs = 0, cphase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      constexpr int kM = PAIR ? 2 * kBM : kBM;  // a pair's MMA covers both CTAs' weight rows
      for (int tile = tile0; ok && tile < total; tile += tstep) {
        Tile t;
        decode(tile, t);
        const int npad = (t.ntok + 15) & ~15;
        // f16 x f16 (A and B formats 0), fp32 accumulate
        const uint32_t idesc =
            (1u << 4) | ((uint32_t)(npad >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
        if (!wait_bar(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc * S::kAccCols + o * NT;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(&b_full[bs], bphase, abort_flag, p.status) ||
              !wait_bar(&c_full[cs], cphase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t da = sw128_desc(smem_u32(cring + cs * S::kCSlot) + o * kATileBytes);
          const uint64_t db = sw128_desc(smem_u32(bring + bs * S::kBSlot));
          if (PAIR) {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_ss_pair(d0, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
            mma_commit_pair(&b_empty[bs]);   // token rows consumed, in both CTAs
            mma_commit_pair(&c_empty[cs]);   // dequantised weights consumed, in both CTAs
          } else {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16_ss(d0, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
            mma_commit(&b_empty[bs]);        // token rows consumed
            mma_commit(&c_empty[cs]);        // dequantised weights consumed
          }
          if (++bs == BS) { bs = 0; bphase ^= 1u; }
          if (++cs == CS) { cs = 0; cphase ^= 1u; }
        }
        if (!ok) break;
        if (PAIR)
          mma_commit_pair(&acc_full[acc]);
        else
          mma_commit(&acc_full[acc]);
        if (++acc == ACCB) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else if (warp < kConvWarp0) {
    // ---------------- epilogue (warps 2..5) ----------------
    run_epilogue<GATEUP, NT, S::kAccCols, KA, ACCB, true>(p, total, tmem_base, acc_full, acc_empty,
                                                        abort_flag, tile0, tstep,
                                                        PAIR ? rank : -1, CL,
                                                        PAIR && !issuer_cta);
  } else if (MX) {
    // ---------------- dequantisers, MXFP4 (warps 6..13) ----------------
    // thread = (row r, 32-code chunk j) of every weight tile a: 16 bytes of code pairs and their
    // scale byte -> four 16-byte f16 chunks (4j .. 4j+3 of the row's eight)
    const int ct = threadIdx.x - 32 * kConvWarp0;
    const int r = ct >> 1, j = ct & 1;
    const uint8_t* wsc = static_cast<const uint8_t*>(scales);
    const int ksb = p.K / 32;
    uint32_t qs = 0, qphase = 0, cs = 0, cphase = 0;
    bool ok = true;
    for (int tile = tile0; ok && tile < total; tile += tstep) {
      Tile t;
      decode(tile, t);
      const int wrow = t.e * p.rows_per_expert + t.mt * (GATEUP ? kBM : kBM * KA);
      const int wrow1 = GATEUP ? wrow + p.f : wrow + kBM;
      const uint8_t* s0p = wsc + (size_t)(wrow + r) * ksb + j;   // byte for stage kb: + 2 kb
      const uint8_t* s1p = wsc + (size_t)(wrow1 + r) * ksb + j;
      // scale bytes run one stage ahead so their load latency hides behind the conversion
      uint32_t e0 = __ldg(s0p), e1 = KA == 2 ? __ldg(s1p) : 127u;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_bar(&q_full[qs], qphase, abort_flag, p.status) ||
            !wait_bar(&c_empty[cs], cphase ^ 1u, abort_flag, p.status)) { ok = false; break; }
        const bool more = kb + 1 < kblocks;
        const uint32_t e0n = more ? __ldg(s0p + 2 * (kb + 1)) : 127u;
        const uint32_t e1n = (KA == 2 && more) ? __ldg(s1p + 2 * (kb + 1)) : 127u;
        const uint32_t src = smem_u32(smem + qs * S::kQSlot);
        const uint32_t dst = smem_u32(cring + cs * S::kCSlot);
#pragma unroll
        for (int a = 0; a < KA; ++a) {
          // source: 32-byte rows, 32-byte swizzle (16-byte chunk j ^ ((r >> 2) & 1))
          const uint4 raw =
              lds_u4(src + a * code_tile_bytes<MX>() + r * 32 + ((j ^ ((r >> 2) & 1)) << 4));
          const uint32_t s2 = f16x2_pow2(a ? e1 : e0);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          const uint32_t rowb = dst + a * kATileBytes + r * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t o[4];
            dequant_e2m1x8(w[q], s2, o);
            // destination: 128-byte rows, 128-byte swizzle (16-byte chunk c ^ (r & 7))
            sts_u4(rowb + (((4 * j + q) ^ (r & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
          }
        }
        fence_proxy_async_smem();      // f16 weights -> visible to the MMA
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&q_empty[qs]);   // this warp is done with the codes of this stage
          if (PAIR && !issuer_cta)     // the even CTA's MMA reads both CTAs' weights
            mbar_arrive_cluster(mapa_shared(smem_u32(&c_full[cs]), 0));
          else
            mbar_arrive(&c_full[cs]);
        }
        e0 = e0n;
        e1 = e1n;
        if (++qs == QS) { qs = 0; qphase ^= 1u; }
        if (++cs == CS) { cs = 0; cphase ^= 1u; }
      }
    }
  } else {
    // ---------------- dequantisers (warps 6..13) ----------------
    // task = (weight tile a, row r, 16-code chunk j): 16 codes -> two 16-byte f16 chunks
    const int ct = threadIdx.x - 32 * kConvWarp0;
    const int kbl = p.K / 128;               // scale blocks along K
    uint32_t qs = 0, qphase = 0, cs = 0, cphase = 0;
    bool ok = true;
    for (int tile = tile0; ok && tile < total; tile += tstep) {
      Tile t;
      decode(tile, t);
      const float* sc = static_cast<const float*>(scales) + (size_t)t.e * (p.rows_per_expert / 128) * kbl;
      const int rb0 = GATEUP ? t.mt : t.mt * KA;   // scale row block of the first weight tile
      const int rb1 = GATEUP ? p.f / 128 + t.mt : rb0 + 1;
      // scales run one stage ahead so their load latency hides behind the conversion
      float s0 = __ldg(sc + rb0 * kbl), s1 = KA == 2 ? __ldg(sc + rb1 * kbl) : 0.f;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_bar(&q_full[qs], qphase, abort_flag, p.status) ||
            !wait_bar(&c_empty[cs], cphase ^ 1u, abort_flag, p.status)) { ok = false; break; }
        const bool more = kb + 1 < kblocks;
        const float s0_next = more ? __ldg(sc + rb0 * kbl + ((kb + 1) >> 1)) : 0.f;
        const float s1_next = (KA == 2 && more) ? __ldg(sc + rb1 * kbl + ((kb + 1) >> 1)) : 0.f;
        const uint32_t src = smem_u32(smem + qs * S::kQSlot);
        const uint32_t dst = smem_u32(cring + cs * S::kCSlot);
        const uint32_t s0h = f16x2_of(s0), s1h = f16x2_of(s1);
#pragma unroll
        for (int i = 0; i < KA * kBM * 4 / kConvThreads; ++i) {
          const int task = ct + i * kConvThreads;
          const int a = task / (kBM * 4);
          const int r = (task >> 2) & (kBM - 1);
          const int j = task & 3;
          // source: 64-byte rows, 64-byte swizzle (16-byte chunk j ^ ((r >> 1) & 3))
          const uint4 raw = lds_u4(src + a * kCodeTileBytes + r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
          const uint32_t s2 = a ? s1h : s0h;
          uint4 lo, hi;  // codes 0..7 -> chunk 2j, codes 8..15 -> chunk 2j+1
          dequant4_f16(raw.x, s2, lo.x, lo.y);
          dequant4_f16(raw.y, s2, lo.z, lo.w);
          dequant4_f16(raw.z, s2, hi.x, hi.y);
          dequant4_f16(raw.w, s2, hi.z, hi.w);
          // destination: 128-byte rows, 128-byte swizzle (16-byte chunk c ^ (r & 7))
          const uint32_t rowb = dst + a * kATileBytes + r * 128;
          sts_u4(rowb + (((2 * j) ^ (r & 7)) << 4), lo);
          sts_u4(rowb + (((2 * j + 1) ^ (r & 7)) << 4), hi);
        }
        fence_proxy_async_smem();      // f16 weights -> visible to the MMA
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&q_empty[qs]);   // this warp is done with the codes of this stage
          if (PAIR && !issuer_cta)     // the even CTA's MMA reads both CTAs' weights
            mbar_arrive_cluster(mapa_shared(smem_u32(&c_full[cs]), 0));
          else
            mbar_arrive(&c_full[cs]);
        }
        s0 = s0_next;
        s1 = s1_next;
        if (++qs == QS) { qs = 0; qphase ^= 1u; }
        if (++cs == CS) { cs = 0; cphase ^= 1u; }
      }
    }
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

template <bool GATEUP, int NT, int QS, int BS, int CS, int KA, int ACCB, bool PAIR, bool MX>
cudaError_t launch_variant(const CUtensorMap& w, const CUtensorMap& b0, const CUtensorMap& b1,
                           const CUtensorMap& b0w, const CUtensorMap& b1w, const TcParams& p,
                           const void* scales, cudaStream_t st) {
  using S = SmemW<NT, QS, BS, CS, KA, ACCB, MX, PAIR>;
  static_assert(S::kTotal <= 227 * 1024, "shared memory");
  auto kern = k_tc_ffn_fp8_wide<GATEUP, NT, QS, BS, CS, KA, ACCB, PAIR, MX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S::kTotal);
  if (e != cudaSuccess) return e;
  count_launches(1);
  if (PAIR)
    return launch_pdl_cluster(kern, dim3((unsigned)(num_sms() / 2 * 2)), dim3(kThreadsW),
                              S::kTotal, st, 2u, w, b0, b1, b0w, b1w, p, scales);
  return launch_pdl(kern, dim3(num_sms()), dim3(kThreadsW), S::kTotal, st, w, b0, b1, b0w, b1w, p,
                    scales);
}

struct Maps {
  CUtensorMap w, b0, b1, b0w, b1w;
};

// 256 tokens per tile: a measured sweep with 128-token tiles and deeper rings was slower at
// every batch size tried (more tiles per expert, each converting the same weights).
constexpr int kNT = 256;

// Weight rows per tile of a pass: 2 x 128 (gate + up, or two W_d tiles when d allows), else 128.
bool paired_tiles(bool gateup, int d) { return gateup || tc_tile_rows(false, false, d) == 2 * kBM; }

// CTA pairs (cta_group::2) take two consecutive m-tiles: when an expert's m-tile count is even,
// else single CTAs (1).
int cluster_size(bool gateup, int d, int f) {
  if (!paired_tiles(gateup, d)) return 1;
  const int mtiles = gateup ? f / kBM : d / (2 * kBM);
  return mtiles % 2 == 0 ? 2 : 1;
}

// One pass with kNT-token tiles; rings (codes, tokens, converted weights): CTA pairs 4/4/3 slots
// (a token slot holds half a tile: 224 KB of shared memory); single CTAs 4/3/2 for paired weight
// tiles (224 KB), 8/3/3 for single tiles; fewer token slots measured slower.
template <bool PAIR, bool MX>
cudaError_t launch_pass(const Maps& m, const TcParams& p, const void* sc, bool gateup,
                        bool paired, cudaStream_t st) {
  constexpr int BS = PAIR ? 4 : 3, CS = PAIR ? 3 : 2;
  if (gateup)
    return launch_variant<true, kNT, 4, BS, CS, 2, 1, PAIR, MX>(m.w, m.b0, m.b1, m.b0w, m.b1w, p,
                                                                sc, st);
  if (paired)
    return launch_variant<false, kNT, 4, BS, CS, 2, 1, PAIR, MX>(m.w, m.b0, m.b1, m.b0w, m.b1w, p,
                                                                 sc, st);
  return launch_variant<false, kNT, 8, 3, 3, 1, 2, false, MX>(m.w, m.b0, m.b1, m.b0w, m.b1w, p,
                                                              sc, st);
}

}  // namespace

int tc_fp8_wide_tile_tokens() { return kNT; }

int tc_fp8_wide_plan_mtiles(bool gateup, int d, int f) {
  const int rows = paired_tiles(gateup, d) && !gateup ? 2 * kBM : kBM;
  const int mtiles = (gateup ? f : d) / rows;
  return mtiles / cluster_size(gateup, d, f);
}

cudaError_t launch_tc_fp8_wide(const FfnArgs& a, const int32_t* prefix, bool gateup,
                               cudaStream_t st) {
  TcParams p{};
  p.T = a.T; p.k = a.k; p.E = a.E; p.n_shared = a.n_shared;
  p.f = a.f; p.d = a.d;
  p.K = gateup ? a.d : a.f;
  p.mtiles = tc_fp8_wide_plan_mtiles(gateup, a.d, a.f);
  p.rows_per_expert = gateup ? 2 * a.f : a.d;
  p.offsets = a.offsets;
  p.prefix = prefix;
  p.h = a.h;
  p.y_perm = a.y_perm;
  p.status = a.status;
  const int cl = cluster_size(gateup, a.d, a.f);
  const uint32_t wide_rows = kNT / cl;  // in a CTA pair each CTA loads half of a full tile
  const uint64_t E1 = (uint64_t)a.E + a.n_shared;
  const uint64_t routed = (uint64_t)a.T * a.k;
  const uint64_t slots = routed + (uint64_t)a.T;  // rows of the workspace's f16 x and h
  Maps m;
  cudaError_t e;
  if (gateup) {
    // f16 token rows of every slot (the gather writes them), the shared expert's from T*k on
    const uint16_t* xs = a.x_perm + routed * (uint64_t)a.d;
    e = encode_u8_2d(&m.w, a.w13, E1 * 2 * a.f, a.d, kBM, 64);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b0, a.x_perm, slots, a.d, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b1, xs, a.T, a.d, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b0w, a.x_perm, slots, a.d, wide_rows);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b1w, xs, a.T, a.d, wide_rows);
  } else {
    e = encode_u8_2d(&m.w, a.w2, E1 * a.d, a.f, kBM, 64);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b0, a.h, slots, a.f, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b0w, a.h, slots, a.f, wide_rows);
    m.b1 = m.b0;
    m.b1w = m.b0w;
  }
  if (e != cudaSuccess) return e;
  const void* sc = gateup ? a.s13 : a.s2;
  const bool paired = paired_tiles(gateup, a.d);
  if (cl == 2) return launch_pass<true, false>(m, p, sc, gateup, paired, st);
  return launch_pass<false, false>(m, p, sc, gateup, paired, st);
}

// MXFP4 weights on the same prefill tiles, with the same f16 token rows.
cudaError_t launch_tc_mx_wide(const FfnArgs& a, const int32_t* prefix, bool gateup,
                              cudaStream_t st) {
  TcParams p{};
  p.T = a.T; p.k = a.k; p.E = a.E; p.n_shared = a.n_shared;
  p.f = a.f; p.d = a.d;
  p.K = gateup ? a.d : a.f;
  p.mtiles = tc_fp8_wide_plan_mtiles(gateup, a.d, a.f);
  p.rows_per_expert = gateup ? 2 * a.f : a.d;
  p.offsets = a.offsets;
  p.prefix = prefix;
  p.h = a.h;
  p.y_perm = a.y_perm;
  p.status = a.status;
  const int cl = cluster_size(gateup, a.d, a.f);
  const uint32_t wide_rows = kNT / cl;
  const uint64_t E1 = (uint64_t)a.E + a.n_shared;
  const uint64_t routed = (uint64_t)a.T * a.k;
  const uint64_t slots = routed + (uint64_t)a.T;  // rows of the workspace's f16 x and h
  Maps m;
  cudaError_t e;
  if (gateup) {
    const uint16_t* xs = a.x_perm + routed * (uint64_t)a.d;  // the shared segment's rows
    e = encode_u8_2d(&m.w, a.w13, E1 * 2 * a.f, a.d / 2, kBM, 32);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b0, a.x_perm, slots, a.d, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b1, xs, a.T, a.d, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b0w, a.x_perm, slots, a.d, wide_rows);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b1w, xs, a.T, a.d, wide_rows);
  } else {
    e = encode_u8_2d(&m.w, a.w2, E1 * a.d, a.f / 2, kBM, 32);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b0, a.h, slots, a.f, kBoxRows);
    if (e == cudaSuccess) e = encode_bf16_2d(&m.b0w, a.h, slots, a.f, wide_rows);
    m.b1 = m.b0;
    m.b1w = m.b0w;
  }
  if (e != cudaSuccess) return e;
  const void* sc = gateup ? a.s13 : a.s2;
  const bool paired = paired_tiles(gateup, a.d);
  if (cl == 2) return launch_pass<true, true>(m, p, sc, gateup, paired, st);
  return launch_pass<false, true>(m, p, sc, gateup, paired, st);
}

}  // namespace moe
