// Pieces shared by the tensor-core expert GEMMs (bf16 and FP8 weights): tile list decoding,
// bounded mbarrier waits, tensor-map encoding.
#pragma once

#include "ffn.h"
#include "sm100_ptx.cuh"

namespace moe {
namespace tc {

using namespace ptx;

constexpr int kBM = 128;               // weight rows per tile (MMA M)
constexpr int kBK = 64;                // K per stage: one 128-byte swizzle row of bf16
constexpr int kBoxRows = 16;           // token rows per TMA box
constexpr uint32_t kATileBytes = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kBBoxBytes = kBoxRows * kBK * 2; // 2 KB
constexpr uint64_t kWaitLimitNs = 2000000000ull;    // 2 s
constexpr int kThreads = 192;

struct TcParams {
  int T, k, E, n_shared;
  int K;                 // reduction width: d (gate/up) or f (down)
  int mtiles;            // 128-row weight tiles per expert
  int rows_per_expert;   // rows of the weight map per expert: 2f (gate/up) or d (down)
  int f, d;
  const int32_t* offsets;  // global memory, or a shared-memory copy (stage_tile_list)
  const int32_t* prefix;   // [E1 + 1] tile prefix over experts (idem)
  uint16_t* h;
  float* y_perm;
  int* status;
  // number of CTAs that take tiles (device memory, written by the plan kernel), or null for
  // all of them: the others leave at once
  const int32_t* active;
  // small-batch gate/up pass: the front's per-CTA tile descriptors (enter_one_tile), or null
  const int4* tile1;
  // one-tile mode (single != 0): this CTA's only tile, {e, m-tile, slot0, ntok} (e < 0: none),
  // read from the small-batch front's descriptors instead of decoding the tile list
  int single;
  int4 one;
};

struct Tile {
  int e, mt, slot0, ntok, brow0;
  bool shared;
  bool multi;  // the expert has more token tiles than this one: its weights are read again
};

// Gate/up pass of the small-batch path: every thread reads this CTA's descriptor (after the
// wait: the front writes it); if the pass has no more tiles than CTAs, the CTA runs in one-tile
// mode (returns the tile count to loop to: blockIdx.x + 1, or 0 without a tile), else -1.
__device__ __forceinline__ int enter_one_tile(TcParams& p) {
  if (!p.tile1 || blockIdx.x >= (unsigned)kTile1Max) return -1;
  const int4 q = p.tile1[blockIdx.x];
  if (q.w >> 16) return -1;
  p.single = 1;
  p.one = q;
  return q.x >= 0 ? (int)blockIdx.x + 1 : 0;
}

// Shared-memory copy of a tile list (prefix and offsets, E1 + 1 entries each; E1 <= 1025).
constexpr uint32_t kTileListBytes = 2 * (1025 + 1) * 4;

// All threads of the block copy the tile list into `sm` (kTileListBytes) and point p at the
// copy, so that the roles decode their tiles from shared memory instead of a chain of dependent
// global loads. Call after the wait for the kernel that wrote the list, with every thread.
__device__ __forceinline__ void stage_tile_list(TcParams& p, int32_t* sm) {
  const int E1 = p.E + p.n_shared;
  for (int i = threadIdx.x; i <= E1; i += blockDim.x) {
    sm[i] = p.prefix[i];
    sm[E1 + 1 + i] = p.offsets[i];
  }
  __syncthreads();
  p.prefix = sm;
  p.offsets = sm + E1 + 1;
}

// stage_tile_list for a list written two or more kernels back, called BEFORE this kernel's
// griddepcontrol.wait: the kernel that wrote the list completed before the previous kernel's
// wait returned, and this kernel was launched after that, so the list is complete in L2; the
// loads bypass L1 (ld.global.cg), whose lines may predate it.
__device__ __forceinline__ void stage_tile_list_early(TcParams& p, int32_t* sm) {
  const int E1 = p.E + p.n_shared;
  for (int i = threadIdx.x; i <= E1; i += blockDim.x) {
    sm[i] = __ldcg(p.prefix + i);
    sm[E1 + 1 + i] = __ldcg(p.offsets + i);
  }
  __syncthreads();
  p.prefix = sm;
  p.offsets = sm + E1 + 1;
}

// Token rows of the gate/up pass come from the gathered rows (routed experts) or straight from
// x (the shared expert, whose slot T*k + t is token t); the down pass reads h in slot order.
template <bool GATEUP, int NT>
__device__ __forceinline__ void decode_tile(const TcParams& p, int tile, Tile& t) {
  if (p.single) {
    t.e = p.one.x;
    t.mt = p.one.y;
    t.slot0 = p.one.z;
    t.ntok = p.one.w & 0xFFFF;
    t.multi = false;
    t.shared = t.e == p.E;
    t.brow0 = (GATEUP && t.shared) ? t.slot0 - p.T * p.k : t.slot0;
    return;
  }
  const int E1 = p.E + p.n_shared;
  int lo = 0, hi = E1;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int seg0 = p.offsets[e];
  const int cnt = p.offsets[e + 1] - seg0;
  const int ntn = (cnt + NT - 1) / NT;
  const int local = tile - p.prefix[e];
  const int mt = local / ntn, nt = local - mt * ntn;
  t.e = e;
  t.mt = mt;
  t.slot0 = seg0 + nt * NT;
  t.ntok = min(NT, cnt - nt * NT);
  t.multi = ntn > 1;
  t.shared = (e == p.E);
  t.brow0 = (GATEUP && t.shared) ? t.slot0 - p.T * p.k : t.slot0;
}

// Bounded wait on an mbarrier phase. Returns false (after recording a timeout) if it gave up
// or if another role already gave up.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        record_error(status, MOE_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag: used to drain this CTA's own copies in flight
// before it exits.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, int* status) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      record_error(status, MOE_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
}

// Epilogue warps (four consecutive warps, so every TMEM lane quadrant is covered): for each
// tile, wait for its accumulator, read it 16 columns at a time, and store SiLU(gate) * up as
// bf16 h (gate/up pass: gate in columns [0, NT), up in [NT, 2NT)) or the fp32 expert output
// (down pass: KA weight tiles of 128 output rows each, tile a in columns [a*NT, (a+1)*NT));
// then hand the accumulator back. ACCB accumulator buffers (1 or 2) rotate. H_F16 writes h as
// f16 (round to nearest, saturating at +-65504) instead of bf16.
template <bool GATEUP, int NT, uint32_t ACC_COLS, int KA = 1, int ACCB = 2, bool H_F16 = false>
// Tiles tile0, tile0 + tstep, ...; cl_rank >= 0 marks clusters of cl CTAs, where a listed tile
// is a group of cl consecutive m-tiles and this CTA takes m-tile cl * mt + cl_rank. With
// empty_in_cta0 (CTA pairs whose MMAs the even CTA issues), the accumulator is handed back on
// the even CTA's acc_empty barrier, wherever this CTA is.
__device__ __forceinline__ void run_epilogue(const TcParams& p, int total, uint32_t tmem_base,
                                             uint64_t* acc_full, uint64_t* acc_empty,
                                             volatile int* abort_flag, int tile0, int tstep,
                                             int cl_rank, int cl = 2, bool empty_in_cta0 = false) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;                 // TMEM lane quadrant this warp may access
  const int row = q * 32 + lane;          // weight row within a 128-row tile
  uint32_t acc = 0, acc_phase = 0;
  for (int tile = tile0; tile < total; tile += tstep) {
    Tile t;
    decode_tile<GATEUP, NT>(p, tile, t);
    if (cl_rank >= 0) t.mt = cl * t.mt + cl_rank;
    const int npad = (t.ntok + 15) & ~15;
    if (!wait_bar(&acc_full[acc], acc_phase, abort_flag, p.status)) break;
    tc_fence_after();
    const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * ACC_COLS;
    if (GATEUP) {
      const int orow = t.mt * kBM + row;  // output feature
      for (int c0 = 0; c0 < npad; c0 += 16) {
        uint32_t g[16], u[16];
        tmem_ld16(tbase + c0, g);
        tmem_ld16(tbase + NT + c0, u);
        tmem_ld_wait2(g, u);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = c0 + j;
          if (n < t.ntok) {
            const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
            const float silu = gv / (1.0f + __expf(-gv));
            p.h[(size_t)(t.slot0 + n) * p.f + orow] =
                H_F16 ? f32_to_f16_satfinite(silu * uv) : f32_to_bf16_rn(silu * uv);
          }
        }
      }
    } else {
#pragma unroll
      for (int a = 0; a < KA; ++a) {
        const int orow = t.mt * (kBM * KA) + a * kBM + row;
        for (int c0 = 0; c0 < npad; c0 += 16) {
          uint32_t g[16];
          tmem_ld16(tbase + a * NT + c0, g);
          tmem_ld_wait(g);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = c0 + j;
            if (n < t.ntok) p.y_perm[(size_t)(t.slot0 + n) * p.d + orow] = __uint_as_float(g[j]);
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (empty_in_cta0)
        mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[acc]), 0));
      else
        mbar_arrive(&acc_empty[acc]);
    }
    if (++acc == ACCB) { acc = 0; acc_phase ^= 1u; }
  }
}

// One CTA per tile list entry, tiles blockIdx.x, blockIdx.x + gridDim.x, ...
template <bool GATEUP, int NT, uint32_t ACC_COLS, int KA = 1, int ACCB = 2>
__device__ __forceinline__ void run_epilogue(const TcParams& p, int total, uint32_t tmem_base,
                                             uint64_t* acc_full, uint64_t* acc_empty,
                                             volatile int* abort_flag) {
  run_epilogue<GATEUP, NT, ACC_COLS, KA, ACCB>(p, total, tmem_base, acc_full, acc_empty,
                                               abort_flag, (int)blockIdx.x, (int)gridDim.x, -1);
}

// ---- host side -------------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Row-major [rows, cols] bf16 matrix, box of box_rows x 64 columns, 128-byte swizzle.
inline cudaError_t encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


// Row-major [rows, cols] byte matrix (E4M3 codes, or MXFP4 code pairs), box of box_rows x
// box_cols bytes, swizzled to match the box width (128, 64 or 32 bytes).
inline cudaError_t encode_u8_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                                uint32_t box_rows, uint32_t box_cols = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_cols == 64   ? CU_TENSOR_MAP_SWIZZLE_64B
                        : box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                         : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tc
}  // namespace moe
