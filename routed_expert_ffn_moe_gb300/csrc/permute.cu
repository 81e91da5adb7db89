// Token -> expert permutation: a deterministic, stable counting sort of the T*k (token, choice)
// pairs by expert ("第 6 章 超節點", 6.2.6: the receiver reorders its input rows by expert before
// the matrix multiply and restores token order afterwards).
//
// Tokens are cut into 32-token chunks, one warp each. For its chunk a warp builds, in shared
// memory, one 32-bit mask per expert of the lanes (tokens) that chose it; the popcount of a
// mask is the chunk's count for that expert, and the popcount of the mask below a lane is that
// token's rank among the chunk's tokens of the same expert. An exclusive scan over
// (expert, chunk) in expert-major order then gives every pair its slot. No atomic decides an
// order: the OR of bits is order-independent.
#include "internal.h"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

// Valid choice: in range and not a repeat of an earlier choice of the same token.
__device__ __forceinline__ bool valid_choice(const int32_t* row, int j, int E) {
  const int e = row[j];
  if ((unsigned)e >= (unsigned)E) return false;
  for (int j2 = 0; j2 < j; ++j2)
    if (row[j2] == e) return false;
  return true;
}

// Builds this warp's expert -> lane mask table for its chunk.
__device__ __forceinline__ void build_masks(uint32_t* sel, const int32_t* topk_idx, int T, int E,
                                            int k, int chunk, int nchunk, int* status) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < E; e += 32) sel[e] = 0;
  __syncwarp();
  const int t = chunk * kChunkTokens + lane;
  if (chunk < nchunk && t < T) {
    const int32_t* row = topk_idx + (size_t)t * k;
    for (int j = 0; j < k; ++j) {
      if (valid_choice(row, j, E))
        atomicOr(&sel[row[j]], 1u << lane);
      else
        record_error(status, MOE_ERR_DEVICE_BOUNDS);
    }
  }
  __syncwarp();
}

__global__ void __launch_bounds__(256) k_perm_count(const int32_t* __restrict__ topk_idx, int T,
                                                    int E, int k, int nchunk,
                                                    int32_t* __restrict__ hist, int* status) {
  pdl_wait_then_release();
  extern __shared__ uint32_t sel_all[];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kWarpsPerBlock + wid;
  uint32_t* sel = sel_all + (size_t)wid * E;
  build_masks(sel, topk_idx, T, E, k, chunk, nchunk, status);
  if (chunk < nchunk)
    for (int e = lane; e < E; e += 32) hist[(size_t)e * nchunk + chunk] = __popc(sel[e]);
}

// One block: exclusive scan of hist (expert-major) into base; expert offsets from it. The array
// is walked in coalesced 4096-entry pieces (4 per thread, int4 loads), each block-scanned and
// offset by the running total of the pieces before it.
__global__ void __launch_bounds__(1024) k_perm_scan(const int32_t* __restrict__ hist, int E,
                                                    int nchunk, int T, int k, int n_shared,
                                                    int32_t* __restrict__ base,
                                                    int32_t* __restrict__ offsets) {
  pdl_wait_then_release();
  // One block scans the expert-major [E, nchunk] counts in pieces of 16 entries per thread;
  // each piece's loads are issued one piece ahead so their latency overlaps the block scan.
  constexpr int kPer = 16;
  const long n = (long)E * nchunk;
  const long step = (long)kPer * blockDim.x;
  const auto load = [&](long b0, int (&v)[kPer]) {
    const long i0 = b0 + (long)kPer * threadIdx.x;
    if (i0 + kPer <= n) {  // hist is 256-byte aligned and i0 a multiple of 16 entries
#pragma unroll
      for (int q = 0; q < kPer / 4; ++q) {
        const int4 w = __ldg(reinterpret_cast<const int4*>(hist + i0) + q);
        v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < kPer; ++q) v[q] = (i0 + q < n) ? __ldg(hist + i0 + q) : 0;
    }
  };
  int cur[kPer], nxt[kPer];
  load(0, cur);
  int carry = 0;
  for (long b0 = 0; b0 < n; b0 += step) {
    if (b0 + step < n) load(b0 + step, nxt);
    int sum = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) sum += cur[q];
    int total;
    int run = carry + block_exclusive_scan(sum, &total);
    const long i0 = b0 + (long)kPer * threadIdx.x;
    if (i0 + kPer <= n) {
#pragma unroll
      for (int q = 0; q < kPer / 4; ++q) {
        int4 w;
        w.x = run; run += cur[4 * q];
        w.y = run; run += cur[4 * q + 1];
        w.z = run; run += cur[4 * q + 2];
        w.w = run; run += cur[4 * q + 3];
        reinterpret_cast<int4*>(base + i0)[q] = w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        if (i0 + q < n) base[i0 + q] = run;
        run += cur[q];
      }
    }
    carry += total;
#pragma unroll
    for (int q = 0; q < kPer; ++q) cur[q] = nxt[q];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    offsets[e] = nchunk ? base[(size_t)e * nchunk] : 0;
  if (threadIdx.x == 0) {
    offsets[E] = T * k;
    offsets[E + 1] = T * k + n_shared * T;
  }
}

__global__ void __launch_bounds__(256) k_perm_scatter(const int32_t* __restrict__ topk_idx, int T,
                                                      int E, int k, int nchunk,
                                                      const int32_t* __restrict__ base,
                                                      int32_t* __restrict__ perm_token,
                                                      int32_t* __restrict__ inv_slot) {
  pdl_wait_then_release();
  extern __shared__ uint32_t sel_all[];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kWarpsPerBlock + wid;
  uint32_t* sel = sel_all + (size_t)wid * E;
  build_masks(sel, topk_idx, T, E, k, chunk, nchunk, nullptr);
  const int t = chunk * kChunkTokens + lane;
  if (chunk >= nchunk || t >= T) return;
  const int32_t* row = topk_idx + (size_t)t * k;
  const uint32_t below = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    if (!valid_choice(row, j, E)) {
      inv_slot[(size_t)t * k + j] = -1;
      continue;
    }
    const int e = row[j];
    const int slot = base[(size_t)e * nchunk + chunk] + __popc(sel[e] & below);
    perm_token[slot] = t;
    inv_slot[(size_t)t * k + j] = slot;
  }
}

// Small batches (at most kWarpsPerBlock chunks): the three steps above in one block. Warp w
// builds the masks of chunk w; the (expert, chunk) counts go to shared memory, are scanned there
// in expert-major order, and the same masks then give every pair its slot. Same result as the
// three kernels, one launch instead of three.
__global__ void __launch_bounds__(256) k_perm_small(const int32_t* __restrict__ topk_idx, int T,
                                                    int E, int k, int nchunk, int n_shared,
                                                    int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ perm_token,
                                                    int32_t* __restrict__ inv_slot, int* status) {
  pdl_wait_then_release();
  extern __shared__ uint32_t sm[];
  uint32_t* sel_all = sm;                                       // [kWarpsPerBlock][E]
  int* cnt = reinterpret_cast<int*>(sm + (size_t)kWarpsPerBlock * E);  // [E][nchunk]
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* sel = sel_all + (size_t)wid * E;
  build_masks(sel, topk_idx, T, E, k, wid, nchunk, status);
  if (wid < nchunk)
    for (int e = lane; e < E; e += 32) cnt[e * nchunk + wid] = __popc(sel[e]);
  __syncthreads();
  // exclusive scan of cnt in place, each thread a run of consecutive entries
  const int n = E * nchunk;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int i0 = min(n, (int)threadIdx.x * per), i1 = min(n, i0 + per);
  int sum = 0;
  for (int i = i0; i < i1; ++i) sum += cnt[i];
  int total;
  int run = block_exclusive_scan(sum, &total);
  for (int i = i0; i < i1; ++i) {
    const int v = cnt[i];
    cnt[i] = run;
    run += v;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = cnt[e * nchunk];
  if (threadIdx.x == 0) {
    offsets[E] = T * k;
    offsets[E + 1] = T * k + n_shared * T;
  }
  const int t = wid * kChunkTokens + lane;
  if (wid >= nchunk || t >= T) return;
  const int32_t* row = topk_idx + (size_t)t * k;
  const uint32_t below = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    if (!valid_choice(row, j, E)) {
      inv_slot[(size_t)t * k + j] = -1;
      continue;
    }
    const int e = row[j];
    const int slot = cnt[e * nchunk + wid] + __popc(sel[e] & below);
    perm_token[slot] = t;
    inv_slot[(size_t)t * k + j] = slot;
  }
}

}  // namespace

cudaError_t launch_permute(const moe_shape& s, const int32_t* topk_idx, int32_t* offsets,
                           int32_t* perm_token, int32_t* inv_slot, char* ws, const WsLayout& L,
                           cudaStream_t st) {
  int* status = reinterpret_cast<int*>(ws + L.status);
  int32_t* hist = reinterpret_cast<int32_t*>(ws + L.hist);
  int32_t* base = reinterpret_cast<int32_t*>(ws + L.base);
  const int nchunk = L.nchunk;
  const unsigned blocks = (unsigned)((nchunk + kWarpsPerBlock - 1) / kWarpsPerBlock);
  const size_t smem = (size_t)kWarpsPerBlock * s.E * sizeof(uint32_t);
  const size_t smem_small = smem + (size_t)s.E * nchunk * sizeof(int);
  if (blocks == 1 && smem_small <= 48 * 1024) {
    count_launches(1);
    return launch_pdl(k_perm_small, dim3(1), dim3(32 * kWarpsPerBlock), smem_small, st, topk_idx,
                      s.T, s.E, s.k, nchunk, s.n_shared, offsets, perm_token, inv_slot, status);
  }
  if (blocks) {
    cudaError_t e = launch_pdl(k_perm_count, dim3(blocks), dim3(32 * kWarpsPerBlock), smem, st,
                               topk_idx, s.T, s.E, s.k, nchunk, hist, status);
    if (e != cudaSuccess) return e;
  }
  count_launches(blocks ? 3 : 1);
  cudaError_t e = launch_pdl(k_perm_scan, dim3(1), dim3(1024), 0, st, hist, s.E, nchunk, s.T, s.k,
                             s.n_shared, base, offsets);
  if (e != cudaSuccess || !blocks) return e;
  return launch_pdl(k_perm_scatter, dim3(blocks), dim3(32 * kWarpsPerBlock), smem, st, topk_idx,
                    s.T, s.E, s.k, nchunk, base, perm_token, inv_slot);
}

}  // namespace moe
