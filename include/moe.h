/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed-expert MoE FFN layer, inference hot path.
 *
 * The layer, as the pages state it:
 *   router     -- score every routed expert for each token, keep the top-k
 *                 ("DeepSeek-V4-Pro on NVIDIA H200", section 0.2.2, step D4);
 *   permute    -- reorder the token rows by expert ("第 6 章 超節點", section 6.2.6: the receiver
 *                 reorders rows by expert, multiplies, then restores token order);
 *   expert FFN -- per expert Y = [SiLU(X W_g) (.) (X W_u)] W_d ("第 6 章 超節點", section 6.2.2),
 *                 three GEMMs per expert ("DeepSeek V3/R1 Inference Efficiency (1)", Parameters);
 *   combine    -- routing-weighted sum of the experts' outputs, a1*y1 + a6*y6, plus the
 *                 always-on shared expert ("第 6 章 超節點", sections 6.2.6 and 6.4.1;
 *                 "DeepSeek-V4-Pro on NVIDIA H200", section 0.1.2 and step D7).
 * On one GPU the dispatch and combine exchanges become in-HBM gathers.
 *
 * One GPU. The library has no multi-GPU path: every call works on buffers of the current
 * device only, and no kernel loads from another GPU's memory or multicasts a load. Its prefill
 * tiles run on CTA pairs (tcgen05 cta_group::2): each CTA of a 2-CTA cluster loads its own
 * weight rows and half of the token tile, and one MMA of the pair reads both CTAs' operands.
 *
 * Conventions shared by every entry point
 *   - Pointers named x, wg, bias, topk_*, expert_offsets, perm_token, inv_slot, w13, s13, w2,
 *     s2, y_perm, y and ws are DEVICE pointers, allocated and owned by the caller. The library
 *     never allocates, frees or synchronises in these calls; work is enqueued on `stream`
 *     (a cudaStream_t, NULL = legacy default stream) and the call returns immediately
 *     (moe_expert_ffn may also use one library-owned stream per device; see there).
 *   - `shape` is a host pointer read during the call only.
 *   - Arguments are validated on the host first: a negative status is returned before any
 *     launch and nothing is written (no side effects).
 *   - Device-side checks (an index out of range, a duplicated expert in a token's top-k row, a
 *     bounded wait that gave up) never fault: the kernel skips the bad access and records the
 *     first error code in the workspace; moe_check_device_status() reports it.
 *   - Tensors are dense row-major; "bf16" is IEEE-style bfloat16, "E4M3" is OCP FP8 E4M3;
 *     "MXFP4" is the OCP Microscaling (MX) v1.0 FP4 format: E2M1 elements with one E8M0 scale
 *     per 32 consecutive elements of a row.
 *   - Every pointer must be 16-byte aligned (256-byte for ws; 32-byte for MXFP4 w13 and w2).
 *   - Shapes: 1 <= E <= 1024, 1 <= k <= min(E, 32), n_shared in {0, 1}, d and f multiples of
 *     128 with 128 <= d <= 16384 and 128 <= f <= 16384, 0 <= T and T*(k+1) <= 2^30.
 *   - Not thread-safe per workspace: calls that share a workspace must be ordered on one stream.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,     /* bad pointer, shape or alignment (host check)             */
  MOE_ERR_UNSUPPORTED = -2,     /* valid request this build does not serve (e.g. no GPU)    */
  MOE_ERR_WORKSPACE = -3,       /* ws_bytes < moe_workspace_size(shape)                     */
  MOE_ERR_CUDA = -4,            /* a CUDA runtime/driver call or a launch failed            */
  MOE_ERR_DEVICE_TIMEOUT = -5,  /* a bounded device wait gave up (reported by the check)    */
  MOE_ERR_DEVICE_BOUNDS = -6    /* a device-side index check failed (reported by the check) */
} moe_status;

typedef enum {
  MOE_W_BF16 = 0,            /* expert weights bf16                                          */
  MOE_W_FP8_E4M3_B128 = 1,   /* expert weights E4M3 with one fp32 scale per 128x128 block    */
  MOE_W_MXFP4_E8M0_B32 = 2   /* expert weights MXFP4: E2M1 codes, one E8M0 scale per 32      */
} moe_wdtype;

typedef struct {
  int32_t T;         /* tokens in the batch                                                   */
  int32_t d;         /* hidden size                                                           */
  int32_t E;         /* routed experts                                                        */
  int32_t k;         /* routed experts chosen per token                                       */
  int32_t f;         /* expert intermediate size                                              */
  int32_t n_shared;  /* shared (always-on) experts, 0 or 1; the shared expert is index E      */
  int32_t wdtype;    /* moe_wdtype of w13/w2                                                  */
} moe_shape;

/* Bytes of scratch (`ws`) the four calls need for this shape; 0 for an invalid shape. One
 * workspace serves all four calls of a layer. Its first 4 bytes are the device status word:
 * moe_route clears it (a layer starts there); a caller that skips moe_route must zero those
 * 4 bytes once before its first call. Nothing else in it needs initialisation. */
MOE_API size_t moe_workspace_size(const moe_shape* shape);

/* Router ("DeepSeek-V4-Pro on NVIDIA H200", 0.2.2 D4; "CANN DeepSeek-V4推理优化", MoE
 * 专家模型规格, soft routing).
 *   x        [T, d] bf16 tokens.        wg [E, d] bf16 router weight (one row per expert).
 *   bias     [E] fp32 added to the logits, or NULL.
 *   topk_idx [T, k] int32 out: the k experts with the largest logits, by descending logit,
 *            ties to the lower expert index.
 *   topk_w   [T, k] fp32 out: softmax over all E logits, renormalised over the k chosen
 *            (= softmax over the k chosen logits).
 * The logit l[t,e] = x[t].wg[e] (+ bias[e]) is formed in fp32 in one fixed order, so the
 * choice is reproducible bit for bit: d is cut into 8-element chunks, lane j of 32 accumulates
 * chunks j, j+32, ... element by element with fused multiply-add from +0, the 32 lane sums
 * are combined by an xor butterfly (offsets 16, 8, 4, 2, 1), then the bias is added.
 * Batches of 1024 tokens or more, with E a multiple of 128 and d a multiple of 64, first form
 * approximate logits on the tensor cores; each is taken to lie within 2^-12 |x[t]| |wg[e]| of
 * the defined logit (a bound checked on every logit recomputed), so only the experts that can
 * still reach the top k (the candidates) get their logits recomputed in the order above, and the
 * choice and the gate weights are the same bits. Words
 * 1 and 2 of the workspace (bytes 4..11) then hold the number of tokens whose logits were all
 * recomputed because a recomputed logit missed its bound (0 on every test input), and the largest
 * share of the bound a candidate used (fp32 bits). Inputs must be finite. */
MOE_API moe_status moe_route(const moe_shape* shape, const void* x, const void* wg, const float* bias,
                     int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* The router of moe_route without a workspace, for callers that cannot allocate device memory
 * themselves -- for instance a plugin whose host process owns every device allocation through
 * its own pool and lends it no scratch, or a deployment that fixes its device memory budget at
 * start-up and forbids allocations afterwards. The pages have no counterpart of this entry point.
 * Same arguments, results and validation as moe_route, minus ws/ws_bytes; it allocates nothing
 * and calls no allocating routine. Its logits scratch is a fixed 4 MiB device array inside the
 * library (one copy per GPU that loads the library, kept until the process exits), so it serves
 * shapes with T*E <= 1,048,576 (e.g. T <= 4096 at E = 256) and rejects larger ones with
 * MOE_ERR_INVALID_ARG. Each call looks up that array's device address in the current context
 * (cudaGetSymbolAddress, which allocates nothing), so the address stays right after a
 * cudaDeviceReset; a device's first call also loads the library's device code there, so make
 * that first call before any stream capture. Every call shares the one array, so calls
 * that overlap on the GPU (different streams, or different host threads on the same device)
 * race on it; order them on one stream. Nothing in the array needs to start at zero: each call
 * overwrites the logits it reads. It records no device status. */
MOE_API moe_status moe_route_noalloc(const moe_shape* shape, const void* x, const void* wg,
                                     const float* bias, int32_t* topk_idx, float* topk_w,
                                     void* stream);

/* Hash routing ("CANN DeepSeek-V4推理优化", MoE 专家模型规格: V4's first layers pick experts by
 * hash routing, the others by learned soft routing). The page gives no hash function; here the
 * choice is a table supplied with the model, and the gate weights are the soft router's:
 *   token_ids      [T] int32 token ids in [0, vocab).
 *   tid2eid        [vocab, k] int32: row v holds the k distinct experts (in [0, E)) of token
 *                  id v.
 *   topk_idx       [T, k] int32 out: tid2eid[token_ids[t]], in the table's order.
 *   topk_w         [T, k] fp32 out: softmax over the token's E router logits, kept at those k
 *                  experts and renormalised -- equal to exp(l_j - max) / sum over the k, in
 *                  fp32, so only the k hashed logits are formed (each in moe_route's order).
 * x, wg, bias, ws as in moe_route (the status word is cleared: a layer starts here). A token id or table entry out of range is recorded as MOE_ERR_DEVICE_BOUNDS
 * (the entry is replaced by 0). Returns MOE_ERR_INVALID_ARG for vocab < 1. */
MOE_API moe_status moe_route_hash(const moe_shape* shape, const void* x, const void* wg,
                                  const float* bias, const int32_t* token_ids,
                                  const int32_t* tid2eid, int32_t vocab, int32_t* topk_idx,
                                  float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* Token -> expert permutation ("第 6 章 超節點", 6.2.6).
 *   topk_idx       [T, k] int32, each row k distinct experts in [0, E).
 *   expert_offsets [E+2] int32 out: expert e (< E) owns slots [offsets[e], offsets[e+1]);
 *                  offsets[E] = T*k starts the shared expert's segment and
 *                  offsets[E+1] = T*k + n_shared*T ends it.
 *   perm_token     [T*k] int32 out: token of each routed slot; slots are expert-major and,
 *                  within an expert, in ascending token order (a stable counting sort).
 *   inv_slot       [T*k] int32 out: inv_slot[t*k + j] = slot of token t's j-th choice.
 * The shared segment is implicit: slot T*k + t belongs to token t. Deterministic (no atomics
 * decide any order). */
MOE_API moe_status moe_permute(const moe_shape* shape, const int32_t* topk_idx, int32_t* expert_offsets,
                       int32_t* perm_token, int32_t* inv_slot, void* ws, size_t ws_bytes,
                       void* stream);

/* Per-expert SwiGLU FFN over every slot ("第 6 章 超節點", 6.2.2: Y = [SiLU(X W_g) (.) (X W_u)] W_d).
 *   x              [T, d] bf16 tokens; perm_token and expert_offsets as made by moe_permute.
 *   w13            [E+n_shared, 2f, d]: rows 0..f-1 of expert e are its gate projection, rows
 *                  f..2f-1 its up projection (one row per output feature, d contiguous).
 *   w2             [E+n_shared, d, f]: the down projection (one row per output feature).
 *                  bf16; E4M3 codes (one byte each) for MOE_W_FP8_E4M3_B128; or, for
 *                  MOE_W_MXFP4_E8M0_B32, E2M1 codes two per byte ([E+n_shared, 2f, d/2] and
 *                  [E+n_shared, d, f/2] bytes; element 2j of a row in the low nibble of byte j,
 *                  element 2j+1 in the high nibble), 32-byte aligned.
 *   s13, s2        E4M3 weights: fp32 block scales [E+n_shared, 2f/128, d/128] and
 *                  [E+n_shared, d/128, f/128] (weight = code value * scale of its 128x128
 *                  block). MXFP4 weights: E8M0 bytes [E+n_shared, 2f, d/32] and
 *                  [E+n_shared, d, f/32], one per 32 consecutive elements of a row (weight =
 *                  element value * 2^(scale - 127); "DeepSeek-V4-Pro on NVIDIA H200", 0.1.3:
 *                  FP4 expert weights; "CANN DeepSeek-V4推理优化", 量化策略: MXFP4). NULL for
 *                  bf16.
 *   y_perm         [T*k + n_shared*T, d] fp32 out: row s = expert output for slot s, i.e.
 *                  W_d^T (SiLU(W_g^T x) * (W_u^T x)) for the slot's token and expert.
 * The intermediate h = SiLU(G) * U is kept in bf16; accumulation is fp32. With MXFP4 weights
 * the tensor cores multiply the E2M1 codes as stored, so the activations (x, then h) enter the
 * products as two E4M3 terms with their own E8M0 scales per 32 elements, within 2^-8 of each
 * 32-element block's largest magnitude (about one bf16 rounding of that element).
 * Prefill-sized batches with bf16 weights (more than 32 routed tokens per expert on average)
 * run the experts with few tokens and those with many on two streams at once: `stream` and a
 * second stream the library creates on its first such call on each device (a host-side object;
 * no device memory is allocated), ordered against `stream` with events inside the call, so the
 * call still behaves as work enqueued on `stream` (also under CUDA-graph capture). */
MOE_API moe_status moe_expert_ffn(const moe_shape* shape, const void* x, const int32_t* perm_token,
                          const int32_t* expert_offsets, const void* w13, const void* s13,
                          const void* w2, const void* s2, float* y_perm, void* ws,
                          size_t ws_bytes, void* stream);

/* Combine ("第 6 章 超節點", 6.2.6 and 6.4.1: send back, restore token order, sum with the
 * routing weights).
 *   y[t] = y_perm[T*k + t] (if n_shared) + sum_j topk_w[t, j] * y_perm[inv_slot[t*k + j]],
 *   accumulated in fp32 in that order and rounded once to bf16 (nearest even).
 *   y [T, d] bf16 out. ws is used only to record device-side index errors. */
MOE_API moe_status moe_combine(const moe_shape* shape, const float* y_perm, const int32_t* inv_slot,
                       const float* topk_w, void* y, void* ws, size_t ws_bytes, void* stream);

/* The whole layer in one call: moe_route, moe_permute, moe_expert_ffn and moe_combine with the
 * same arguments and results (every output buffer above is filled), with one difference in
 * scheduling: the shared expert does not depend on the routing, so its FFN runs on a second,
 * library-owned stream (one per device, created on the first such call; no device memory is
 * allocated) while the router, the permutation and the row gather run on `stream` ("CANN
 * DeepSeek-V4推理优化", 多流并行优化: the shared and the routed experts on parallel streams). The
 * call joins both before the combine, so it behaves as work enqueued on `stream`. Calls that
 * overlap on the GPU (different streams, same device) order their shared-expert work through
 * that one second stream. The overlap is used for prefill-sized batches (more than 32 routed
 * tokens per expert on average) with n_shared = 1; otherwise the four steps run in order on
 * `stream`. y_perm [T*k + n_shared*T, d] fp32 and y [T, d] bf16 as in moe_expert_ffn and
 * moe_combine. The status word is cleared as the call starts (batches of at most 8 tokens: by
 * the call's first kernel, so that a CUDA graph of consecutive calls holds no memset node). */
MOE_API moe_status moe_forward(const moe_shape* shape, const void* x, const void* wg,
                               const float* bias, const void* w13, const void* s13,
                               const void* w2, const void* s2, int32_t* topk_idx, float* topk_w,
                               int32_t* expert_offsets, int32_t* perm_token, int32_t* inv_slot,
                               float* y_perm, void* y, void* ws, size_t ws_bytes, void* stream);

/* Reads (and clears) the first device-side error recorded in `ws` since the last check.
 * Synchronises `stream`. Returns MOE_OK, MOE_ERR_DEVICE_BOUNDS or MOE_ERR_DEVICE_TIMEOUT (or
 * MOE_ERR_CUDA if the read itself fails). */
MOE_API moe_status moe_check_device_status(void* ws, void* stream);

/* Failure-path self-test (no counterpart on the pages). Launches one kernel whose single thread
 * waits on a shared-memory mbarrier that nothing ever completes, using the same bounded-wait
 * pattern as the tensor-core pipelines but with a limit of `limit_us` microseconds
 * (1 .. 2,000,000; MOE_ERR_INVALID_ARG otherwise). When the limit passes the kernel records
 * MOE_ERR_DEVICE_TIMEOUT in the status word of `ws` (first error wins) and returns, so the
 * context stays usable; moe_check_device_status() then reports and clears it. `ws` is a
 * workspace of any shape (only its status word is touched). Asynchronous like the other calls. */
MOE_API moe_status moe_selftest_bounded_wait(void* ws, uint32_t limit_us, void* stream);

/* Phase timing for benchmarks and profilers (no counterpart on the pages).
 * moe_profile_enable(1) starts a session (and clears the previous one): from then on every
 * moe_expert_ffn call records three CUDA events on its stream -- before its gate/up kernels,
 * between them and its down kernels, and after -- and every call counts the kernels it
 * launches. Events are created by the library while a session is on (host-side objects; no
 * device memory is allocated). moe_profile_enable(0) stops recording.
 * The events are recorded as external events, so a moe_expert_ffn call captured into a CUDA
 * graph records them on every replay (moe_profile_read then reports the latest replay).
 * moe_profile_read waits for the recorded events and returns the summed device milliseconds of
 * the gate/up and down phases over the session, the number of moe_expert_ffn calls timed, and
 * the number of kernels launched by all four calls; any output pointer may be NULL. */
MOE_API moe_status moe_profile_enable(int on);
MOE_API moe_status moe_profile_read(double* ms_gate_up, double* ms_down, int64_t* ffn_calls,
                                    int64_t* kernel_launches);

/* Message for the last non-OK status returned on the calling thread (thread-local storage;
 * valid until the next call on that thread). */
MOE_API const char* moe_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
