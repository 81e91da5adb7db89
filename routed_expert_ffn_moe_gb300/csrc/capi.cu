// The C ABI (include/moe.h): host-side validation, workspace carving, kernel dispatch.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"

namespace moe {

namespace {
thread_local char g_err[512] = "";

moe_status fail(moe_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
moe_status fail(moe_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return st;
}

moe_status cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status check_shape(const moe_shape* s) {
  if (!s) return fail(MOE_ERR_INVALID_ARG, "shape is NULL");
  if (s->E < 1 || s->E > 1024) return fail(MOE_ERR_INVALID_ARG, "E=%d not in [1, 1024]", s->E);
  if (s->k < 1 || s->k > s->E || s->k > 32)
    return fail(MOE_ERR_INVALID_ARG, "k=%d not in [1, min(E, 32)]", s->k);
  if (s->n_shared != 0 && s->n_shared != 1)
    return fail(MOE_ERR_INVALID_ARG, "n_shared=%d not 0 or 1", s->n_shared);
  if (s->d < 128 || s->d > 16384 || s->d % 128)
    return fail(MOE_ERR_INVALID_ARG, "d=%d not a multiple of 128 in [128, 16384]", s->d);
  if (s->f < 128 || s->f > 16384 || s->f % 128)
    return fail(MOE_ERR_INVALID_ARG, "f=%d not a multiple of 128 in [128, 16384]", s->f);
  if (s->T < 0 || (long long)s->T * (s->k + 1) > (1LL << 30))
    return fail(MOE_ERR_INVALID_ARG, "T=%d out of range (need 0 <= T, T*(k+1) <= 2^30)", s->T);
  if (s->wdtype != MOE_W_BF16 && s->wdtype != MOE_W_FP8_E4M3_B128 &&
      s->wdtype != MOE_W_MXFP4_E8M0_B32)
    return fail(MOE_ERR_INVALID_ARG, "wdtype=%d unknown", s->wdtype);
  return MOE_OK;
}

#define REQUIRE_PTR(p, align)                                                          \
  do {                                                                                  \
    if (!(p)) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", #p);                       \
    if (!aligned((p), (align)))                                                         \
      return fail(MOE_ERR_INVALID_ARG, "%s not %d-byte aligned", #p, (int)(align));     \
  } while (0)

// Expert weights and their scales: bf16 has none; E4M3 and MXFP4 need both. MXFP4 code arrays
// are read through tensor maps that want 32-byte aligned bases.
moe_status check_weights(const moe_shape* s, const void* w13, const void* s13, const void* w2,
                         const void* s2) {
  const size_t wa = s->wdtype == MOE_W_MXFP4_E8M0_B32 ? 32 : 16;
  REQUIRE_PTR(w13, wa);
  REQUIRE_PTR(w2, wa);
  if (s->wdtype == MOE_W_BF16) {
    if (s13 || s2) return fail(MOE_ERR_INVALID_ARG, "s13/s2 must be NULL for bf16 weights");
    return MOE_OK;
  }
  REQUIRE_PTR(s13, 16);
  REQUIRE_PTR(s2, 16);
  return MOE_OK;
}

moe_status check_ws(const moe_shape* s, const void* ws, size_t ws_bytes, WsLayout* L) {
  REQUIRE_PTR(ws, 256);
  *L = ws_layout(*s);
  if (ws_bytes < L->total)
    return fail(MOE_ERR_WORKSPACE, "workspace %zu bytes < %zu required", ws_bytes, L->total);
  return MOE_OK;
}

}  // namespace

// ---- profiling session ------------------------------------------------------------------
namespace {
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<PhaseEvents> g_prof_events;
int64_t g_prof_calls = 0;
std::atomic<int64_t> g_launches{0};
}  // namespace

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

PhaseEvents profile_phase_events() {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  PhaseEvents ev;
  if (!g_prof_on) return ev;
  if (cudaEventCreate(&ev.begin) != cudaSuccess || cudaEventCreate(&ev.mid) != cudaSuccess ||
      cudaEventCreate(&ev.end) != cudaSuccess)
    return PhaseEvents{};
  g_prof_events.push_back(ev);
  return ev;
}

namespace {
void destroy_events() {
  for (auto& ev : g_prof_events) {
    cudaEventDestroy(ev.begin);
    cudaEventDestroy(ev.mid);
    cudaEventDestroy(ev.end);
  }
  g_prof_events.clear();
}
}  // namespace

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_shape* shape) {
  if (check_shape(shape) != MOE_OK) return 0;
  return ws_layout(*shape).total;
}

moe_status moe_route(const moe_shape* shape, const void* x, const void* wg, const float* bias,
                     int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->T > 0) {
    REQUIRE_PTR(x, 16);
    REQUIRE_PTR(topk_idx, 16);
    REQUIRE_PTR(topk_w, 16);
  }
  REQUIRE_PTR(wg, 16);
  if (bias && !aligned(bias, 16)) return fail(MOE_ERR_INVALID_ARG, "bias not 16-byte aligned");
  WsLayout L;
  if ((st = check_ws(shape, ws, ws_bytes, &L)) != MOE_OK) return st;
  // A layer starts here: clear the device status word.
  cudaError_t e = cudaMemsetAsync(static_cast<char*>(ws) + L.status, 0, sizeof(int),
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_route status reset");
  e = launch_route(*shape, static_cast<const uint16_t*>(x),
                               static_cast<const uint16_t*>(wg), bias, topk_idx, topk_w,
                               static_cast<char*>(ws), L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_route launch");
}

moe_status moe_route_hash(const moe_shape* shape, const void* x, const void* wg, const float* bias,
                          const int32_t* token_ids, const int32_t* tid2eid, int32_t vocab,
                          int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                          void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (vocab < 1) return fail(MOE_ERR_INVALID_ARG, "vocab=%d not positive", vocab);
  if (shape->T > 0) {
    REQUIRE_PTR(x, 16);
    REQUIRE_PTR(token_ids, 16);
    REQUIRE_PTR(topk_idx, 16);
    REQUIRE_PTR(topk_w, 16);
  }
  REQUIRE_PTR(wg, 16);
  REQUIRE_PTR(tid2eid, 16);
  if (bias && !aligned(bias, 16)) return fail(MOE_ERR_INVALID_ARG, "bias not 16-byte aligned");
  WsLayout L;
  if ((st = check_ws(shape, ws, ws_bytes, &L)) != MOE_OK) return st;
  cudaError_t e = cudaMemsetAsync(static_cast<char*>(ws) + L.status, 0, sizeof(int),
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_route_hash status reset");
  e = launch_route_hash(*shape, static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(wg),
                        bias, token_ids, tid2eid, vocab, topk_idx, topk_w, static_cast<char*>(ws),
                        L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_route_hash launch");
}

moe_status moe_route_noalloc(const moe_shape* shape, const void* x, const void* wg,
                             const float* bias, int32_t* topk_idx, float* topk_w, void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->T > 0) {
    REQUIRE_PTR(x, 16);
    REQUIRE_PTR(topk_idx, 16);
    REQUIRE_PTR(topk_w, 16);
  }
  REQUIRE_PTR(wg, 16);
  if (bias && !aligned(bias, 16)) return fail(MOE_ERR_INVALID_ARG, "bias not 16-byte aligned");
  const size_t need = (size_t)shape->T * (size_t)shape->E;
  if (need > route_noalloc_max_logits())
    return fail(MOE_ERR_INVALID_ARG,
                "moe_route_noalloc: T*E = %zu logits exceed its built-in scratch of %zu fp32 "
                "values (4 MiB); use moe_route with a workspace for this shape",
                need, route_noalloc_max_logits());
  cudaError_t e = launch_route_noalloc(*shape, static_cast<const uint16_t*>(x),
                                       static_cast<const uint16_t*>(wg), bias, topk_idx, topk_w,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_route_noalloc");
}

moe_status moe_permute(const moe_shape* shape, const int32_t* topk_idx, int32_t* expert_offsets,
                       int32_t* perm_token, int32_t* inv_slot, void* ws, size_t ws_bytes,
                       void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->T > 0) {
    REQUIRE_PTR(topk_idx, 16);
    REQUIRE_PTR(perm_token, 16);
    REQUIRE_PTR(inv_slot, 16);
  }
  REQUIRE_PTR(expert_offsets, 16);
  WsLayout L;
  if ((st = check_ws(shape, ws, ws_bytes, &L)) != MOE_OK) return st;
  cudaError_t e = launch_permute(*shape, topk_idx, expert_offsets, perm_token, inv_slot,
                                 static_cast<char*>(ws), L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_permute launch");
}

moe_status moe_expert_ffn(const moe_shape* shape, const void* x, const int32_t* perm_token,
                          const int32_t* expert_offsets, const void* w13, const void* s13,
                          const void* w2, const void* s2, float* y_perm, void* ws,
                          size_t ws_bytes, void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->T > 0) {
    REQUIRE_PTR(x, 16);
    REQUIRE_PTR(perm_token, 16);
    REQUIRE_PTR(y_perm, 16);
  }
  REQUIRE_PTR(expert_offsets, 16);
  if ((st = check_weights(shape, w13, s13, w2, s2)) != MOE_OK) return st;
  WsLayout L;
  if ((st = check_ws(shape, ws, ws_bytes, &L)) != MOE_OK) return st;
  cudaError_t e = launch_expert_ffn(*shape, static_cast<const uint16_t*>(x), perm_token,
                                    expert_offsets, w13, s13, w2, s2, y_perm,
                                    static_cast<char*>(ws), L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_expert_ffn launch");
}

moe_status moe_combine(const moe_shape* shape, const float* y_perm, const int32_t* inv_slot,
                       const float* topk_w, void* y, void* ws, size_t ws_bytes, void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->T > 0) {
    REQUIRE_PTR(y_perm, 16);
    REQUIRE_PTR(inv_slot, 16);
    REQUIRE_PTR(topk_w, 16);
    REQUIRE_PTR(y, 16);
  }
  WsLayout L;
  if ((st = check_ws(shape, ws, ws_bytes, &L)) != MOE_OK) return st;
  int* status = reinterpret_cast<int*>(static_cast<char*>(ws) + L.status);
  cudaError_t e = launch_combine(*shape, y_perm, inv_slot, topk_w, static_cast<uint16_t*>(y),
                                 status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_combine launch");
}

moe_status moe_forward(const moe_shape* shape, const void* x, const void* wg, const float* bias,
                       const void* w13, const void* s13, const void* w2, const void* s2,
                       int32_t* topk_idx, float* topk_w, int32_t* expert_offsets,
                       int32_t* perm_token, int32_t* inv_slot, float* y_perm, void* y, void* ws,
                       size_t ws_bytes, void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (shape->T > 0) {
    REQUIRE_PTR(x, 16);
    REQUIRE_PTR(topk_idx, 16);
    REQUIRE_PTR(topk_w, 16);
    REQUIRE_PTR(perm_token, 16);
    REQUIRE_PTR(inv_slot, 16);
    REQUIRE_PTR(y_perm, 16);
    REQUIRE_PTR(y, 16);
  }
  REQUIRE_PTR(wg, 16);
  REQUIRE_PTR(expert_offsets, 16);
  if (bias && !aligned(bias, 16)) return fail(MOE_ERR_INVALID_ARG, "bias not 16-byte aligned");
  if ((st = check_weights(shape, w13, s13, w2, s2)) != MOE_OK) return st;
  WsLayout L;
  if ((st = check_ws(shape, ws, ws_bytes, &L)) != MOE_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (shape->T == 0) {  // no token: only the expert offsets are defined
    // A layer starts here: clear the device status word.
    e = cudaMemsetAsync(static_cast<char*>(ws) + L.status, 0, sizeof(int), cs);
    if (e != cudaSuccess) return cuda_fail(e, "moe_forward status reset");
    e = launch_permute(*shape, topk_idx, expert_offsets, perm_token, inv_slot,
                       static_cast<char*>(ws), L, cs);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_forward launch");
  }
  // launch_forward clears the status word first (with a memset, or in its first kernel)
  e = launch_forward(*shape, static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(wg),
                     bias, w13, s13, w2, s2, topk_idx, topk_w, expert_offsets, perm_token,
                     inv_slot, y_perm, static_cast<uint16_t*>(y), static_cast<char*>(ws), L, cs);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_forward launch");
}

moe_status moe_check_device_status(void* ws, void* stream) {
  REQUIRE_PTR(ws, 256);
  int code = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&code, ws, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && code != 0) e = cudaMemsetAsync(ws, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "moe_check_device_status");
  if (code == MOE_ERR_DEVICE_BOUNDS)
    return fail(MOE_ERR_DEVICE_BOUNDS, "a device-side index check failed");
  if (code == MOE_ERR_DEVICE_TIMEOUT)
    return fail(MOE_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up");
  if (code != 0) return fail(MOE_ERR_CUDA, "unknown device status %d", code);
  return MOE_OK;
}

moe_status moe_selftest_bounded_wait(void* ws, uint32_t limit_us, void* stream) {
  REQUIRE_PTR(ws, 256);
  if (limit_us < 1 || limit_us > 2000000)
    return fail(MOE_ERR_INVALID_ARG, "limit_us=%u not in [1, 2000000]", limit_us);
  cudaError_t e = launch_selftest_bounded_wait(static_cast<int*>(ws), 1000ull * limit_us,
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_selftest_bounded_wait launch");
}

moe_status moe_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (on) {
    destroy_events();
    g_prof_calls = 0;
    g_launches.store(0);
  }
  g_prof_on = on != 0;
  return MOE_OK;
}

moe_status moe_profile_read(double* ms_gate_up, double* ms_down, int64_t* ffn_calls,
                            int64_t* kernel_launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double up = 0.0, dn = 0.0;
  for (auto& ev : g_prof_events) {
    float a = 0.f, b = 0.f;
    cudaError_t e = cudaEventSynchronize(ev.end);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&a, ev.begin, ev.mid);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&b, ev.mid, ev.end);
    if (e != cudaSuccess) return cuda_fail(e, "moe_profile_read");
    up += a;
    dn += b;
  }
  if (ms_gate_up) *ms_gate_up = up;
  if (ms_down) *ms_down = dn;
  if (ffn_calls) *ffn_calls = (int64_t)g_prof_events.size();
  if (kernel_launches) *kernel_launches = g_launches.load();
  return MOE_OK;
}

const char* moe_last_error_string(void) { return g_err; }

}  // extern "C"
