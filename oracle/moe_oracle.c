/*
 * CPU oracle for the routed-expert MoE FFN layer -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct restatement of what the layer computes. Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product path never does.
 * It shares no code with the CUDA library.
 *
 * Arithmetic: fp64 throughout, except the router logits, which are the fp32 values whose order
 * decides the integer top-k choice and are therefore formed in a fixed fp32 order (below).
 *
 * Passages followed (page title, section):
 *   - router scores every routed expert for a token, keeps the top-k, shared expert always on:
 *     "DeepSeek-V4-Pro on NVIDIA H200", 0.1.2 (MoE) and 0.2.2 step D4;
 *     "CANN DeepSeek-V4推理优化", MoE 专家模型规格 ("soft routing").
 *   - reorder rows by expert, multiply, restore token order; combine = routing-weighted sum
 *     a1*y1 + a6*y6 of the experts' outputs: "第 6 章 超節點", 6.2.6 and 6.4.1.
 *   - expert FFN Y = [SiLU(X W_g) (.) (X W_u)] W_d: "第 6 章 超節點", 6.2.2.
 *   - three GEMMs per expert (up, down, gate): "DeepSeek V3/R1 Inference Efficiency (1)",
 *     Parameters.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - gate: softmax over all E logits (fp64), keep the k largest logits (ties -> lower expert
 *     index), renormalise the k kept probabilities to sum to 1. Selection compares the fp32
 *     logits, not the probabilities.
 *   - logit l[t,e] is formed in fp32 in a fixed order: with d split into 8-element chunks,
 *     lane j (0..31) accumulates chunks j, j+32, j+64, ... element by element with fused
 *     multiply-add starting from +0; then the 32 lane sums are combined by an xor butterfly
 *     (partner offsets 16, 8, 4, 2, 1, plain fp32 add); then + bias[e] if a bias is given.
 *   - topk_idx lists the chosen experts by descending logit, ties by ascending index.
 *   - hash routing ("CANN DeepSeek-V4推理优化", MoE 专家模型规格: V4's first layers choose
 *     experts by hash routing, the others by learned soft routing; the page defines no hash):
 *     a token's k experts are a fixed function of its token id, given as a table
 *     tid2eid[vocab][k] of distinct experts and listed in the table's order; the gate weights
 *     are the soft router's gate at those experts (softmax over all E, keep the k, renormalise).
 *   - slots: expert-major, ascending token within an expert; the shared expert's segment
 *     follows the routed ones, in token order; shared weight 1; no routed scaling factor.
 *   - FP8 E4M3 expert weights with one fp32 scale per 128x128 block: weight = code value * s.
 *   - FP4 expert weights ("DeepSeek-V4-Pro on NVIDIA H200", 0.1.3: V4-Pro's MoE experts are
 *     stored in FP4; "CANN DeepSeek-V4推理优化", 量化策略: the MoE module quantised to MXFP4)
 *     in the MXFP4 format of the OCP Microscaling Formats spec v1.0: E2M1 elements, one E8M0
 *     scale per 32 consecutive elements of a row; weight = element value * 2^(e - 127). The
 *     pages name the format but not its byte layout: two codes per byte, element 2j in the low
 *     nibble; scales row-major [rows, cols/32].
 *
 * Parity of this file is pinned by tests against the pages' worked example, closed forms,
 * library-routine reductions, brute force and invariants; see tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define WD_BF16 0
#define WD_FP8 1
#define WD_MXFP4 2

/* ---- number formats ----------------------------------------------------------------------- */

/* bf16: sign, 8 exponent bits (bias 127), 7 fraction bits -- the upper half of an IEEE fp32. */
double oracle_bf16_value(uint16_t h) {
  uint32_t b = (uint32_t)h << 16;
  float f;
  memcpy(&f, &b, sizeof f);
  return (double)f;
}

static float bf16f(uint16_t h) { return (float)oracle_bf16_value(h); }

/* OCP FP8 E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is
 * subnormal (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities. */
double oracle_e4m3_value(uint8_t q) {
  int s = (q >> 7) & 1, E = (q >> 3) & 15, m = q & 7;
  double v;
  if (E == 15 && m == 7) return NAN;
  if (E == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, E - 7);
  return s ? -v : v;
}

/* OCP MX FP4 E2M1: sign (bit 3), 2 exponent bits (bias 1), 1 mantissa bit; exponent field 0 is
 * subnormal (m * 0.5); no infinities or NaN. Magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_value(uint8_t code) {
  int s = (code >> 3) & 1, E = (code >> 1) & 3, m = code & 1;
  double v = E == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, E - 1);
  return s ? -v : v;
}

/* OCP MX E8M0 shared scale: 2^(e - 127); 0xFF is NaN. */
double oracle_e8m0_value(uint8_t e) { return e == 0xFF ? NAN : ldexp(1.0, (int)e - 127); }

/* Weight w[r][c] of a row-major [rows, cols] matrix stored as bf16; as E4M3 codes with fp32
 * scales s[r/128][c/128]; or as MXFP4 code pairs w[r][c/2] (element c in the low nibble when c
 * is even) with E8M0 scales s[r][c/32]. */
static double weight(int wdtype, const void* w, const void* s, int64_t cols, int64_t r,
                     int64_t c) {
  if (wdtype == WD_BF16) return oracle_bf16_value(((const uint16_t*)w)[r * cols + c]);
  if (wdtype == WD_MXFP4) {
    const uint8_t pair = ((const uint8_t*)w)[r * (cols / 2) + c / 2];
    const uint8_t code = (uint8_t)((c & 1) ? pair >> 4 : pair & 15);
    return oracle_e2m1_value(code) *
           oracle_e8m0_value(((const uint8_t*)s)[r * (cols / 32) + c / 32]);
  }
  return oracle_e4m3_value(((const uint8_t*)w)[r * cols + c]) *
         (double)((const float*)s)[(r / 128) * (cols / 128) + (c / 128)];
}

/* ---- a1: router ---------------------------------------------------------------------------- */

/* logits [T, E] fp32 in the fixed order described in the header. Requires d % 8 == 0. */
void oracle_router_logits(const uint16_t* x, const uint16_t* wg, const float* bias, int T, int d,
                          int E, float* logits) {
  const int chunks = d / 8;
#pragma omp parallel for schedule(dynamic)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      const uint16_t* xr = x + (int64_t)t * d;
      const uint16_t* wr = wg + (int64_t)e * d;
      float lane[32], next[32];
      for (int j = 0; j < 32; ++j) {
        float acc = 0.0f;
        for (int c = j; c < chunks; c += 32)
          for (int i = 8 * c; i < 8 * c + 8; ++i) acc = fmaf(bf16f(xr[i]), bf16f(wr[i]), acc);
        lane[j] = acc;
      }
      for (int off = 16; off >= 1; off /= 2) {
        for (int j = 0; j < 32; ++j) next[j] = lane[j] + lane[j ^ off];
        memcpy(lane, next, sizeof lane);
      }
      logits[(int64_t)t * E + e] = bias ? lane[0] + bias[e] : lane[0];
    }
  }
}

typedef struct { float l; int e; } scored;

static int by_logit_desc(const void* a, const void* b) {
  const scored* p = (const scored*)a;
  const scored* q = (const scored*)b;
  if (p->l > q->l) return -1;
  if (p->l < q->l) return 1;
  return (p->e > q->e) - (p->e < q->e);
}

/* Top-k selection and gate weights for every token. topk_w gets the fp32-rounded weights,
 * topk_w64 (nullable) the fp64 ones. */
void oracle_route(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w,
                  double* topk_w64) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    scored* order = (scored*)malloc(sizeof(scored) * (size_t)E);
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double lmax = -INFINITY, z = 0.0, zsel = 0.0;
    for (int e = 0; e < E; ++e) {
      order[e].l = l[e];
      order[e].e = e;
      if ((double)l[e] > lmax) lmax = (double)l[e];
    }
    qsort(order, (size_t)E, sizeof(scored), by_logit_desc);
    for (int e = 0; e < E; ++e) z += (p[e] = exp((double)l[e] - lmax));
    for (int e = 0; e < E; ++e) p[e] /= z;               /* softmax over all E */
    for (int j = 0; j < k; ++j) zsel += p[order[j].e];
    for (int j = 0; j < k; ++j) {
      const double g = p[order[j].e] / zsel;             /* renormalised over the chosen k */
      topk_idx[(int64_t)t * k + j] = order[j].e;
      topk_w[(int64_t)t * k + j] = (float)g;
      if (topk_w64) topk_w64[(int64_t)t * k + j] = g;
    }
    free(order);
    free(p);
  }
}

/* Hash routing: topk_idx[t] = tid2eid[token_ids[t]] (k entries, in the table's order);
 * topk_w[t, j] = p[e_j] / sum_j' p[e_j'] with p = softmax over all E of the token's logits
 * (fp64), i.e. the soft router's renormalised gate at the hashed experts. */
void oracle_route_hash(const float* logits, const int32_t* token_ids, const int32_t* tid2eid,
                       int T, int E, int k, int32_t* topk_idx, float* topk_w, double* topk_w64) {
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    const int32_t* row = tid2eid + (int64_t)token_ids[t] * k;
    double lmax = -INFINITY, z = 0.0, zsel = 0.0;
    for (int e = 0; e < E; ++e)
      if ((double)l[e] > lmax) lmax = (double)l[e];
    for (int e = 0; e < E; ++e) z += exp((double)l[e] - lmax);
    for (int j = 0; j < k; ++j) zsel += exp((double)l[row[j]] - lmax) / z;
    for (int j = 0; j < k; ++j) {
      const double g = exp((double)l[row[j]] - lmax) / z / zsel;
      topk_idx[(int64_t)t * k + j] = row[j];
      topk_w[(int64_t)t * k + j] = (float)g;
      if (topk_w64) topk_w64[(int64_t)t * k + j] = g;
    }
  }
}

/* ---- a2: permutation ----------------------------------------------------------------------- */

/* Counting sort of the T*k (token, choice) pairs by expert, stable in token order.
 * offsets[E+2]: offsets[e] = first slot of expert e (e < E), offsets[E] = T*k = first slot of the
 * shared segment, offsets[E+1] = T*k + n_shared*T. perm_token[slot] = token of that slot;
 * inv_slot[t*k + j] = slot holding choice j of token t. */
void oracle_permute(const int32_t* topk_idx, int T, int E, int k, int n_shared, int32_t* offsets,
                    int32_t* perm_token, int32_t* inv_slot) {
  int64_t* count = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  for (int64_t i = 0; i < (int64_t)T * k; ++i) count[topk_idx[i]] += 1;
  int64_t run = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = (int32_t)run;
    run += count[e];
  }
  offsets[E] = (int32_t)run;
  offsets[E + 1] = (int32_t)(run + (int64_t)n_shared * T);
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      const int e = topk_idx[(int64_t)t * k + j];
      const int64_t slot = offsets[e] + fill[e]++;
      perm_token[slot] = t;
      inv_slot[(int64_t)t * k + j] = (int32_t)slot;
    }
  free(count);
  free(fill);
}

/* ---- a3 + a4: one expert's SwiGLU FFN -------------------------------------------------------- */

/* y[r] = sum_c W[row0 + r][c] * x[c] for r < nrows, over a row-major weight with `cols`
 * columns, in fp64 (the matrix-vector product that each of the gate, up and down projections
 * is). */
void oracle_matvec(int wdtype, const void* w, const void* s, int64_t cols, int64_t row0,
                   int64_t nrows, const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    double acc = 0.0;
    for (int64_t c = 0; c < cols; ++c) acc += weight(wdtype, w, s, cols, row0 + r, c) * x[c];
    y[r] = acc;
  }
}

/* Expert FFN on n input rows xrows [n, d] (bf16):
 *   G = x W_g^T, U = x W_u^T (w13 rows 0..f-1 are gate, f..2f-1 are up), h = SiLU(G) * U with
 *   SiLU(z) = z / (1 + e^-z), y = h W_d^T (w2 is [d, f]).  y [n, d] fp64; h_out [n, f] nullable. */
void oracle_expert_rows(const uint16_t* xrows, int n, int d, int f, int wdtype, const void* w13,
                        const void* s13, const void* w2, const void* s2, double* y,
                        double* h_out) {
  for (int i = 0; i < n; ++i) {
    double* xv = (double*)malloc(sizeof(double) * (size_t)d);
    double* g = (double*)malloc(sizeof(double) * (size_t)f);
    double* u = (double*)malloc(sizeof(double) * (size_t)f);
    for (int c = 0; c < d; ++c) xv[c] = oracle_bf16_value(xrows[(int64_t)i * d + c]);
    oracle_matvec(wdtype, w13, s13, d, 0, f, xv, g);   /* gate rows 0..f-1 */
    oracle_matvec(wdtype, w13, s13, d, f, f, xv, u);   /* up rows f..2f-1 */
    for (int r = 0; r < f; ++r) {
      const double silu = g[r] / (1.0 + exp(-g[r]));
      g[r] = silu * u[r];                                   /* h */
      if (h_out) h_out[(int64_t)i * f + r] = g[r];
    }
    oracle_matvec(wdtype, w2, s2, f, 0, d, g, y + (int64_t)i * d);
    free(xv);
    free(g);
    free(u);
  }
}

/* ---- a5: combine --------------------------------------------------------------------------- */

/* y[t] = (shared row of t) + sum_j g[t,j] * y_perm[inv_slot[t,j]], fp64. */
void oracle_combine(const double* y_perm, const int32_t* inv_slot, const double* topk_w, int T,
                    int k, int d, int n_shared, double* y) {
  for (int t = 0; t < T; ++t) {
    double* out = y + (int64_t)t * d;
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    if (n_shared)
      for (int c = 0; c < d; ++c) out[c] += y_perm[((int64_t)T * k + t) * d + c];
    for (int j = 0; j < k; ++j) {
      const double g = topk_w[(int64_t)t * k + j];
      const double* row = y_perm + (int64_t)inv_slot[(int64_t)t * k + j] * d;
      for (int c = 0; c < d; ++c) out[c] += g * row[c];
    }
  }
}

/* ---- the whole layer (small shapes) --------------------------------------------------------- */

/* Runs a1..a5. Expert weights are the contiguous [E+n_shared] stacks as stored on the device.
 * Outputs: logits [T,E], topk_idx [T,k], topk_w [T,k] (fp32) and topk_w64 (fp64), offsets
 * [E+2], perm_token [T*k], inv_slot [T*k], y_perm [T*k + n_shared*T, d] and y [T, d] (fp64). */
void oracle_moe_layer(int T, int d, int E, int k, int f, int n_shared, int wdtype,
                      const uint16_t* x, const uint16_t* wg, const float* bias, const void* w13,
                      const void* s13, const void* w2, const void* s2, float* logits,
                      int32_t* topk_idx, float* topk_w, double* topk_w64, int32_t* offsets,
                      int32_t* perm_token, int32_t* inv_slot, double* y_perm, double* y) {
  const int64_t n13 = 2LL * f * d, n2 = (int64_t)d * f;
  /* bytes of one expert's weights and scales in the stacked arrays */
  const int64_t b13 = wdtype == WD_BF16 ? 2 * n13 : wdtype == WD_FP8 ? n13 : n13 / 2;
  const int64_t b2 = wdtype == WD_BF16 ? 2 * n2 : wdtype == WD_FP8 ? n2 : n2 / 2;
  const int64_t bs13 = wdtype == WD_FP8 ? 4 * (n13 / (128 * 128)) : n13 / 32;
  const int64_t bs2 = wdtype == WD_FP8 ? 4 * (n2 / (128 * 128)) : n2 / 32;
  const int64_t slots = (int64_t)T * k + (int64_t)n_shared * T;
  uint16_t* xrow = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)d);
  oracle_router_logits(x, wg, bias, T, d, E, logits);
  oracle_route(logits, T, E, k, topk_idx, topk_w, topk_w64);
  oracle_permute(topk_idx, T, E, k, n_shared, offsets, perm_token, inv_slot);
  for (int64_t slot = 0; slot < slots; ++slot) {
    int e, t;
    if (slot < (int64_t)T * k) {
      e = 0;
      while (offsets[e + 1] <= slot) ++e;   /* the expert whose segment holds this slot */
      t = perm_token[slot];
    } else {
      e = E;
      t = (int)(slot - (int64_t)T * k);
    }
    memcpy(xrow, x + (int64_t)t * d, sizeof(uint16_t) * (size_t)d);
    oracle_expert_rows(xrow, 1, d, f, wdtype, (const char*)w13 + e * b13,
                       s13 ? (const char*)s13 + e * bs13 : NULL, (const char*)w2 + e * b2,
                       s2 ? (const char*)s2 + e * bs2 : NULL, y_perm + slot * d, NULL);
  }
  oracle_combine(y_perm, inv_slot, topk_w64, T, k, d, n_shared, y);
  free(xrow);
}
