// Seeded synthetic inputs for the routed-expert MoE FFN layer.
//
// This module is the only code shared by the CPU oracle and the CUDA layer: it draws the
// activations, router weights and expert weights, and it block-quantises expert weights to FP8
// for the FP8 workloads. It holds none of the layer's own arithmetic (no routing, no dequant, no
// GEMM, no combine).
//
// Every value is a pure function of (seed, stream, element index), written only with integer
// operations, one IEEE double multiply and IEEE fp32 divisions, so the host functions and the
// device kernels below produce bit-identical output on any machine:
//
//   * uniform bits: the SplitMix64 sequence (Steele, Lea, Flood, "Fast splittable pseudorandom
//     number generators", OOPSLA 2014): draw n of a stream keyed K is mix64(K + (n+1)*GAMMA).
//   * normal variates: Irwin-Hall with twelve 16-bit uniforms, Z = sum((u_j + 1/2)/2^16) - 6,
//     which has mean 0 and variance 1 - 2^-32 and is exact in double; value = sigma * Z,
//     rounded once to bf16 (round to nearest even).
//   * FP8 E4M3 (OCP 8-bit floating point spec, bias 7, max 448, no infinities): per 128x128
//     block of a row-major [rows, cols] matrix, s = amax/448 (s = 1 if amax = 0),
//     q = round-to-nearest-even(w / s) saturated to +-448.
//   * MXFP4 (OCP Microscaling Formats v1.0: E2M1 elements, one E8M0 scale per block of 32):
//     per 32 consecutive elements of a row, X = 2^(floor(log2 amax) - 2) (2 = the largest
//     E2M1 exponent; X = 1 if amax = 0), q = E2M1 round-to-nearest-even(w / X) saturated to
//     +-6; two codes per byte, element 2j in the low nibble; the scale byte is log2(X) + 127.
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#define SYN_HD __host__ __device__ __forceinline__

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

SYN_HD uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

SYN_HD uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed + kGamma) ^ (stream * 0xD1B54A32D192ED03ull));
}

SYN_HD uint64_t draw(uint64_t key, uint64_t n) { return mix64(key + (n + 1) * kGamma); }

// Irwin-Hall(12) standard normal for element i: uses draws 3i, 3i+1, 3i+2 (four 16-bit fields each).
SYN_HD double normal_at(uint64_t key, uint64_t i) {
  int64_t s = 0;
  for (int j = 0; j < 3; ++j) {
    const uint64_t u = draw(key, 3 * i + (uint64_t)j);
    s += (int64_t)(u & 0xFFFFu) + (int64_t)((u >> 16) & 0xFFFFu) +
         (int64_t)((u >> 32) & 0xFFFFu) + (int64_t)(u >> 48);
  }
  // sum((u_j + 0.5) / 65536) - 6 == (s + 6 - 6 * 65536) / 65536, exact in double.
  return (double)(s - 393210) * (1.0 / 65536.0);
}

SYN_HD uint64_t dbits(double v) { uint64_t b; memcpy(&b, &v, 8); return b; }
SYN_HD uint32_t fbits(float v) { uint32_t b; memcpy(&b, &v, 4); return b; }
SYN_HD float bf16_to_f32(uint16_t h) { uint32_t b = (uint32_t)h << 16; float f; memcpy(&f, &b, 4); return f; }

// double -> bf16, round to nearest even, with bf16 subnormals; overflow -> inf.
SYN_HD uint16_t double_to_bf16(double v) {
  const uint64_t b = dbits(v);
  const uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
  const int ex = (int)((b >> 52) & 0x7FF);
  const uint64_t man = b & ((1ull << 52) - 1);
  if (ex == 0x7FF) return (uint16_t)(sign | (man ? 0x7FC0u : 0x7F80u));
  if (ex == 0) return sign;  // zero or a double subnormal (far below bf16's range)
  const int e = ex - 1023;
  const uint64_t sig = (1ull << 52) | man;
  const int shift = (e >= -126) ? 45 : (-81 - e);
  if (shift >= 60) return sign;
  uint64_t keep = sig >> shift;
  const uint64_t rem = sig & ((1ull << shift) - 1);
  const uint64_t half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (keep & 1))) keep += 1;
  if (e >= -126) {
    int be = e + 127;
    if (keep == 256) { keep = 128; be += 1; }
    if (be >= 255) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (be << 7) | (keep & 0x7F));
  }
  return (uint16_t)(sign | keep);  // keep == 128 becomes the smallest normal
}

// fp32 -> E4M3, round to nearest even, saturating finite values to +-448; NaN -> 0x7F.
SYN_HD uint8_t f32_to_e4m3(float v) {
  const uint32_t b = fbits(v);
  const uint8_t sign = (uint8_t)((b >> 24) & 0x80u);
  const uint32_t a = b & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint8_t)(sign | 0x7F);
  if (a == 0x7F800000u) return (uint8_t)(sign | 0x7E);
  const int ex = (int)(a >> 23);
  if (ex == 0) return sign;
  const int e = ex - 127;
  const uint32_t sig = (1u << 23) | (a & 0x7FFFFFu);
  const int shift = (e >= -6) ? 20 : (14 - e);
  if (shift >= 25) return sign;
  uint32_t keep = sig >> shift;
  const uint32_t rem = sig & ((1u << shift) - 1);
  const uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (keep & 1))) keep += 1;
  if (e >= -6) {
    int E = e + 7;
    if (keep == 16) { keep = 8; E += 1; }
    uint32_t code = ((uint32_t)E << 3) | (keep & 7);
    if (E > 15 || code > 0x7E) code = 0x7E;
    return (uint8_t)(sign | code);
  }
  return (uint8_t)(sign | keep);  // keep == 8 becomes the smallest normal
}

// fp32 -> E2M1 (sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0; magnitudes 0, 0.5,
// 1, 1.5, 2, 3, 4, 6), round to nearest with ties to the even code, saturating to +-6.
SYN_HD uint8_t f32_to_e2m1(float v) {
  const uint8_t sign = (uint8_t)((fbits(v) >> 28) & 0x8u);
  const float a = v < 0.f ? -v : v;
  uint8_t m;
  if (a <= 0.25f) m = 0;
  else if (a < 0.75f) m = 1;
  else if (a <= 1.25f) m = 2;
  else if (a < 1.75f) m = 3;
  else if (a <= 2.5f) m = 4;
  else if (a < 3.5f) m = 5;
  else if (a <= 5.0f) m = 6;
  else m = 7;  // above 5, and NaN (which the generator never draws)
  return (uint8_t)(sign | m);
}

// One block of 32 bf16 weights -> 16 bytes of E2M1 codes and its E8M0 scale byte.
SYN_HD void mxfp4_block(const uint16_t* w, uint8_t* q, uint8_t* s) {
  float amax = 0.f;
  for (int i = 0; i < 32; ++i) {
    const float a = bf16_to_f32((uint16_t)(w[i] & 0x7FFFu));
    amax = a > amax ? a : amax;
  }
  int e = 127;
  if (amax > 0.f) {
    e = (int)((fbits(amax) >> 23) & 0xFFu) - 2;  // floor(log2 amax) - 2, biased by 127
    if (e < 0) e = 0;
  }
  uint32_t xb = e >= 1 ? (uint32_t)e << 23 : 0x00400000u;  // X = 2^(e - 127) as fp32
  float X;
  memcpy(&X, &xb, 4);
  for (int i = 0; i < 16; ++i) {
    const uint8_t lo = f32_to_e2m1(bf16_to_f32(w[2 * i]) / X);
    const uint8_t hi = f32_to_e2m1(bf16_to_f32(w[2 * i + 1]) / X);
    q[i] = (uint8_t)(lo | (hi << 4));
  }
  *s = (uint8_t)e;
}

__global__ void quant_mxfp4_kernel(const uint16_t* w, uint8_t* q, uint8_t* s, int64_t nblk) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += stride)
    mxfp4_block(w + b * 32, q + b * 16, s + b);
}

__global__ void normal_bf16_kernel(uint16_t* out, uint64_t n, uint64_t key, double sigma,
                                   uint64_t offset) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = double_to_bf16(__dmul_rn(sigma, normal_at(key, offset + i)));
}

// One CTA per 128x128 block.
__global__ void quant_e4m3_kernel(const uint16_t* w, uint8_t* q, float* s, int64_t rows,
                                  int64_t cols) {
  const int64_t nbc = cols / 128;
  const int64_t rb = blockIdx.x / nbc, cb = blockIdx.x % nbc;
  __shared__ float red[256];
  float amax = 0.f;
  for (int i = threadIdx.x; i < 128 * 128; i += blockDim.x) {
    const int64_t r = rb * 128 + i / 128, c = cb * 128 + i % 128;
    const float a = fabsf(bf16_to_f32(w[r * cols + c]));
    amax = a > amax ? a : amax;
  }
  red[threadIdx.x] = amax;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + o]);
    __syncthreads();
  }
  amax = red[0];
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (threadIdx.x == 0) s[rb * nbc + cb] = sc;
  for (int i = threadIdx.x; i < 128 * 128; i += blockDim.x) {
    const int64_t r = rb * 128 + i / 128, c = cb * 128 + i % 128;
    q[r * cols + c] = f32_to_e4m3(__fdiv_rn(bf16_to_f32(w[r * cols + c]), sc));
  }
}

}  // namespace

extern "C" {

uint64_t synth_key(uint64_t seed, uint64_t stream) { return stream_key(seed, stream); }

void synth_normal_bf16_host(uint16_t* out, uint64_t n, uint64_t key, double sigma,
                            uint64_t offset) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = double_to_bf16(sigma * normal_at(key, offset + (uint64_t)i));
}

int synth_normal_bf16_device(uint16_t* out, uint64_t n, uint64_t key, double sigma,
                             uint64_t offset, void* stream) {
  if (n == 0) return 0;
  uint64_t blocks = (n + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  normal_bf16_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, n, key, sigma,
                                                                          offset);
  return (int)cudaGetLastError();
}

void synth_quant_e4m3_host(const uint16_t* w, uint8_t* q, float* s, int64_t rows,
                           int64_t cols) {
  const int64_t nbr = rows / 128, nbc = cols / 128;
#pragma omp parallel for schedule(static)
  for (int64_t blk = 0; blk < nbr * nbc; ++blk) {
    const int64_t rb = blk / nbc, cb = blk % nbc;
    float amax = 0.f;
    for (int64_t r = rb * 128; r < rb * 128 + 128; ++r)
      for (int64_t c = cb * 128; c < cb * 128 + 128; ++c) {
        const float a = bf16_to_f32((uint16_t)(w[r * cols + c] & 0x7FFFu));
        amax = a > amax ? a : amax;
      }
    const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
    s[rb * nbc + cb] = sc;
    for (int64_t r = rb * 128; r < rb * 128 + 128; ++r)
      for (int64_t c = cb * 128; c < cb * 128 + 128; ++c)
        q[r * cols + c] = f32_to_e4m3(bf16_to_f32(w[r * cols + c]) / sc);
  }
}

int synth_quant_e4m3_device(const uint16_t* w, uint8_t* q, float* s, int64_t rows, int64_t cols,
                            void* stream) {
  if (rows % 128 || cols % 128) return 1;
  const int64_t nblk = (rows / 128) * (cols / 128);
  if (nblk == 0) return 0;
  if (nblk > 0x7FFFFFFF) return 1;
  quant_e4m3_kernel<<<(unsigned)nblk, 256, 0, (cudaStream_t)stream>>>(w, q, s, rows, cols);
  return (int)cudaGetLastError();
}

// Row-major [rows, cols] bf16 -> q [rows, cols/2] E2M1 code pairs and s [rows, cols/32] E8M0.
// The blocks of a row are consecutive, so block b covers elements 32b .. 32b+31 of the matrix.
void synth_quant_mxfp4_host(const uint16_t* w, uint8_t* q, uint8_t* s, int64_t rows,
                            int64_t cols) {
  const int64_t nblk = rows * (cols / 32);
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblk; ++b) mxfp4_block(w + b * 32, q + b * 16, s + b);
}

int synth_quant_mxfp4_device(const uint16_t* w, uint8_t* q, uint8_t* s, int64_t rows,
                             int64_t cols, void* stream) {
  if (cols % 32) return 1;
  const int64_t nblk = rows * (cols / 32);
  if (nblk == 0) return 0;
  int64_t blocks = (nblk + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  quant_mxfp4_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(w, q, s, nblk);
  return (int)cudaGetLastError();
}

void synth_f32_to_e2m1_host(const float* v, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_e2m1(v[i]);
}

void synth_double_to_bf16_host(const double* v, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(v[i]);
}

void synth_f32_to_e4m3_host(const float* v, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_e4m3(v[i]);
}

}  // extern "C"
