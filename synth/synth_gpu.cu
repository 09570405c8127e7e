// Device twin of the seeded input generator in synth/__init__.py.
//
// Same definition, step for step: SplitMix64 counter stream -> two odd 24-bit
// uniforms -> Box-Muller with our own fp32 ln / cos polynomials, every
// operation an explicitly rounded IEEE fp32 op (__fmul_rn, __fadd_rn, ...), so
// that no multiply-add is contracted and the bits equal the numpy version.
// Holds no arithmetic of the MoE layer. Built as its own small shared library.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float fbits(uint32_t b) { return __uint_as_float(b); }

__device__ __forceinline__ float log_f32(float u) {
  uint32_t bits = __float_as_uint(u);
  int e = (int)(bits >> 23) - 127;
  float m = __uint_as_float((bits & 0x7FFFFFu) | 0x3F800000u);
  if (m > fbits(0x3FB504F3u)) { m = __fmul_rn(m, 0.5f); e += 1; }
  float y = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
  float y2 = __fmul_rn(y, y);
  float p = fbits(0x3DE38E39u);
  p = __fadd_rn(__fmul_rn(p, y2), fbits(0x3E124925u));
  p = __fadd_rn(__fmul_rn(p, y2), fbits(0x3E4CCCCDu));
  p = __fadd_rn(__fmul_rn(p, y2), fbits(0x3EAAAAABu));
  p = __fadd_rn(__fmul_rn(p, y2), 1.0f);
  float lnm = __fmul_rn(__fmul_rn(2.0f, y), p);
  return __fadd_rn(__fmul_rn((float)e, fbits(0x3F317218u)), lnm);
}

__device__ __forceinline__ float cos2pi_f32(float u) {
  float r = (u < 0.5f) ? u : __fsub_rn(u, 1.0f);
  float a = fabsf(r);
  bool neg = a > 0.25f;
  float b = neg ? __fsub_rn(0.5f, a) : a;
  bool use_sin = b > 0.125f;
  float c = use_sin ? __fsub_rn(0.25f, b) : b;
  float x = __fmul_rn(c, fbits(0x40C90FDBu));
  float x2 = __fmul_rn(x, x);
  float pc = fbits(0xB493F27Eu);
  pc = __fadd_rn(__fmul_rn(pc, x2), fbits(0x37D00D01u));
  pc = __fadd_rn(__fmul_rn(pc, x2), fbits(0xBAB60B61u));
  pc = __fadd_rn(__fmul_rn(pc, x2), fbits(0x3D2AAAABu));
  pc = __fadd_rn(__fmul_rn(pc, x2), fbits(0xBF000000u));
  pc = __fadd_rn(__fmul_rn(pc, x2), 1.0f);
  float ps = fbits(0x3638EF1Du);
  ps = __fadd_rn(__fmul_rn(ps, x2), fbits(0xB9500D01u));
  ps = __fadd_rn(__fmul_rn(ps, x2), fbits(0x3C088889u));
  ps = __fadd_rn(__fmul_rn(ps, x2), fbits(0xBE2AAAABu));
  ps = __fadd_rn(__fmul_rn(ps, x2), 1.0f);
  ps = __fmul_rn(ps, x);
  float v = use_sin ? ps : pc;
  return neg ? -v : v;
}

__device__ __forceinline__ float normal_at(uint64_t key, uint64_t idx, float stdv) {
  uint64_t h = mix64(key + (idx + 1ull) * 0x9E3779B97F4A7C15ull);
  float u1 = __fmul_rn((float)((uint32_t)(h >> 41) * 2u + 1u), 5.9604644775390625e-8f);
  float u2 = __fmul_rn((float)((uint32_t)((h >> 17) & 0x7FFFFFull) * 2u + 1u), 5.9604644775390625e-8f);
  float rad = __fsqrt_rn(__fmul_rn(-2.0f, log_f32(u1)));
  return __fmul_rn(__fmul_rn(rad, cos2pi_f32(u2)), stdv);
}

__device__ __forceinline__ uint16_t bf16_rne(float v) {
  uint32_t b = __float_as_uint(v);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

// out[(a*d1 + b)*d2 + c] = value at logical index a*s0 + b*s1 + c*s2 (any
// permutation of a 3-D tensor), written as bf16 or fp32.
__global__ void fill_kernel(void* out, int64_t d0, int64_t d1, int64_t d2, int64_t s0,
                            int64_t s1, int64_t s2, int64_t index0, uint64_t key, float stdv,
                            int as_bf16) {
  const int64_t n = d0 * d1 * d2;
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < n;
       o += (int64_t)gridDim.x * blockDim.x) {
    int64_t c = o % d2, ab = o / d2, b = ab % d1, a = ab / d1;
    float v = normal_at(key, (uint64_t)(index0 + a * s0 + b * s1 + c * s2), stdv);
    if (as_bf16) ((uint16_t*)out)[o] = bf16_rne(v);
    else ((float*)out)[o] = v;
  }
}

uint64_t host_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

}  // namespace

extern "C" {

// Fills a device buffer of d0*d1*d2 elements with generator values of
// (seed, stream). Output element (a,b,c) takes counter index
// index0 + a*s0 + b*s1 + c*s2. Returns 0, or the cudaError_t of the launch.
int synth_fill_normal(void* out, int64_t d0, int64_t d1, int64_t d2, int64_t s0, int64_t s1,
                      int64_t s2, int64_t index0, uint64_t seed, uint32_t stream, float stdv,
                      int as_bf16, cudaStream_t st) {
  const int64_t n = d0 * d1 * d2;
  if (n <= 0) return 0;
  const uint64_t key = host_mix64((seed << 8) | (uint64_t)(stream & 0xFFu));
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  fill_kernel<<<(unsigned)blocks, 256, 0, st>>>(out, d0, d1, d2, s0, s1, s2, index0, key, stdv,
                                                 as_bf16);
  return (int)cudaGetLastError();
}

}  // extern "C"
