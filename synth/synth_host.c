/*
 * Host (C, OpenMP) twin of the seeded input generator defined in
 * synth/__init__.py; same steps and constants, every fp32 operation rounded
 * on its own (build with -ffp-contract=off), so the bits equal the numpy
 * definition and the CUDA twin. Holds no arithmetic of the MoE layer.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static float fbits(uint32_t b) {
  float f;
  memcpy(&f, &b, 4);
  return f;
}

static uint32_t bitsf(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  return b;
}

static float log_f32(float u) {
  uint32_t bits = bitsf(u);
  int e = (int)(bits >> 23) - 127;
  float m = fbits((bits & 0x7FFFFFu) | 0x3F800000u);
  if (m > fbits(0x3FB504F3u)) { m = m * 0.5f; e += 1; }
  float y = (m - 1.0f) / (m + 1.0f);
  float y2 = y * y;
  float p = fbits(0x3DE38E39u);
  p = p * y2 + fbits(0x3E124925u);
  p = p * y2 + fbits(0x3E4CCCCDu);
  p = p * y2 + fbits(0x3EAAAAABu);
  p = p * y2 + 1.0f;
  float lnm = (2.0f * y) * p;
  return (float)e * fbits(0x3F317218u) + lnm;
}

static float cos2pi_f32(float u) {
  float r = (u < 0.5f) ? u : u - 1.0f;
  float a = fabsf(r);
  int neg = a > 0.25f;
  float b = neg ? 0.5f - a : a;
  int use_sin = b > 0.125f;
  float c = use_sin ? 0.25f - b : b;
  float x = c * fbits(0x40C90FDBu);
  float x2 = x * x;
  float pc = fbits(0xB493F27Eu);
  pc = pc * x2 + fbits(0x37D00D01u);
  pc = pc * x2 + fbits(0xBAB60B61u);
  pc = pc * x2 + fbits(0x3D2AAAABu);
  pc = pc * x2 + fbits(0xBF000000u);
  pc = pc * x2 + 1.0f;
  float ps = fbits(0x3638EF1Du);
  ps = ps * x2 + fbits(0xB9500D01u);
  ps = ps * x2 + fbits(0x3C088889u);
  ps = ps * x2 + fbits(0xBE2AAAABu);
  ps = ps * x2 + 1.0f;
  ps = ps * x;
  float v = use_sin ? ps : pc;
  return neg ? -v : v;
}

static float normal_at(uint64_t key, uint64_t idx, float stdv) {
  uint64_t h = mix64(key + (idx + 1ull) * 0x9E3779B97F4A7C15ull);
  float u1 = (float)((uint32_t)(h >> 41) * 2u + 1u) * 5.9604644775390625e-8f;
  float u2 = (float)((uint32_t)((h >> 17) & 0x7FFFFFull) * 2u + 1u) * 5.9604644775390625e-8f;
  float rad = sqrtf(-2.0f * log_f32(u1));
  return (rad * cos2pi_f32(u2)) * stdv;
}

void synth_normal_f32(float* out, int64_t n, int64_t index0, uint64_t seed, uint32_t stream,
                      float stdv) {
  const uint64_t key = mix64((seed << 8) | (uint64_t)(stream & 0xFFu));
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(key, (uint64_t)(index0 + i), stdv);
}

void synth_normal_bf16(uint16_t* out, int64_t n, int64_t index0, uint64_t seed, uint32_t stream,
                       float stdv) {
  const uint64_t key = mix64((seed << 8) | (uint64_t)(stream & 0xFFu));
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const uint32_t b = bitsf(normal_at(key, (uint64_t)(index0 + i), stdv));
    out[i] = (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
  }
}
