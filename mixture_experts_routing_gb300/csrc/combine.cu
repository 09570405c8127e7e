// Contention-free gather-combine and the one-time weight packing transposes.
//
// Combine: "Permute-Free Grouped GEMM for MoE (bf16, gfx950)", section 2 Core
// idea and section 5 (route_gather_combine): each output token pulls its own
// routes through the token_routes inverse map and reduces them in registers,
// instead of expert outputs being scattered with atomics. One CTA per token
// row; 16-byte vector loads and stores; fp32 accumulation in k order.
#include <cuda_fp8.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 128;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  // round-to-nearest-even; values are finite
  uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  ua = (ua + 0x7FFFu + ((ua >> 16) & 1u)) >> 16;
  ub = (ub + 0x7FFFu + ((ub >> 16) & 1u)) >> 16;
  return ua | (ub << 16);
}

template <int KMAX>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const uint16_t* __restrict__ o, const int32_t* __restrict__ token_routes,
    const float* __restrict__ topk_p, uint16_t* __restrict__ y, int N,
    const int32_t* __restrict__ n_dev, int H, int K) {
  griddep_wait();  // launched after the kernel that writes this one's inputs
  griddep_launch_dependents();
  const int t = blockIdx.x;
  if (n_dev && t >= *n_dev) {  // a token past the live count: zero row
    for (int v = threadIdx.x; v < H / 8; v += kCombineThreads)
      reinterpret_cast<uint4*>(y + (size_t)t * H)[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  int slot[KMAX];
  float w[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    slot[k] = (k < K) ? token_routes[(size_t)t * K + k] : -1;
    w[k] = (k < K) ? (topk_p ? topk_p[(size_t)t * K + k] : 1.0f) : 0.0f;  // null: unit weights
  }
  const int nv = H / 8;
  for (int v = threadIdx.x; v < nv; v += kCombineThreads) {
    uint4 in[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (slot[k] >= 0) in[k] = __ldg(reinterpret_cast<const uint4*>(o + (size_t)slot[k] * H) + v);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (slot[k] < 0) continue;
      float f[8];
      bf16x8_to_f32(in[k], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(w[k], f[i], acc[i]);
    }
    uint4 out;
    out.x = pack_bf16x2(acc[0], acc[1]);
    out.y = pack_bf16x2(acc[2], acc[3]);
    out.z = pack_bf16x2(acc[4], acc[5]);
    out.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(y + (size_t)t * H)[v] = out;
  }
}

// Backward of the combine ("Permute-Free Grouped GEMM for MoE (bf16, gfx950)",
// section 3: FC1's input gradient is reduced per token by the same
// gather-combine): dX[t] = sum_k dXr[token_routes[t,k]] with unit weights, the
// routing probability having been applied inside the FC2 dgrad. Threads
// 0..K-1 also reduce dprob[t,k] from the slot's per-32-feature partials.
template <int KMAX>
__global__ void __launch_bounds__(kCombineThreads) combine_bwd_kernel(
    const uint16_t* __restrict__ dxr, const float* __restrict__ part, int n_part,
    const int32_t* __restrict__ token_routes, uint16_t* __restrict__ dx,
    float* __restrict__ dprob, int N, int H, int K) {
  const int t = blockIdx.x;
  int slot[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) slot[k] = (k < K) ? token_routes[(size_t)t * K + k] : -1;
  if (threadIdx.x < K) {
    const int sl = token_routes[(size_t)t * K + threadIdx.x];
    float acc = 0.0f;
    if (sl >= 0)
      for (int j = 0; j < n_part; ++j) acc += part[(size_t)sl * n_part + j];
    dprob[(size_t)t * K + threadIdx.x] = acc;
  }
  const int nv = H / 8;
  for (int v = threadIdx.x; v < nv; v += kCombineThreads) {
    uint4 in[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (slot[k] >= 0) in[k] = __ldg(reinterpret_cast<const uint4*>(dxr + (size_t)slot[k] * H) + v);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (slot[k] < 0) continue;
      float f[8];
      bf16x8_to_f32(in[k], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
    uint4 out;
    out.x = pack_bf16x2(acc[0], acc[1]);
    out.y = pack_bf16x2(acc[2], acc[3]);
    out.z = pack_bf16x2(acc[4], acc[5]);
    out.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(dx + (size_t)t * H)[v] = out;
  }
}

// Row-wise FP8 (E4M3) quantisation of a bf16 matrix, one warp per row:
// scale = max|v| / 448 (1 for an all-zero row, so it encodes to zeros), then
// q = E4M3(v / scale) rounded to nearest even with saturation at +-448 (the
// division in fp32). The max is exact in any order, so codes and scales are
// reproducible.
constexpr int kQuantWarps = 8;

// The quotient v / s that the codes encode. A row whose scale s lies in
// [2^-100, FLT_MAX] takes y = RN(1/s) once and, per value, q = RN(v y), the
// exact residual r = v - s q (one fma) and RN(q + r y): Markstein's division
// step (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990), which gives the
// correctly rounded quotient when nothing underflows. An exhaustive check over
// the quantiser's whole domain in that range (every bf16 row maximum amax with
// s = RN(amax/448), every bf16 value up to it; tests/test_quantize_division.py)
// finds it equal to RN(v/s) wherever |v/s| >= 2^-12 and of the same sign
// below that, where both encode as a zero code. Other rows divide directly.
struct RowDivisor {
  float s, y;
  bool fast;
};

__device__ __forceinline__ RowDivisor row_divisor(float s) {
  RowDivisor d;
  d.s = s;
  d.fast = s >= 0x1p-100f && s <= 3.40282347e38f;
  d.y = d.fast ? __frcp_rn(s) : 0.0f;
  return d;
}

__device__ __forceinline__ float row_div(float v, const RowDivisor& d) {
  if (!d.fast) return __fdiv_rn(v, d.s);
  const float q = __fmul_rn(v, d.y);
  const float r = __fmaf_rn(-d.s, q, v);
  // the quotient has v's sign; the sign restores it for v = -0, where the
  // residual sum gives +0
  return copysignf(__fmaf_rn(r, d.y, q), v);
}

// Eight bf16 values (one 16-byte group) to eight E4M3 codes, lowest first.
__device__ __forceinline__ uint2 quantize8_e4m3(const uint4 w, const RowDivisor& d) {
  const uint32_t a[4] = {w.x, w.y, w.z, w.w};
  uint32_t packed[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = row_div(__uint_as_float(a[i] << 16), d);
    const float hi = row_div(__uint_as_float(a[i] & 0xFFFF0000u), d);
    const uint32_t pair =
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);  // lo: low byte
    if (i & 1)
      packed[i >> 1] |= pair << 16;
    else
      packed[i >> 1] = pair;
  }
  return make_uint2(packed[0], packed[1]);
}

__global__ void __launch_bounds__(kQuantWarps * 32) quantize_rows_fp8_kernel(
    const uint16_t* __restrict__ m, int64_t rows, const int32_t* __restrict__ rows_dev, int cols,
    uint8_t* __restrict__ q, float* __restrict__ scale) {
  griddep_wait();  // launched after the kernel that writes this one's inputs
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kQuantWarps + warp;
  if (rows_dev && r >= (int64_t)*rows_dev) return;  // rows past the live extent
  if (r >= rows) return;
  const uint16_t* row = m + (size_t)r * cols;
  const int nv = cols / 8;  // 16-byte groups of 8 values (cols is a multiple of 8)
  float amax = 0.0f;
  for (int v = lane; v < nv; v += 32) {
    const uint4 w = reinterpret_cast<const uint4*>(row)[v];
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      amax = fmaxf(amax, fabsf(__uint_as_float(a[i] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(a[i] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (lane == 0) scale[r] = s;
  uint8_t* qr = q + (size_t)r * cols;
  const RowDivisor dv = row_divisor(s);
  for (int v = lane; v < nv; v += 32)
    reinterpret_cast<uint2*>(qr)[v] = quantize8_e4m3(reinterpret_cast<const uint4*>(row)[v], dv);
}

// The same quantisation with the whole row held in registers: WPR warps per
// row, and lane l of the row's warps loads 16-byte groups l, l + 32*WPR, ...
// (at most NV of them, all issued before any is used), so each row is read
// from memory once. The row's warps combine their maxima through shared
// memory; warps of rows past the bound skip the work but reach the barrier.
template <int NV, int WPR>
__global__ void __launch_bounds__(kQuantWarps * 32) quantize_rows_fp8_reg_kernel(
    const uint16_t* __restrict__ m, int64_t rows, const int32_t* __restrict__ rows_dev, int cols,
    uint8_t* __restrict__ q, float* __restrict__ scale) {
  griddep_wait();  // launched after the kernel that writes this one's inputs
  griddep_launch_dependents();
  __shared__ float part[kQuantWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (kQuantWarps / WPR) + warp / WPR;
  const int64_t live = rows_dev ? min(rows, (int64_t)*rows_dev) : rows;
  const bool active = r < live;
  const int li = (warp % WPR) * 32 + lane;  // lane within the row's warps
  const int nv = cols / 8;
  uint4 w[NV];
  float amax = 0.0f;
  if (active) {
    const uint4* row = reinterpret_cast<const uint4*>(m + (size_t)r * cols);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int v = li + 32 * WPR * j;
      w[j] = v < nv ? row[v] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const uint32_t a[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(a[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(a[i] & 0xFFFF0000u)));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if (WPR > 1) {
    if (lane == 0) part[warp] = amax;
    __syncthreads();
    const int w0 = warp - warp % WPR;
#pragma unroll
    for (int k = 0; k < WPR; ++k) amax = fmaxf(amax, part[w0 + k]);
  }
  if (!active) return;
  const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (li == 0) scale[r] = s;
  uint2* qr = reinterpret_cast<uint2*>(q + (size_t)r * cols);
  const RowDivisor dv = row_divisor(s);
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int v = li + 32 * WPR * j;
    if (v < nv) qr[v] = quantize8_e4m3(w[j], dv);
  }
}

// MX block-scaled FP8 (MXFP8 E4M3, the OCP Microscaling Formats v1.0
// conversion): each block of 32 consecutive values of a row shares the scale
// 2^s, s = floor(log2(amax of the block)) - 8 clamped to [-127, 127] (-127 for
// an all-zero block), stored as the E8M0 byte s + 127; each value becomes
// E4M3(v * 2^-s), round to nearest even, saturating at +-448. The scaling is by
// a power of two, so it is exact and the codes do not depend on the order of
// anything. One warp takes 256 consecutive values of a row (8 blocks): lanes
// 4b..4b+3 hold block b's 32 values (one 16-byte group each) and combine their
// maxima with two shuffles.
constexpr int kMxWarps = 8;

// 2^-s for s in [-127, 127], from its bits (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float pow2_neg(int s) {
  const int e = 127 - s;
  return e > 0 ? __int_as_float(e << 23) : __int_as_float(0x00400000);
}

// floor(log2(a)) - 8 clamped to [-127, 127] for a finite a >= 0; -127 for a = 0.
__device__ __forceinline__ int mx_block_exponent(float a) {
  const uint32_t b = __float_as_uint(a);
  if (b == 0u) return -127;
  const int ef = (int)(b >> 23);
  const int fl = ef > 0 ? ef - 127 : (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
  return min(127, max(-127, fl - 8));
}

// atoms: scale bytes in the layout the GEMM's tensor-core copies read (rows and
// columns multiples of 128): for a row tile rt = r/128 and a k tile kt = b/4,
// a 512-byte atom at (rt * (nb/4) + kt) * 512 holding row r's block b at
// (r%32)*16 + ((r%128)/32)*4 + b%4. Otherwise scale[r * nb + b].
__global__ void __launch_bounds__(kMxWarps * 32) quantize_mx_fp8_kernel(
    const uint16_t* __restrict__ m, int64_t rows, const int32_t* __restrict__ rows_dev, int cols,
    uint8_t* __restrict__ q, uint8_t* __restrict__ scale, int atoms) {
  griddep_wait();  // launched after the kernel that writes this one's inputs
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = cols / 32;
  const int groups = (nb + 7) / 8;
  const int64_t item = (int64_t)blockIdx.x * kMxWarps + warp;
  const int64_t r = item / groups;
  if (r >= rows || (rows_dev && r >= (int64_t)*rows_dev)) return;
  const int b = (int)(item - r * groups) * 8 + (lane >> 2);
  const bool valid = b < nb;
  uint4 w = make_uint4(0u, 0u, 0u, 0u);
  if (valid) w = reinterpret_cast<const uint4*>(m + (size_t)r * cols + (size_t)b * 32)[lane & 3];
  const uint32_t a[4] = {w.x, w.y, w.z, w.w};
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    amax = fmaxf(amax, fabsf(__uint_as_float(a[i] << 16)));
    amax = fmaxf(amax, fabsf(__uint_as_float(a[i] & 0xFFFF0000u)));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  if (!valid) return;
  const int sx = mx_block_exponent(amax);
  const float f = pow2_neg(sx);
  uint32_t packed[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __fmul_rn(__uint_as_float(a[i] << 16), f);
    const float hi = __fmul_rn(__uint_as_float(a[i] & 0xFFFF0000u), f);
    const uint32_t pair =
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);  // lo: low byte
    if (i & 1)
      packed[i >> 1] |= pair << 16;
    else
      packed[i >> 1] = pair;
  }
  reinterpret_cast<uint2*>(q + (size_t)r * cols + (size_t)b * 32)[lane & 3] =
      make_uint2(packed[0], packed[1]);
  if ((lane & 3) == 0) {
    const uint8_t code = (uint8_t)(sx + 127);
    if (atoms)
      scale[((size_t)(r / 128) * (nb / 4) + b / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 +
            b % 4] = code;
    else
      scale[(size_t)r * nb + b] = code;
  }
}

__global__ void transpose_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, int R,
                                 int C, int64_t in_es, int64_t out_es, int64_t out_off) {
  __shared__ uint16_t tile[32][33];
  const int e = blockIdx.z;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const uint16_t* src = in + (size_t)e * in_es;
  uint16_t* dst = out + (size_t)e * out_es + out_off;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < R && c < C) tile[i][threadIdx.x] = src[(size_t)r * C + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < R && c < C) dst[(size_t)c * R + r] = tile[threadIdx.x][i];
  }
}

}  // namespace

int launch_quantize_mx_fp8(const uint16_t* m, int64_t rows, const int32_t* rows_dev, int cols,
                           uint8_t* q, uint8_t* scale, int atoms, cudaStream_t s) {
  if (rows <= 0) return 0;
  const int64_t items = rows * ((cols / 32 + 7) / 8);
  const int64_t blocks = (items + kMxWarps - 1) / kMxWarps;
  launch_pdl(quantize_mx_fp8_kernel, dim3((unsigned)blocks), dim3(kMxWarps * 32), 0, s, m, rows,
             rows_dev, cols, q, scale, atoms);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? 1 : -(int)err;
}

int launch_combine(const CombineArgs& a, cudaStream_t s) {
  if (a.N <= 0) return 0;
  if (a.K <= 2)
    launch_pdl(combine_kernel<2>, dim3(a.N), dim3(kCombineThreads), 0, s, a.o, a.token_routes, a.topk_p, a.y, a.N, a.n_dev, a.H, a.K);
  else if (a.K <= 4)
    launch_pdl(combine_kernel<4>, dim3(a.N), dim3(kCombineThreads), 0, s, a.o, a.token_routes, a.topk_p, a.y, a.N, a.n_dev, a.H, a.K);
  else if (a.K <= 8)
    launch_pdl(combine_kernel<8>, dim3(a.N), dim3(kCombineThreads), 0, s, a.o, a.token_routes, a.topk_p, a.y, a.N, a.n_dev, a.H, a.K);
  else
    launch_pdl(combine_kernel<16>, dim3(a.N), dim3(kCombineThreads), 0, s, a.o, a.token_routes, a.topk_p, a.y, a.N, a.n_dev, a.H, a.K);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? 1 : -(int)err;
}

int launch_combine_bwd(const uint16_t* dxr, const float* part, int n_part,
                       const int32_t* token_routes, int N, int H, int K, uint16_t* dx,
                       float* dprob, cudaStream_t s) {
  if (N <= 0) return 0;
#define MOE_COMBINE_BWD(KM)                                                                  \
  combine_bwd_kernel<KM><<<N, kCombineThreads, 0, s>>>(dxr, part, n_part, token_routes, dx, \
                                                        dprob, N, H, K)
  if (K <= 2)
    MOE_COMBINE_BWD(2);
  else if (K <= 4)
    MOE_COMBINE_BWD(4);
  else if (K <= 8)
    MOE_COMBINE_BWD(8);
  else
    MOE_COMBINE_BWD(16);
#undef MOE_COMBINE_BWD
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? 1 : -(int)err;
}

int launch_quantize_rows_fp8(const uint16_t* m, int64_t rows, const int32_t* rows_dev, int cols,
                             uint8_t* q, float* scale, cudaStream_t s) {
  if (rows <= 0) return 0;
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  const int nv = cols / 8;  // 16-byte groups per row
  const dim3 b(kQuantWarps * 32);
  const unsigned g1 = (unsigned)blocks;                                        // 8 rows per CTA
  const unsigned g2 = (unsigned)((rows + kQuantWarps / 2 - 1) / (kQuantWarps / 2));  // 4 rows
  const unsigned g4 = (unsigned)((rows + kQuantWarps / 4 - 1) / (kQuantWarps / 4));  // 2 rows
  const unsigned g8 = (unsigned)rows;                                          // 1 row
  if (nv <= 64)
    launch_pdl(quantize_rows_fp8_reg_kernel<2, 1>, dim3(g1), dim3(b), 0, s, m, rows, rows_dev, cols, q, scale);
  else if (nv <= 128)
    launch_pdl(quantize_rows_fp8_reg_kernel<4, 1>, dim3(g1), dim3(b), 0, s, m, rows, rows_dev, cols, q, scale);
  else if (nv <= 256)
    launch_pdl(quantize_rows_fp8_reg_kernel<8, 1>, dim3(g1), dim3(b), 0, s, m, rows, rows_dev, cols, q, scale);
  else if (nv <= 512)
    launch_pdl(quantize_rows_fp8_reg_kernel<8, 2>, dim3(g2), dim3(b), 0, s, m, rows, rows_dev, cols, q, scale);
  else if (nv <= 1024)
    launch_pdl(quantize_rows_fp8_reg_kernel<8, 4>, dim3(g4), dim3(b), 0, s, m, rows, rows_dev, cols, q, scale);
  else if (nv <= 2048)
    launch_pdl(quantize_rows_fp8_reg_kernel<8, 8>, dim3(g8), dim3(b), 0, s, m, rows, rows_dev, cols, q, scale);
  else  // rows wider than 16384 values: two passes over the row
    launch_pdl(quantize_rows_fp8_kernel, dim3(g1), dim3(b), 0, s, m, rows, rows_dev, cols, q, scale);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? 1 : -(int)err;
}

int launch_transpose(const uint16_t* in, uint16_t* out, int E, int R, int C, int64_t in_es,
                     int64_t out_es, int64_t out_off, cudaStream_t s) {
  if (E <= 0 || R <= 0 || C <= 0) return 0;
  dim3 grid((C + 31) / 32, (R + 31) / 32, E);
  transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(in, out, R, C, in_es, out_es, out_off);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? 1 : -(int)err;
}

}  // namespace moe
