// Router and route-list kernels (sm_103a).
//
//  R1 router_logits : l[t,e] = (sum over h ascending of x[t,h]*W_r[h,e], one fp32
//                     fma per term) + b[e]. A SIMT SGEMM whose every output is
//                     one sequential fma chain, so the logits (and hence the
//                     top-K indices) are bit-reproducible.
//  R2 router_topk   : one warp per token: softmax with our own fp32 exp, K rounds
//                     of warp-shuffle argmax on a packed (p, ~e) key, renormalise;
//                     the CTA also counts its chunk's routes per expert and ranks
//                     each route among its chunk's same-expert routes.
//  R3 route_scan    : per-expert exclusive scan over chunks (counts, offsets).
//  R3 route_scatter : route list grouped by expert, ascending token order.
//  R4 route_select  : one CTA per expert: radix select of the `cap` highest
//                     renormalised probabilities (ties to the lower token), then
//                     the block-padded layout of sorted_slot_ids / expert_ids /
//                     token_routes.
// Route-list contract: "Permute-Free Grouped GEMM for MoE (bf16, gfx950)",
// section 4 Data structures and section 5 Kernels (route_list_scan,
// route_list_align). Capacity and drop-and-pad: "feat(cuda-graphs): capture
// fixed-capacity MoE execution", Design notes.
#include <math.h>

#include "moe_internal.h"

namespace moe {
namespace {

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

// fp32 exp: Cody-Waite reduction v = n ln2 + r (ln 2 split into an fp32 head
// and an fp32 tail), degree-7 Taylor polynomial of e^r in Horner form with
// fma, scale by 2^n through the exponent field. Domain v <= 0 (softmax);
// v < -87 gives +0. Every operation is an explicitly rounded IEEE op.
__device__ __forceinline__ float route_exp(float v) {
  if (v < -87.0f) return 0.0f;
  const float log2e = __uint_as_float(0x3FB8AA3Bu);
  const float ln2_hi = __uint_as_float(0x3F317218u);
  const float ln2_lo = __uint_as_float(0xB102E308u);
  const float n = rintf(__fmul_rn(v, log2e));
  float r = __fmaf_rn(-n, ln2_hi, v);
  r = __fmaf_rn(-n, ln2_lo, r);
  float p = __uint_as_float(0x39500D01u);         // 1/7!
  p = __fmaf_rn(p, r, __uint_as_float(0x3AB60B61u));  // 1/6!
  p = __fmaf_rn(p, r, __uint_as_float(0x3C088889u));  // 1/5!
  p = __fmaf_rn(p, r, __uint_as_float(0x3D2AAAABu));  // 1/4!
  p = __fmaf_rn(p, r, __uint_as_float(0x3E2AAAABu));  // 1/3!
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const float scale = __uint_as_float((uint32_t)((int)n + 127) << 23);
  return __fmul_rn(p, scale);
}

// ---------------------------------------------------------------- R1
constexpr int LBM = 64, LBN = 64, LBK = 16;  // 256 threads, 4x4 outputs each

__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ wr,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ logits, int N,
                                                            int H, int E) {
  __shared__ __align__(16) float As[2][LBK][LBM];
  __shared__ __align__(16) float Bs[2][LBK][LBN];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * LBM, n0 = blockIdx.x * LBN;
  const int a_row = tid >> 2, a_col = (tid & 3) * 4;
  const int b_row = tid >> 4, b_col = (tid & 15) * 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  float ra[4], rb[4];
  auto load = [&](int k0) {
    const int t = m0 + a_row;
    if (t < N) {
      const uint2 v = *reinterpret_cast<const uint2*>(x + (size_t)t * H + k0 + a_col);
      ra[0] = bf16_to_f32((uint16_t)(v.x & 0xFFFFu));
      ra[1] = bf16_to_f32((uint16_t)(v.x >> 16));
      ra[2] = bf16_to_f32((uint16_t)(v.y & 0xFFFFu));
      ra[3] = bf16_to_f32((uint16_t)(v.y >> 16));
    } else {
      ra[0] = ra[1] = ra[2] = ra[3] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = n0 + b_col + j;
      rb[j] = (e < E) ? wr[(size_t)(k0 + b_row) * E + e] : 0.0f;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int j = 0; j < 4; ++j) As[buf][a_col + j][a_row] = ra[j];
#pragma unroll
    for (int j = 0; j < 4; ++j) Bs[buf][b_row][b_col + j] = rb[j];
  };
  load(0);
  store(0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < H; k0 += LBK) {
    const bool more = k0 + LBK < H;
    if (more) load(k0 + LBK);
#pragma unroll
    for (int kk = 0; kk < LBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
    }
    if (more) store(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = m0 + ty * 4 + i;
    if (t >= N) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = n0 + tx * 4 + j;
      if (e < E) logits[(size_t)t * E + e] = __fadd_rn(acc[i][j], bias ? bias[e] : 0.0f);
    }
  }
}

// ---------------------------------------------------------------- R2
constexpr int kTopkWarps = 16;

__global__ void __launch_bounds__(kTopkWarps * 32) router_topk_kernel(
    const float* __restrict__ logits, int N, int E, int K, int renorm, int32_t* __restrict__ topk_ids,
    float* __restrict__ topk_p, int32_t* __restrict__ chunk_rank,
    int32_t* __restrict__ chunk_counts) {
  __shared__ float zbuf[kTopkWarps][kMaxExperts];
  __shared__ int32_t ids_s[kTokensPerChunk * kMaxTopK];
  __shared__ int32_t hist[kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTokensPerChunk;
  const int nt = min(kTokensPerChunk, N - t0);
  constexpr int PER = kMaxExperts / 32;
  for (int tl = warp; tl < nt; tl += kTopkWarps) {
    const int t = t0 + tl;
    const float* l = logits + (size_t)t * E;
    float v[PER];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = lane + 32 * j;
      v[j] = (e < E) ? l[e] : -INFINITY;
      m = fmaxf(m, v[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = lane + 32 * j;
      if (e < E) {
        v[j] = route_exp(__fsub_rn(v[j], m));
        zbuf[warp][e] = v[j];
      }
    }
    __syncwarp();
    float s = 0.0f;
    if (lane == 0)
      for (int e = 0; e < E; ++e) s = __fadd_rn(s, zbuf[warp][e]);  // ascending e
    s = __shfl_sync(0xFFFFFFFFu, s, 0);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < PER; ++j) v[j] = __fdiv_rn(v[j], s);
    uint32_t taken = 0;
    float d = 0.0f, my_p = 0.0f;
    int my_id = 0;
    for (int k = 0; k < K; ++k) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u)) {
          const unsigned long long key =
              ((unsigned long long)__float_as_uint(v[j]) << 32) | (0xFFFFFFFFu - (uint32_t)e);
          best = key > best ? key : best;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = other > best ? other : best;
      }
      const int eb = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
      const float pb = __uint_as_float((uint32_t)(best >> 32));
      if ((eb & 31) == lane) taken |= 1u << (eb >> 5);
      d = __fadd_rn(d, pb);  // pick order
      if (lane == k) { my_id = eb; my_p = pb; }
      if (lane == 0) ids_s[tl * K + k] = eb;
    }
    if (lane < K) {
      topk_ids[(size_t)t * K + lane] = my_id;
      topk_p[(size_t)t * K + lane] = renorm ? __fdiv_rn(my_p, d) : my_p;
    }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  for (int r = threadIdx.x; r < nt * K; r += blockDim.x) {
    const int tl = r / K;
    const int e = ids_s[r];
    int cnt = 0;
    for (int r2 = 0; r2 < tl * K; ++r2) cnt += (ids_s[r2] == e);
    chunk_rank[(size_t)t0 * K + r] = cnt;
    atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// ---------------------------------------------------------------- R3
__global__ void route_scan_kernel(const int32_t* __restrict__ chunk_counts,
                                  int32_t* __restrict__ chunk_off,
                                  int32_t* __restrict__ expert_counts,
                                  int32_t* __restrict__ expert_off, int C, int E) {
  __shared__ int32_t tot[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int c = 0; c < C; ++c) {
      const int v = chunk_counts[(size_t)c * E + e];
      chunk_off[(size_t)c * E + e] = run;
      run += v;
    }
    tot[e] = run;
    expert_counts[e] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      expert_off[e] = acc;
      acc += tot[e];
    }
    expert_off[E] = acc;
  }
}

__global__ void route_scatter_kernel(const int32_t* __restrict__ topk_ids,
                                     const int32_t* __restrict__ chunk_rank,
                                     const int32_t* __restrict__ chunk_off,
                                     const int32_t* __restrict__ expert_off,
                                     int32_t* __restrict__ route_list, int N, int K, int E) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= (int64_t)N * K) return;
  const int t = (int)(r / K);
  const int c = t / kTokensPerChunk;
  const int e = topk_ids[r];
  if (e < 0 || e >= E) return;
  const int64_t pos = (int64_t)expert_off[e] + chunk_off[(size_t)c * E + e] + chunk_rank[r];
  if (pos >= 0 && pos < (int64_t)N * K) route_list[pos] = (int32_t)r;
}

// ---------------------------------------------------------------- R4
constexpr int kSelThreads = 1024;

// Exclusive scan of v over the CTA (kSelThreads threads, all must call).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = (lane < (kSelThreads >> 5)) ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += u;
    }
    warp_tot[lane] = wi - w;
  }
  __syncthreads();
  return warp_tot[warp] + incl - v;
}

__global__ void __launch_bounds__(kSelThreads) route_select_kernel(
    const int32_t* __restrict__ expert_counts, const int32_t* __restrict__ expert_off,
    const int32_t* __restrict__ route_list, const float* __restrict__ topk_p, int N, int E, int K,
    int cap, int cpad, int bm, uint8_t* __restrict__ keep, int32_t* __restrict__ kept_counts,
    int32_t* __restrict__ sorted_slot_ids, int32_t* __restrict__ expert_ids,
    int32_t* __restrict__ block_start, int32_t* __restrict__ ntpp,
    int32_t* __restrict__ token_routes) {
  extern __shared__ uint32_t dyn[];
  __shared__ int32_t hist[256];
  __shared__ int32_t warp_tot[32];
  __shared__ uint32_t s_prefix;
  __shared__ int32_t s_remaining;
  const int e = blockIdx.x;
  const int tid = threadIdx.x;
  // a token picks each expert at most once, so n <= N; the clamps only guard
  // the staging buffers and the route list
  const int n = min(max(expert_counts[e], 0), N);
  const int off = min(max(expert_off[e], 0), N * K - n);
  uint32_t* keys = dyn;                                  // p' bits, list order
  int32_t* rids = reinterpret_cast<int32_t*>(dyn + N);   // route index t*K+k
  for (int i = tid; i < n; i += kSelThreads) {
    const int r = route_list[off + i];
    rids[i] = r;
    keys[i] = __float_as_uint(topk_p[r]);
  }
  __syncthreads();
  const bool select = n > cap;
  uint32_t thr = 0;
  int needed = 0;
  if (select) {
    // k-th largest key (k = cap), 8 bits at a time from the top
    uint32_t prefix = 0, mask = 0;
    int remaining = cap;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < n; i += kSelThreads) {
        const uint32_t k = keys[i];
        if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int cum = 0, d = 255;
        for (; d > 0; --d) {
          if (cum + hist[d] >= remaining) break;
          cum += hist[d];
        }
        s_remaining = remaining - cum;
        s_prefix = prefix | ((uint32_t)d << shift);
      }
      __syncthreads();
      remaining = s_remaining;
      prefix = s_prefix;
      mask |= 0xFFu << shift;
    }
    thr = prefix;
    needed = remaining;  // how many keys equal to thr are kept (lowest tokens first)
  }
  // each thread owns a contiguous run of the list, so scans follow list order
  const int ipt = (n + kSelThreads - 1) / kSelThreads;
  const int i0 = min(n, tid * ipt), i1 = min(n, i0 + ipt);
  int ties = 0;
  if (select)
    for (int i = i0; i < i1; ++i) ties += (keys[i] == thr);
  const int tie_base = block_exclusive_scan(ties, warp_tot);
  int tie_rank = tie_base;
  int kept_local = 0;
  for (int i = i0; i < i1; ++i) {
    bool kp = true;
    if (select) {
      const uint32_t k = keys[i];
      kp = k > thr || (k == thr && tie_rank < needed);
      tie_rank += (k == thr);
    }
    kept_local += kp;
  }
  int pos = block_exclusive_scan(kept_local, warp_tot);
  // second pass: same keep decisions, now writing the layout
  tie_rank = tie_base;
  const int base = e * cpad;
  for (int i = i0; i < i1; ++i) {
    bool kp = true;
    if (select) {
      const uint32_t k = keys[i];
      kp = k > thr || (k == thr && tie_rank < needed);
      tie_rank += (k == thr);
    }
    const int r = rids[i];
    if (kp) {
      const int slot = base + pos;
      ++pos;
      sorted_slot_ids[slot] = r / K;
      token_routes[r] = slot;
      keep[r] = 1;
    } else {
      token_routes[r] = -1;
      keep[r] = 0;
    }
  }
  const int kept_e = select ? cap : n;
  for (int s = kept_e + tid; s < cpad; s += kSelThreads) sorted_slot_ids[base + s] = N;
  const int nb = cpad / bm;
  for (int b = tid; b < nb; b += kSelThreads)
    expert_ids[(size_t)e * nb + b] = (b * bm < kept_e) ? e : -1;
  if (tid == 0) {
    block_start[e] = e * nb;
    kept_counts[e] = kept_e;
    if (e == 0) *ntpp = E * cpad;
  }
}

}  // namespace

int launch_route(const RouteArgs& a, cudaStream_t s) {
  int launched = 0;
  const int C = (a.N + kTokensPerChunk - 1) / kTokensPerChunk;
  if (a.N > 0) {
    dim3 g1((a.E + LBN - 1) / LBN, (a.N + LBM - 1) / LBM);
    router_logits_kernel<<<g1, 256, 0, s>>>(a.x, a.wr, a.bias, a.ws.logits, a.N, a.H, a.E);
    ++launched;
    router_topk_kernel<<<C, kTopkWarps * 32, 0, s>>>(a.ws.logits, a.N, a.E, a.K, a.renorm,
                                                     a.topk_ids, a.topk_p, a.ws.chunk_rank,
                                                     a.ws.chunk_counts);
    ++launched;
  }
  route_scan_kernel<<<1, 256, 0, s>>>(a.ws.chunk_counts, a.ws.chunk_off, a.expert_counts,
                                      a.ws.expert_off, C, a.E);
  ++launched;
  if (a.N > 0) {
    const int64_t R = (int64_t)a.N * a.K;
    route_scatter_kernel<<<(unsigned)((R + 255) / 256), 256, 0, s>>>(
        a.topk_ids, a.ws.chunk_rank, a.ws.chunk_off, a.ws.expert_off, a.ws.route_list, a.N, a.K,
        a.E);
    ++launched;
  }
  const size_t dyn = (size_t)a.N * 8;
  cudaError_t err = cudaFuncSetAttribute(route_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (err != cudaSuccess) return -(int)err;
  const int cap = (int)(a.cap < a.N ? a.cap : a.N);
  route_select_kernel<<<a.E, kSelThreads, dyn, s>>>(
      a.expert_counts, a.ws.expert_off, a.ws.route_list, a.topk_p, a.N, a.E, a.K, cap,
      (int)a.cpad, a.bm, a.keep, a.kept_counts, a.sorted_slot_ids, a.expert_ids, a.block_start,
      a.ntpp, a.token_routes);
  ++launched;
  err = cudaGetLastError();
  if (err != cudaSuccess) return -(int)err;
  return launched;
}

}  // namespace moe
