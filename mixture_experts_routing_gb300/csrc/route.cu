// Router and route-list kernels (sm_103a).
//
//  R1 router_logits : l[t,e] = (sum over h ascending of x[t,h]*W_r[h,e], one fp32
//                     fma per term) + b[e]. A SIMT SGEMM whose every output is
//                     one sequential fma chain, so the logits (and hence the
//                     top-K indices) are bit-reproducible.
//  R2 router_topk   : one warp per token: softmax with our own fp32 exp, K rounds
//                     of warp argmax (max of the p bits, then min of the expert
//                     ids at that max), renormalise; then the CTA sorts its
//                     32-token chunk's routes by expert (stable) and records
//                     per-expert counts and offsets (the scan's first level).
//  R3+R4 route_select: one CTA per expert: exclusive scan of the expert's chunk
//                     counts, gather of its routes in token order, radix select
//                     of the `cap` highest renormalised probabilities (ties to
//                     the lower token), then the block-padded layout of
//                     sorted_slot_ids / expert_ids / token_routes.
// Route-list contract: "Permute-Free Grouped GEMM for MoE (bf16, gfx950)",
// section 4 Data structures and section 5 Kernels (route_list_scan,
// route_list_align). Capacity and drop-and-pad: "feat(cuda-graphs): capture
// fixed-capacity MoE execution", Design notes.
#include <cuda_bf16.h>
#include <math.h>

#include "moe_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

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

// Live token count: *n_dev clamped to [0, Nmax], or Nmax without a device
// count. Buffers and grids are sized for Nmax (the static bound a captured
// graph was built for); tokens at or past the live count are absent.
__device__ __forceinline__ int live_tokens(const int32_t* n_dev, int Nmax) {
  if (!n_dev) return Nmax;
  const int v = *n_dev;
  return v < 0 ? 0 : (v > Nmax ? Nmax : v);
}

// ---------------------------------------------------------------- R1
// A SIMT SGEMM in which every output is one fp32 fma chain over ascending h.
// Work split for the whole GPU: the [N, E] logit matrix is cut into one token
// group per SM (bm = ceil(N / groups) tokens, any integer) by tiles of
// BN = 4*TX experts, one CTA per block. A CTA has TY x TX threads with 7
// tokens x 4 experts each (TY = ceil(bm/7) rounded up to 4; rows past bm
// idle). A warp covers 4 thread rows x 8 thread columns, so each contraction
// step reads 4 distinct token vectors and 8 distinct expert vectors from
// shared memory: three conflict-free 16-byte loads per thread for 28 fmas.
// Stages of BK = 32 contraction elements run in a 4-deep cp.async ring: x
// rows (bf16, converted once per stage into a transposed fp32 tile whose
// 7-token vectors are padded to 8) and W_r rows (fp32). (The earlier
// power-of-two tiling, 64 tokens x 128 experts per CTA, gave the DeepSeek-V3
// router shape 128 CTAs for 152 SMs and ran at 47 % of the fp32 FMA peak.)
constexpr int LBK = 32, LSTAGES = 4;
constexpr int kRTM = 7, kRTN = 4, kRPad = 8, kRMaxThreads = 512;

__device__ __forceinline__ void cpa16(uint32_t dst, const void* src, uint32_t n) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cpa4(uint32_t dst, const void* src, uint32_t n) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}

// Dynamic shared memory of one CTA: x stages, W_r stages, the fp32 x tile.
constexpr size_t router_smem_bytes(int bm, int bn, int ty) {
  return (size_t)LSTAGES * bm * LBK * 2 + (size_t)LSTAGES * LBK * bn * 4 +
         (size_t)LBK * ty * kRPad * 4;
}

// Converts stage rows [0, rows) of bf16 x ([row][KB]) into the transposed
// fp32 tile `as` ([KB][RM], token m at (m/7)*8 + m%7). With kSw128 the rows
// (KB = 64: 128 bytes) are 128-byte swizzled, 16-byte chunk q of row m at
// m*128 + ((q ^ (m % 8)) * 16), so the consecutive rows a warp reads fall on
// distinct banks.
template <int KB, bool kSw128 = false>
__device__ __forceinline__ void router_convert(const uint16_t* xsl, float* as, int rows, int RM,
                                               int tid, int NT) {
  for (int c = tid; c < rows * (KB / 8); c += NT) {
    const int m = c % rows, q = c / rows;
    const int pos = (m / kRTM) * kRPad + m % kRTM;
    const int qs = kSw128 ? (q ^ (m & 7)) : q;
    const uint4 v = *reinterpret_cast<const uint4*>(xsl + m * KB + qs * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      as[(q * 8 + 2 * i) * RM + pos] = __uint_as_float(w[i] << 16);
      as[(q * 8 + 2 * i + 1) * RM + pos] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

// Thread rows of a CTA at most: 512 threads, 32 rows, a multiple of 4.
template <int TX>
__host__ __device__ constexpr int router_ty_max() {
  return (kRMaxThreads / TX < 32 ? kRMaxThreads / TX : 32) / 4 * 4;
}

// The conversion above with each thread's (row, chunk) pairs worked out once
// per CTA: the same pairs recur every stage, and the division by the
// runtime row count and the position arithmetic then leave the stage loop.
// The fp32 tile has the compile-time token stride RMS.
template <int KB, bool kSw128, int RMS, int CMAX>
struct RouterConvertPlan {
  // per chunk: bf16 offset in the stage's x tile << 16 | float offset of its
  // first value in the fp32 tile (both below 2^15); -1 for no chunk
  int item[CMAX];
  static_assert(7 * 32 * KB < (1 << 15) && KB * RMS < (1 << 15), "offsets fit 15 bits");
  __device__ __forceinline__ RouterConvertPlan(int rows, int tid, int NT) {
#pragma unroll
    for (int i = 0; i < CMAX; ++i) {
      const int c = tid + i * NT;
      item[i] = -1;
      if (c < rows * (KB / 8)) {
        const int m = c % rows, q = c / rows;
        const int src = m * KB + (kSw128 ? (q ^ (m & 7)) : q) * 8;
        item[i] = (src << 16) | (q * 8 * RMS + (m / kRTM) * kRPad + m % kRTM);
      }
    }
  }
  __device__ __forceinline__ void run(const uint16_t* xsl, float* as) const {
#pragma unroll
    for (int i = 0; i < CMAX; ++i) {
      if (item[i] < 0) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(xsl + (item[i] >> 16));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float* d = as + (item[i] & 0xFFFF);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        d[(2 * j) * RMS] = __uint_as_float(w[j] << 16);
        d[(2 * j + 1) * RMS] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
};

// One stage of the fma chains with the compile-time token stride RMS: the
// operand loads of step k+1 are issued before the fmas of step k, so their
// shared-memory latency overlaps the 28 fmas (the chains are unchanged).
template <int BN, int KB, int RMS>
__device__ __forceinline__ void router_fma_stage_c(float (&acc)[kRTM][kRTN], const float* as,
                                                   const float* bsl, int ty, int tx) {
  const float* ap = as + ty * kRPad;
  const float* bp = bsl + tx * kRTN;
  float4 a0 = *reinterpret_cast<const float4*>(ap);
  float4 a1 = *reinterpret_cast<const float4*>(ap + 4);
  float4 b = *reinterpret_cast<const float4*>(bp);
#pragma unroll
  for (int kk = 0; kk < KB; ++kk) {
    float4 a0n = a0, a1n = a1, bn = b;
    if (kk + 1 < KB) {
      a0n = *reinterpret_cast<const float4*>(ap + (kk + 1) * RMS);
      a1n = *reinterpret_cast<const float4*>(ap + (kk + 1) * RMS + 4);
      bn = *reinterpret_cast<const float4*>(bp + (kk + 1) * BN);
    }
    const float av[kRTM] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z};
    const float bv[kRTN] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < kRTM; ++i)
#pragma unroll
      for (int j = 0; j < kRTN; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
    a0 = a0n;
    a1 = a1n;
    b = bn;
  }
}

// One stage of the fma chains: acc[i][j] += x[token i][k] * W_r[k][expert j]
// for k ascending over the KB values of the stage.
template <int BN, int KB>
__device__ __forceinline__ void router_fma_stage(float (&acc)[kRTM][kRTN], const float* as,
                                                 const float* bsl, int RM, int ty, int tx) {
#pragma unroll
  for (int kk = 0; kk < KB; ++kk) {
    const float4 a0 = *reinterpret_cast<const float4*>(&as[kk * RM + ty * kRPad]);
    const float4 a1 = *reinterpret_cast<const float4*>(&as[kk * RM + ty * kRPad + 4]);
    const float4 b = *reinterpret_cast<const float4*>(&bsl[kk * BN + tx * kRTN]);
    const float av[kRTM] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z};
    const float bv[kRTN] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < kRTM; ++i)
#pragma unroll
      for (int j = 0; j < kRTN; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
  }
}

__device__ __forceinline__ void router_store(const float (&acc)[kRTM][kRTN], float* logits,
                                             const float* bias, int m0, int rows, int n0, int E,
                                             int ty, int tx) {
#pragma unroll
  for (int i = 0; i < kRTM; ++i) {
    const int r = ty * kRTM + i;
    if (r >= rows) continue;
    float* out = logits + (size_t)(m0 + r) * E;
#pragma unroll
    for (int j = 0; j < kRTN; ++j) {
      const int e = n0 + tx * kRTN + j;
      if (e < E) out[e] = __fadd_rn(acc[i][j], bias ? bias[e] : 0.0f);
    }
  }
}

// cp.async form: any E (W_r rows read 16 or 4 bytes at a time).
template <int TX>
__global__ void __launch_bounds__(kRMaxThreads) router_logits_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ wr, const float* __restrict__ bias,
    float* __restrict__ logits, int Nmax, const int32_t* __restrict__ n_dev, int H, int E, int bm,
    int wr_vec4) {
  griddep_wait();  // launched after the kernel that writes this one's inputs
  griddep_launch_dependents();
  constexpr int BN = TX * kRTN;
  const int NT = blockDim.x, RM = (NT / TX) * kRPad;
  const int N = live_tokens(n_dev, Nmax);
  const int m0 = blockIdx.y * bm;
  if (m0 >= N) return;  // the whole group is past the live tokens
  const int rows = min(bm, N - m0);
  extern __shared__ __align__(16) uint8_t rsm[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(rsm);                             // [S][bm][BK] bf16
  float* bs = reinterpret_cast<float*>(rsm + (size_t)LSTAGES * bm * LBK * 2);   // [S][BK][BN]
  float* as = bs + LSTAGES * LBK * BN;                                          // [BK][RM]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tx = (warp % (TX / 8)) * 8 + (lane & 7);
  const int ty = (warp / (TX / 8)) * 4 + (lane >> 3);
  const int n0 = blockIdx.x * BN;
  // the pad of each token vector and the rows past `rows` stay zero
  for (int i = tid; i < LBK * RM; i += NT) as[i] = 0.0f;
  float acc[kRTM][kRTN];
#pragma unroll
  for (int i = 0; i < kRTM; ++i)
#pragma unroll
    for (int j = 0; j < kRTN; ++j) acc[i][j] = 0.0f;
  const int KT = H / LBK;
  auto issue = [&](int kt) {
    if (kt < KT) {
      const int slot = kt % LSTAGES, k0 = kt * LBK;
      for (int c = tid; c < rows * (LBK / 8); c += NT) {
        const int row = c / (LBK / 8), q = c % (LBK / 8);
        cpa16((uint32_t)__cvta_generic_to_shared(xs + ((size_t)slot * bm + row) * LBK + q * 8),
              x + (size_t)(m0 + row) * H + k0 + q * 8, 16u);
      }
      float* bsl = bs + (size_t)slot * LBK * BN;
      if (wr_vec4) {
        for (int c = tid; c < LBK * BN / 4; c += NT) {
          const int k = c / (BN / 4), q = c % (BN / 4);
          const int e = n0 + q * 4;
          const bool ok = e < E;
          cpa16((uint32_t)__cvta_generic_to_shared(bsl + k * BN + q * 4),
                wr + (size_t)(k0 + k) * E + (ok ? e : 0), ok ? 16u : 0u);
        }
      } else {
        for (int c = tid; c < LBK * BN; c += NT) {
          const int k = c / BN, q = c % BN;
          const int e = n0 + q;
          const bool ok = e < E;
          cpa4((uint32_t)__cvta_generic_to_shared(bsl + k * BN + q),
               wr + (size_t)(k0 + k) * E + (ok ? e : 0), ok ? 4u : 0u);
        }
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  for (int st = 0; st < LSTAGES - 1; ++st) issue(st);
  for (int kt = 0; kt < KT; ++kt) {
    asm volatile("cp.async.wait_group %0;" ::"n"(LSTAGES - 2) : "memory");
    __syncthreads();  // stage kt landed; every thread is done with stage kt-1 and with `as`
    issue(kt + LSTAGES - 1);
    router_convert<LBK>(xs + (size_t)(kt % LSTAGES) * bm * LBK, as, rows, RM, tid, NT);
    __syncthreads();
    router_fma_stage<BN, LBK>(acc, as, bs + (size_t)(kt % LSTAGES) * LBK * BN, RM, ty, tx);
  }
  router_store(acc, logits, bias, m0, rows, n0, E, ty, tx);
}

// Shared-memory layout of the TMA form: NS stages of [x tile bm x KB
// bf16, padded to 128 B | W_r tile BK x BN fp32], two fp32 x tiles, the stage
// barriers.
struct RouterTmaLayout {
  uint32_t xbytes, stage, as_off, bar_off, total;
};
template <int KB, int NS>
__host__ __device__ inline RouterTmaLayout router_tma_layout(int bm, int bn, int rms) {
  RouterTmaLayout L;
  // a 128-byte-swizzled x tile (KB = 64) starts on a 1024-byte boundary
  constexpr uint32_t kAlign = KB == 64 ? 1024u : 128u;
  L.xbytes = ((uint32_t)bm * KB * 2 + kAlign - 1u) & ~(kAlign - 1u);
  L.stage = L.xbytes + (uint32_t)KB * bn * 4;
  L.as_off = NS * L.stage;
  L.bar_off = L.as_off + 2u * KB * rms * 4;
  L.total = L.bar_off + NS * 8 + kAlign;  // + slack for aligning the base
  return L;
}

// TMA form (E a multiple of 4, E >= BN): one thread loads each stage with two
// 2-D tensor copies (x box BK x bm, W_r box BN x BK; rows and experts past
// the tensor read as zero) completing on the stage's mbarrier. The fp32 x
// tile is double-buffered, so one CTA barrier per stage orders everything:
// after it, the tile converted in the previous iteration is visible, and
// every thread is done with the stage slot the producer refills and with the
// x tile the next conversion overwrites. Waits are bounded; a CTA that runs
// out of time records kErrWaitRouter, waits (bounded) for its copies in
// flight and leaves without writing logits. At most one CTA per SM is
// resident (the shared-memory floor below), and declaring it lets the
// compiler keep more operand loads in flight: 64 -> 79..107 registers,
// qwen3_30b's route_align 0.130 -> 0.125 ms, dropless N=16384's 0.236 ->
// 0.229 ms.
template <int TX, int KB, int NS>
__global__ void __launch_bounds__(kRMaxThreads, 1) router_logits_tma_kernel(
    const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
    const float* __restrict__ bias, float* __restrict__ logits, int Nmax,
    const int32_t* __restrict__ n_dev, int H, int E, int bm, uint32_t* __restrict__ err) {
  griddep_wait();  // launched after the kernel that writes this one's inputs
  griddep_launch_dependents();
  constexpr int BN = TX * kRTN;
  constexpr int RMS = router_ty_max<TX>() * kRPad;            // token stride of the fp32 x tile
  constexpr int CMAX = (kRTM * KB + 8 * TX - 1) / (8 * TX);   // conversion chunks a thread takes
  const int NT = blockDim.x;
  const int N = live_tokens(n_dev, Nmax);
  const int m0 = blockIdx.y * bm;
  if (m0 >= N) return;
  const int rows = min(bm, N - m0);
  const RouterTmaLayout L = router_tma_layout<KB, NS>(bm, BN, RMS);
  extern __shared__ __align__(16) uint8_t rsm_raw[];
  constexpr uint32_t kAlign = KB == 64 ? 1024u : 128u;
  uint8_t* rsm = rsm_raw + ((kAlign - (smem_u32(rsm_raw) & (kAlign - 1u))) & (kAlign - 1u));
  const uint32_t sbase = smem_u32(rsm);
  float* as = reinterpret_cast<float*>(rsm + L.as_off);  // [2][BK][RM]
  const uint32_t bar0 = sbase + L.bar_off;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tx = (warp % (TX / 8)) * 8 + (lane & 7);
  const int ty = (warp / (TX / 8)) * 4 + (lane >> 3);
  const int n0 = blockIdx.x * BN;
  const int KT = H / KB;
  const uint32_t tx_bytes = (uint32_t)bm * KB * 2 + (uint32_t)KB * BN * 4;
  for (int i = tid; i < 2 * KB * RMS; i += NT) as[i] = 0.0f;
  const RouterConvertPlan<KB, KB == 64, RMS, CMAX> plan(rows, tid, NT);
  if (tid == 0) {
    tma_prefetch_desc(&tmx);
    tma_prefetch_desc(&tmw);
    for (int st = 0; st < NS; ++st) mbar_init(bar0 + 8u * st, 1);
    mbar_fence_init();
  }
  __syncthreads();
  uint64_t pol_x = 0, pol_w = 0;
  int issued = 0;
  auto issue = [&](int kt) {  // thread 0 only
    const int slot = kt % NS;
    const uint32_t st = sbase + (uint32_t)slot * L.stage, bar = bar0 + 8u * slot;
    mbar_arrive_expect_tx(bar, tx_bytes);
    tma_load_2d(st, &tmx, kt * KB, m0, bar, pol_x);
    tma_load_2d(st + L.xbytes, &tmw, n0, kt * KB, bar, pol_w);
    ++issued;
  };
  if (tid == 0) {
    pol_x = policy_evict_first();
    pol_w = policy_evict_last();
    for (int kt = 0; kt < NS - 1 && kt < KT; ++kt) issue(kt);
  }
  float acc[kRTM][kRTN];
#pragma unroll
  for (int i = 0; i < kRTM; ++i)
#pragma unroll
    for (int j = 0; j < kRTN; ++j) acc[i][j] = 0.0f;
  int waited = 0;  // stages this thread saw arrive
  bool ok = mbar_wait(bar0, 0u, err, kErrWaitRouter);
  if (ok) {
    ++waited;
    plan.run(reinterpret_cast<const uint16_t*>(rsm), as);
  }
  for (int kt = 0; kt < KT; ++kt) {
    if (!__syncthreads_and(ok)) break;
    if (tid == 0 && kt + NS - 1 < KT) issue(kt + NS - 1);
    const int slot = kt % NS;
    router_fma_stage_c<BN, KB, RMS>(
        acc, as + (kt & 1) * KB * RMS,
        reinterpret_cast<const float*>(rsm + (size_t)slot * L.stage + L.xbytes), ty, tx);
    if (kt + 1 < KT) {
      const int ns = (kt + 1) % NS;
      ok = mbar_wait(bar0 + 8u * ns, (uint32_t)((kt + 1) / NS) & 1u, err, kErrWaitRouter);
      if (ok) {
        ++waited;
        plan.run(reinterpret_cast<const uint16_t*>(rsm + (size_t)ns * L.stage),
                 as + ((kt + 1) & 1) * KB * RMS);
      }
    }
  }
  if (!__syncthreads_and(ok)) {
    // out of time: let this CTA's copies in flight land before leaving
    if (tid == 0)
      for (int st = waited; st < issued; ++st)
        if (!mbar_wait(bar0 + 8u * (st % NS), (uint32_t)(st / NS) & 1u, err,
                       kErrWaitRouter))
          break;
    return;
  }
  router_store(acc, logits, bias, m0, rows, n0, E, ty, tx);
}

// Few chains (small N*E, where the tiled kernels leave most lanes idle and
// walk H/32 pipelined stages), and every router with fewer than 32 experts
// (see launch_router_logits): one thread per token and 2 consecutive
// experts, the whole contraction in registers, x rows and W_r rows read from
// global memory (shared between threads through L1), the next 16 values of h
// loaded while the current 16 are multiplied (8 at a time measured 9.0 us on
// a 256-token, H = 128, E = 8 router: one load round trip per 8 values).
// Same chains: ascending h, one fma per term, bias last.
constexpr int kRSmallThreads = 128;
constexpr int kRSmallG = 16;  // values of h per load step (H is a multiple of 128)

template <bool kVec2>
__global__ void __launch_bounds__(kRSmallThreads) router_logits_small_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ wr, const float* __restrict__ bias,
    float* __restrict__ logits, int Nmax, const int32_t* __restrict__ n_dev, int H, int E) {
  griddep_wait();  // launched after the kernel that writes this one's inputs
  griddep_launch_dependents();
  constexpr int XV = kRSmallG / 8;  // 16-byte x loads per step
  const int eg = (E + 1) / 2;       // pairs of experts
  const int64_t gid = (int64_t)blockIdx.x * kRSmallThreads + threadIdx.x;
  const int N = live_tokens(n_dev, Nmax);
  const int t = (int)(gid / eg), e0 = (int)(gid % eg) * 2;
  if (t >= N) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  auto load = [&](int hg, uint4 (&xv)[XV], float (&w)[kRSmallG][2]) {
#pragma unroll
    for (int v = 0; v < XV; ++v) xv[v] = __ldg(xr + hg * XV + v);
#pragma unroll
    for (int i = 0; i < kRSmallG; ++i) {
      const float* wrow = wr + (size_t)(hg * kRSmallG + i) * E + e0;
      if (kVec2) {
        const float2 q = __ldg(reinterpret_cast<const float2*>(wrow));
        w[i][0] = q.x;
        w[i][1] = q.y;
      } else {
        w[i][0] = __ldg(wrow);
        w[i][1] = (e0 + 1 < E) ? __ldg(wrow + 1) : 0.0f;
      }
    }
  };
  float acc0 = 0.0f, acc1 = 0.0f;
  uint4 xv[XV];
  float w[kRSmallG][2];
  load(0, xv, w);
  const int steps = H / kRSmallG;
  for (int hg = 0; hg < steps; ++hg) {
    uint4 xn[XV];
    float wn[kRSmallG][2];
#pragma unroll
    for (int v = 0; v < XV; ++v) xn[v] = xv[v];
    if (hg + 1 < steps) load(hg + 1, xn, wn);
#pragma unroll
    for (int i = 0; i < kRSmallG; ++i) {
      const uint4 q = xv[i >> 3];
      const uint32_t xw[4] = {q.x, q.y, q.z, q.w};
      const int k = i & 7;
      const float xf = __uint_as_float((k & 1) ? (xw[k >> 1] & 0xFFFF0000u) : (xw[k >> 1] << 16));
      acc0 = __fmaf_rn(xf, w[i][0], acc0);
      acc1 = __fmaf_rn(xf, w[i][1], acc1);
    }
#pragma unroll
    for (int v = 0; v < XV; ++v) xv[v] = xn[v];
#pragma unroll
    for (int i = 0; i < kRSmallG; ++i) {
      w[i][0] = wn[i][0];
      w[i][1] = wn[i][1];
    }
  }
  float* out = logits + (size_t)t * E;
  out[e0] = __fadd_rn(acc0, bias ? bias[e0] : 0.0f);
  if (e0 + 1 < E) out[e0 + 1] = __fadd_rn(acc1, bias ? bias[e0 + 1] : 0.0f);
}

int router_sm_count(cudaError_t* err) {
  static DeviceOnce sms;
  int n = 0;
  *err = once_per_device(sms, &n, [](int dev, int* v) {
    return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
  });
  return *err == cudaSuccess ? n : 0;
}

// Dynamic shared memory of a TMA-form CTA, at least kRouterOneCta: the work
// split gives each SM one token group, and two CTAs of less than half the
// SM's 228 KB may share an SM while another idles (measured with the kernel
// launched while the previous launch's route-list kernels still held SMs:
// qwen3_30b route_align 0.200 ms per call in back-to-back graph replays,
// 0.130 ms with the floor).
constexpr uint32_t kRouterOneCta = 116u * 1024u;
inline uint32_t lg_smem(uint32_t b) { return b < kRouterOneCta ? kRouterOneCta : b; }

template <int TX>
cudaError_t launch_router_logits_tx(const RouteArgs& a, int vec4, int sms, cudaStream_t s) {
  constexpr int BN = TX * kRTN;
  constexpr int kTyMax = router_ty_max<TX>();
  const int gx = (a.E + BN - 1) / BN;
  const int groups = sms / gx > 0 ? sms / gx : 1;
  int bm = (a.N + groups - 1) / groups;
  int ty = ((bm + kRTM - 1) / kRTM + 3) / 4 * 4;
  if (ty > kTyMax) {  // more tokens than one CTA per SM can hold: several waves
    ty = kTyMax;
    bm = ty * kRTM;
  }
  static DeviceOnce smem_set;
  cudaError_t err = once_per_device(smem_set, nullptr, [&](int, int*) {
    cudaError_t e = cudaFuncSetAttribute(router_logits_kernel<TX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)router_smem_bytes(kTyMax * kRTM, BN, kTyMax));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(
        router_logits_tma_kernel<TX, 32, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)lg_smem(router_tma_layout<32, 4>(kTyMax * kRTM, BN, kTyMax * kRPad).total));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(
        router_logits_tma_kernel<TX, 64, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)lg_smem(router_tma_layout<64, 2>(kTyMax * kRTM, BN, kTyMax * kRPad).total));
  });
  if (err != cudaSuccess) return err;
  dim3 g(gx, (a.N + bm - 1) / bm);
  // TMA form: W_r rows a multiple of 16 bytes, boxes inside the tensors
  const bool tma = vec4 && a.E >= BN && a.err &&
                   (reinterpret_cast<uintptr_t>(a.x) & 15u) == 0;
  // stages of 64 contraction elements, two deep, for long rows (measured:
  // dsv3's router 0.40 -> 0.37 ms); 32 x 4 for shorter ones (H = 2048:
  // 0.167 vs 0.188 ms)
  const bool wide = a.H >= 4096;
  const uint32_t kb = wide ? 64u : 32u;
  CUtensorMap tmx, tmw;
  if (tma &&
      make_map_plain(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.x, (uint64_t)a.H, (uint64_t)a.N,
                     kb, (uint32_t)bm,
                     wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE) &&
      make_map_plain(&tmw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.wr, (uint64_t)a.E,
                     (uint64_t)a.H, BN, kb)) {
    if (wide)
      launch_pdl(router_logits_tma_kernel<TX, 64, 2>, dim3(g), dim3(ty * TX),
                 lg_smem(router_tma_layout<64, 2>(bm, BN, kTyMax * kRPad).total), s, tmx, tmw,
                 a.bias, a.ws.logits, a.N, a.n_dev, a.H, a.E, bm, a.err);
    else
      launch_pdl(router_logits_tma_kernel<TX, 32, 4>, dim3(g), dim3(ty * TX),
                 lg_smem(router_tma_layout<32, 4>(bm, BN, kTyMax * kRPad).total), s, tmx, tmw,
                 a.bias, a.ws.logits, a.N, a.n_dev, a.H, a.E, bm, a.err);
  } else {
    launch_pdl(router_logits_kernel<TX>, dim3(g), dim3(ty * TX), router_smem_bytes(bm, BN, ty), s, 
        a.x, a.wr, a.bias, a.ws.logits, a.N, a.n_dev, a.H, a.E, bm, vec4);
  }
  return cudaGetLastError();
}

// Expert tile width from E: the narrowest of 32, 64, 128, 256 experts that
// holds E (several tiles of 256 above that).
cudaError_t launch_router_logits(const RouteArgs& a, cudaStream_t s) {
  const int vec4 = (a.E % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.wr) & 15u) == 0);
  cudaError_t err = cudaSuccess;
  const int sms = router_sm_count(&err);
  if (sms <= 0) return err != cudaSuccess ? err : cudaErrorUnknown;
  const int64_t threads = (int64_t)a.N * ((a.E + 1) / 2);
  // Fewer than 32 experts: always (the tiled forms would run a 32-expert
  // tile, and without TMA: E = 16, N = 4096, H = 4096 took 0.238 ms of
  // route_align tiled, 0.101 ms here; E = 8, N = 16384, H = 2048 0.179 ->
  // 0.086 ms; E = 16, N = 16384, H = 4096 0.334 -> 0.244 ms).
  if (a.E < 32 || threads <= (int64_t)sms * 64) {
    const unsigned blocks = (unsigned)((threads + kRSmallThreads - 1) / kRSmallThreads);
    const bool vec2 = (a.E % 2 == 0) && ((reinterpret_cast<uintptr_t>(a.wr) & 7u) == 0);
    if (vec2)
      launch_pdl(router_logits_small_kernel<true>, dim3(blocks), dim3(kRSmallThreads), 0, s, 
          a.x, a.wr, a.bias, a.ws.logits, a.N, a.n_dev, a.H, a.E);
    else
      launch_pdl(router_logits_small_kernel<false>, dim3(blocks), dim3(kRSmallThreads), 0, s, 
          a.x, a.wr, a.bias, a.ws.logits, a.N, a.n_dev, a.H, a.E);
    return cudaGetLastError();
  }
  if (a.E <= 32) return launch_router_logits_tx<8>(a, vec4, sms, s);
  if (a.E <= 64) return launch_router_logits_tx<16>(a, vec4, sms, s);
  if (a.E <= 128) return launch_router_logits_tx<32>(a, vec4, sms, s);
  return launch_router_logits_tx<64>(a, vec4, sms, s);
}

// ---------------------------------------------------------------- R2
// One warp per token (32 warps, 32 tokens per CTA = one chunk). After the
// chunk's top-K, the CTA sorts its routes by expert (stable, so each expert's
// routes stay in token order) and records per-expert counts and offsets.
constexpr int kTopkWarps = 32;

// PER: expert values per lane (E <= 32 * PER), so the divisions and the pick
// loops run over the experts that exist (one instantiation each for 1, 2, 4
// and 8: with eight regardless of E, the 128-expert layer spent 5.6 us of its
// ~9 us per chunk issuing them)
template <int PER>
__global__ void __launch_bounds__(kTopkWarps * 32) router_topk_kernel(
    const float* __restrict__ logits, int Nmax, const int32_t* __restrict__ n_dev, int E, int K,
    int renorm, int32_t* __restrict__ topk_ids, float* __restrict__ topk_p,
    int32_t* __restrict__ chunk_counts, int32_t* __restrict__ chunk_lofs,
    int32_t* __restrict__ chunk_routes, uint32_t* __restrict__ chunk_keys,
    uint8_t* __restrict__ keep, int32_t* __restrict__ token_routes) {
  griddep_wait();  // launched after the kernel that writes this one's inputs
  griddep_launch_dependents();
  // exp(l - max) of every token of the chunk, one row per token (padded so
  // that lane l reading row l, column e, hits bank (l + e) % 32)
  __shared__ float zbuf[kTokensPerChunk][kMaxExperts + 1];
  __shared__ float ssum[kTokensPerChunk];
  __shared__ int32_t ids_s[kTokensPerChunk * kMaxTopK];
  __shared__ uint32_t pk_s[kTokensPerChunk * kMaxTopK];
  __shared__ uint32_t emask[kMaxExperts];  // bit tl: token tl of the chunk chose e
  __shared__ int32_t offs[kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int t0 = c * kTokensPerChunk;
  const int N = live_tokens(n_dev, Nmax);
  const int nt = min(kTokensPerChunk, N - t0);
  // every route starts dropped (no slot); the select kernel, which runs
  // after this grid, marks the kept ones. Routes of tokens past the live
  // count also get no expert.
  for (int i = threadIdx.x; i < kTokensPerChunk * K; i += blockDim.x) {
    const int t = t0 + i / K;
    if (t < Nmax) {
      keep[(size_t)t0 * K + i] = 0;
      token_routes[(size_t)t0 * K + i] = -1;
      if (t >= N) {
        topk_ids[(size_t)t0 * K + i] = -1;
        topk_p[(size_t)t0 * K + i] = 0.0f;
      }
    }
  }
  static_assert(PER * 32 <= kMaxExperts, "zbuf holds kMaxExperts values a token");
  static_assert(kTopkWarps == kTokensPerChunk, "one token of the chunk per warp");
  // one token per warp: z = exp(l - max) kept in registers and in zbuf
  const int tl = warp;
  float v[PER];
  if (tl < nt) {
    const float* l = logits + (size_t)(t0 + tl) * E;
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
        zbuf[tl][e] = v[j];
      }
    }
  }
  __syncthreads();
  // the softmax denominators, each the sequential fp32 sum over ascending e:
  // lane l of warp 0 sums token l's row, so one warp does all 32 sums at once
  if (warp == 0 && lane < nt) {
    // eight values loaded ahead of their (still sequential) adds, so each add
    // does not wait a shared-memory round trip
    float sacc = 0.0f;
    int e = 0;
    for (; e + 8 <= E; e += 8) {
      float z8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) z8[i] = zbuf[lane][e + i];
#pragma unroll
      for (int i = 0; i < 8; ++i) sacc = __fadd_rn(sacc, z8[i]);
    }
    for (; e < E; ++e) sacc = __fadd_rn(sacc, zbuf[lane][e]);
    ssum[lane] = sacc;
  }
  __syncthreads();
  if (tl < nt) {
    const int t = t0 + tl;
    const float s = ssum[tl];
#pragma unroll
    for (int j = 0; j < PER; ++j) v[j] = __fdiv_rn(v[j], s);
    // K picks of the largest p, ties to the lower e: warp max of the p bit
    // pattern (p >= 0, so bits order like values), then warp min of the expert
    // ids holding that maximum.
    uint32_t taken = 0;
    float d = 0.0f, my_p = 0.0f;
    int my_id = 0;
    for (int k = 0; k < K; ++k) {
      uint32_t best = 0;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u)) best = max(best, __float_as_uint(v[j]));
      }
      const uint32_t pmax = __reduce_max_sync(0xFFFFFFFFu, best);
      uint32_t mine = 0xFFFFFFFFu;
#pragma unroll
      for (int j = PER - 1; j >= 0; --j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u) && __float_as_uint(v[j]) == pmax) mine = (uint32_t)e;
      }
      const int eb = (int)__reduce_min_sync(0xFFFFFFFFu, mine);
      const float pb = __uint_as_float(pmax);
      if ((eb & 31) == lane) taken |= 1u << (eb >> 5);
      d = __fadd_rn(d, pb);  // pick order
      if (lane == k) { my_id = eb; my_p = pb; }
      if (lane == 0) ids_s[tl * K + k] = eb;
    }
    if (lane < K) {
      const float pr = renorm ? __fdiv_rn(my_p, d) : my_p;
      topk_ids[(size_t)t * K + lane] = my_id;
      topk_p[(size_t)t * K + lane] = pr;
      pk_s[tl * K + lane] = __float_as_uint(pr);
    }
  }
  // stable counting sort of the chunk's routes by expert. A token picks an
  // expert at most once, so expert e's routes are its tokens in the mask
  // (32 tokens per chunk), and a route's rank among them is the number of
  // earlier tokens in the mask.
  static_assert(kTokensPerChunk == 32, "one mask bit per token of a chunk");
  for (int e = threadIdx.x; e < E; e += blockDim.x) emask[e] = 0u;
  __syncthreads();
  const int nr = nt * K;
  for (int r = threadIdx.x; r < nr; r += blockDim.x) atomicOr(&emask[ids_s[r]], 1u << (r / K));
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int h = (e < E) ? __popc(emask[e]) : 0;
      int incl = h;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
      }
      if (e < E) offs[e] = run + incl - h;
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  __syncthreads();
  for (int r = threadIdx.x; r < nr; r += blockDim.x) {
    const int e = ids_s[r];
    const int tl = r / K;
    const int rank = __popc(emask[e] & ((1u << tl) - 1u));  // earlier tokens only
    chunk_routes[(size_t)t0 * K + offs[e] + rank] = t0 * K + r;
    chunk_keys[(size_t)t0 * K + offs[e] + rank] = pk_s[r];
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    chunk_counts[(size_t)c * E + e] = __popc(emask[e]);
    chunk_lofs[(size_t)c * E + e] = offs[e];
  }
}

// ---------------------------------------------------------------- R4
constexpr int kMaxChunks = kMaxTokens / kTokensPerChunk;
constexpr int kSelSmallThreads = 256;     // select CTA size for small batches
constexpr int kSelSmallMaxTokens = 2048;  // (one thread per chunk needs <= 8192)

// Exclusive scan of v over the CTA (THREADS threads, all must call).
template <int THREADS>
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
    const int w = (lane < (THREADS >> 5)) ? warp_tot[lane] : 0;
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

// One CTA per expert: assemble the expert's routes in token order from the
// chunk tables, select the `cap` highest p' (ties to the lower token) and
// write the expert's part of the route-list layout. A thread owns one chunk
// column, so THREADS >= the chunk count: 256 threads for batches of up to
// 2048 tokens (fewer CTA-wide barriers to wait on), 1024 above: MINB = 2
// (at most 32 registers a thread, so two such CTAs share an SM) when there
// are more experts than SMs, else MINB = 1 (64 registers: no spills, and the
// gather keeps eight chunk loads of a warp in flight instead of four).
template <int THREADS, int MINB>
__global__ void __launch_bounds__(THREADS, MINB) route_select_kernel(
    const int32_t* __restrict__ chunk_counts, const int32_t* __restrict__ chunk_lofs,
    const int32_t* __restrict__ chunk_routes, const uint32_t* __restrict__ chunk_keys, int Nmax,
    const int32_t* __restrict__ n_dev, int E, int K, int cap_num, int cap_den, int bm,
    int dropless, Ladder ladder, int s_max,
    uint8_t* __restrict__ keep, int32_t* __restrict__ expert_counts,
    int32_t* __restrict__ kept_counts, int32_t* __restrict__ sorted_slot_ids,
    int32_t* __restrict__ expert_ids, int32_t* __restrict__ block_start,
    int32_t* __restrict__ ntpp, int32_t* __restrict__ token_routes,
    int32_t* __restrict__ gemm_sched, float* __restrict__ slot_prob) {
  griddep_wait();  // launched after the kernel that writes this one's inputs
  griddep_launch_dependents();
  extern __shared__ uint32_t dyn[];
  // radix histograms: kHistReps copies, warp w counting into copy w % kHistReps
  // (a hot expert's keys crowd a few bins, and one copy serialised every warp
  // on the same shared-memory words)
  constexpr int kHistReps = 8;
  __shared__ int32_t hist[kHistReps][256];
  // the keys still in the running after the top 16 bits are fixed, gathered
  // during the third pass so the last pass reads only them (a hot expert's
  // 8174 keys leave a few hundred); kept only when they fit
  constexpr int kCBuf = 2048;
  __shared__ uint32_t cbuf[kCBuf];
  __shared__ int32_t s_nc;
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t s_cnt[kMaxChunks];
  __shared__ int32_t s_pos[kMaxChunks];
  __shared__ int32_t s_lo[kMaxChunks];
  __shared__ uint32_t s_prefix;
  __shared__ int32_t s_remaining;
  __shared__ int32_t s_total;
  __shared__ int32_t s_base;      // first slot of this expert
  __shared__ int32_t s_extent;    // slots of this expert
  __shared__ int32_t s_all;       // dropless: total padded extent
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = live_tokens(n_dev, Nmax);
  // capacity of the live batch: cap = ceil(N*K*F/E) (capped at N), its region
  // roundup(cap, bm); dropless keeps every route
  int cap = N, cpad = 0;
  if (!dropless) {
    const long long num = (long long)N * K * cap_num, den = (long long)E * cap_den;
    const long long cc = (num + den - 1) / den;
    cpad = (int)((cc + bm - 1) / bm * bm);
    cap = (int)(cc < N ? cc : N);
  }
  const int C = (N + kTokensPerChunk - 1) / kTokensPerChunk;
  uint32_t* keys = dyn;                                     // p' bits, token order
  int32_t* rids = reinterpret_cast<int32_t*>(dyn + Nmax);  // route index t*K+k
  // column e of the chunk tables -> positions in the expert's list
  // this thread's chunk: the expert's route count in it and where they start
  // in the chunk's sorted list (both read here, before any barrier)
  const int cnt = (tid < C) ? min(max(chunk_counts[(size_t)tid * E + e], 0), kTokensPerChunk) : 0;
  const int lo0 = (tid < C) ? min(max(chunk_lofs[(size_t)tid * E + e], 0), kTokensPerChunk * K) : 0;
  const int pos0 = block_exclusive_scan<THREADS>(cnt, warp_tot);
  if (tid < C) { s_cnt[tid] = cnt; s_pos[tid] = pos0; s_lo[tid] = lo0; }
  if (tid == C - 1) s_total = pos0 + cnt;
  if (C == 0 && tid == 0) s_total = 0;
  __syncthreads();
  const int n = min(s_total, N);
  int base = e * cpad, extent = cpad;  // capacity mode: fixed regions
  if (dropless) {
    // every expert's count (column sums of the chunk table), its extent from
    // the ladder, and the exclusive scan of the extents up to this expert
    __syncthreads();
    const long long R = (long long)N * K;
    int ext = 0;
    if (tid < E) {
      int cnt_e = 0;
      for (int c2 = 0; c2 < C; ++c2) cnt_e += chunk_counts[(size_t)c2 * E + tid];
      ext = -1;
      for (int j = 0; j < ladder.len && ext < 0; ++j) {
        const long long num = (long long)ladder.num[j] * R, den = (long long)ladder.den * E;
        long long rung = (num + den - 1) / den;
        rung = (rung + bm - 1) / bm * bm;
        if (cnt_e <= rung) ext = (int)rung;
      }
      if (ext < 0) ext = (cnt_e + bm - 1) / bm * bm;
    }
    const int before = block_exclusive_scan<THREADS>(ext, warp_tot);
    if (tid == e) {
      s_base = before;
      s_extent = ext;
    }
    if (tid == E - 1) s_all = before + ext;
    __syncthreads();
    base = s_base;
    extent = s_extent;
  }
  // the expert's routes of chunk cc are lanes 0..m-1 (at most one per token
  // of the chunk); a warp loads four of its chunks before storing any, so
  // their load round trips overlap
  {
    constexpr int kG = (THREADS >= 1024 && MINB == 1) ? 8 : 4;
    for (int cc0 = warp; cc0 < C; cc0 += kG * (THREADS / 32)) {
      int rv[kG], at_[kG];
      uint32_t kv[kG];
#pragma unroll
      for (int g = 0; g < kG; ++g) {
        const int cc = cc0 + g * (THREADS / 32);
        at_[g] = -1;
        if (cc < C) {
          const int lo = s_lo[cc];
          const int64_t chunk_base = (int64_t)cc * kTokensPerChunk * K;
          const int m = (int)min((int64_t)min(s_cnt[cc], kTokensPerChunk * K - lo),
                                 (int64_t)N * K - chunk_base - lo);
          const int at = s_pos[cc] + lane;
          if (lane < m && at < n) {
            rv[g] = chunk_routes[chunk_base + lo + lane];
            kv[g] = chunk_keys[chunk_base + lo + lane];
            at_[g] = at;
          }
        }
      }
#pragma unroll
      for (int g = 0; g < kG; ++g) {
        if (at_[g] >= 0) {
          int r = rv[g];
          if ((unsigned)r >= (unsigned)(N * K)) r = 0;  // never taken when the tables agree
          rids[at_[g]] = r;
          keys[at_[g]] = kv[g];
        }
      }
    }
  }
  __syncthreads();
  const bool select = n > cap;
  uint32_t thr = 0;
  int needed = 0;
  if (select) {
    // the cap-th largest key, 8 bits at a time from the top
    uint32_t prefix = 0, mask = 0;
    int remaining = cap;
    int nc = -1;  // keys in cbuf (the last pass's source), -1: read them all
    if (tid == 0) s_nc = 0;  // (the first pass's barriers order this before any append)
    int32_t* my_hist = hist[warp % kHistReps];
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < kHistReps * 256; i += THREADS) (&hist[0][0])[i] = 0;
      __syncthreads();
      const uint32_t* src = nc >= 0 ? cbuf : keys;
      const int ns = nc >= 0 ? nc : n;
      for (int base = warp * 32; base < ns; base += THREADS) {
        const int i = base + lane;
        const uint32_t k = (i < ns) ? src[i] : 0u;
        const bool cand = (i < ns) && ((k & mask) == prefix);
        const int bin = cand ? (int)((k >> shift) & 255u) : -1;
        if (MINB == 1 && shift == 8) {  // (the 32-register form would spill)
          // keep the candidates (top 16 bits fixed) for the last pass
          const uint32_t cb = __ballot_sync(0xFFFFFFFFu, cand);
          int at = 0;
          if (lane == 0 && cb != 0u) at = atomicAdd(&s_nc, __popc(cb));
          at = __shfl_sync(0xFFFFFFFFu, at, 0) + __popc(cb & ((1u << lane) - 1u));
          if (cand && at < kCBuf) cbuf[at] = k;
        }
        if (shift == 24) {
          // the top byte (sign and high exponent bits) of probabilities takes
          // one or two values: aggregate the lanes of each bin first
          const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bin);
          if (cand && lane == __ffs(peers) - 1) atomicAdd(&my_hist[bin], __popc(peers));
        } else if (cand) {
          // lower digits spread over many bins: one atomic per lane (grouping
          // lanes first measured 3x slower on a hot expert's 8174 keys)
          atomicAdd(&my_hist[bin], 1);
        }
      }
      __syncthreads();
      if (warp == 0) {
        // digit holding the remaining-th largest key: lane l owns bins
        // 255-8l .. 248-8l (descending); a warp scan of the lane sums finds
        // the lane, a short walk finds the bin
        int h[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          h[j] = 0;
#pragma unroll
          for (int rr = 0; rr < kHistReps; ++rr) h[j] += hist[rr][255 - 8 * lane - j];
          sum += h[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += u;
        }
        const int before = incl - sum;
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, before < remaining && incl >= remaining);
        if (hit != 0u && lane == __ffs(hit) - 1) {
          int cum = before, j = 0;
          for (; j < 7; ++j) {
            if (cum + h[j] >= remaining) break;
            cum += h[j];
          }
          s_remaining = remaining - cum;
          s_prefix = prefix | ((uint32_t)(255 - 8 * lane - j) << shift);
        }
      }
      __syncthreads();
      remaining = s_remaining;
      prefix = s_prefix;
      mask |= 0xFFu << shift;
      if (MINB == 1 && shift == 8) nc = s_nc <= kCBuf ? s_nc : -1;
    }
    thr = prefix;
    needed = remaining;  // how many keys equal to thr are kept (lowest tokens first)
  }
  // Warp w owns the contiguous segment [s0, s1) of the list (token order) and
  // visits it 32 elements at a time, lane l the l-th: shared-memory reads
  // fall on distinct banks and the kept slots of a step are consecutive.
  // Ties with the threshold are kept lowest token first: a tie's rank is the
  // ties before it (the warps before, then ballots within the segment).
  constexpr int kWarps = THREADS / 32;
  const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int s0 = min(n, warp * seg), s1 = min(n, s0 + seg);
  const uint32_t lt = (1u << lane) - 1u;  // lanes below this one
  // One scan gives both prefixes a warp needs: ties before it (tie_base) and
  // keys above the threshold before it (gt_base), packed as ties | gt << 16
  // (each at most 24576). The kept routes before warp w are gt_base +
  // min(needed, tie_base): every key above the threshold, and the lowest
  // tokens' ties up to the `needed` the select left.
  int ties = 0, gt = 0;
  if (select)
    for (int i = s0 + lane; i < s1; i += 32) {
      const uint32_t k = keys[i];
      ties += (k == thr);
      gt += (k > thr);
    }
  const int packed = __reduce_add_sync(0xFFFFFFFFu, ties | (gt << 16));
  const int before = __shfl_sync(
      0xFFFFFFFFu, block_exclusive_scan<THREADS>(lane == 0 ? packed : 0, warp_tot), 0);
  const int tie_base = before & 0xFFFF;
  int pos = select ? (before >> 16) + min(needed, tie_base) : s0;
  // the keep decision of element i (all lanes of the warp take the step)
  auto keep_step = [&](int i, int& tie_rank) -> bool {
    if (!select) return i < s1;
    const uint32_t k = i < s1 ? keys[i] : 0u;
    const bool tie = i < s1 && k == thr;
    const uint32_t tb = __ballot_sync(0xFFFFFFFFu, tie);
    const bool kp = i < s1 && (k > thr || (tie && tie_rank + __popc(tb & lt) < needed));
    tie_rank += __popc(tb);
    return kp;
  };
  // second walk: same decisions, now writing the layout
  {
    int tie_rank = tie_base;
    for (int i = s0 + lane; i - lane < s1; i += 32) {
      const bool kp = keep_step(i, tie_rank);
      const uint32_t kb = __ballot_sync(0xFFFFFFFFu, kp);
      if (kp) {  // a dropped route keeps the top-K kernel's keep = 0, no slot
        const int r = rids[i];
        const int slot = base + pos + __popc(kb & lt);
        sorted_slot_ids[slot] = r / K;
        slot_prob[slot] = __uint_as_float(keys[i]);  // the key is p' (its bits)
        token_routes[r] = slot;
        keep[r] = 1;
      }
      pos += __popc(kb);
    }
  }
  const int kept_e = select ? cap : n;
  for (int sl = kept_e + tid; sl < extent; sl += THREADS) {
    sorted_slot_ids[base + sl] = Nmax;  // sentinel: one past the static token bound
    slot_prob[base + sl] = 0.0f;
  }
  const int nb = extent / bm;
  for (int b = tid; b < nb; b += THREADS)
    expert_ids[(size_t)base / bm + b] = (b * bm < kept_e) ? e : -1;
  if (e == E - 1) {
    // slots past the padded total up to the allocated bound (dropless, or a
    // live batch below the static bound): sentinel / -1
    const int used = dropless ? s_all : E * cpad;
    for (int sl = used + tid; sl < s_max; sl += THREADS) {
      sorted_slot_ids[sl] = Nmax;
      slot_prob[sl] = 0.0f;
    }
    for (int b = used / bm + tid; b < s_max / bm; b += THREADS) expert_ids[b] = -1;
  }
  if (tid == 0) {
    block_start[e] = base / bm;
    expert_counts[e] = n;
    kept_counts[e] = kept_e;
    if (e == 0) {
      if (!dropless) *ntpp = E * cpad;
      for (int i = 0; i < 4; ++i) gemm_sched[i] = 0;
    }
    if (dropless && e == E - 1) *ntpp = s_all;
  }
}


// ---------------------------------------------------------------- router backward
// The gradient of the routing probabilities p' (dprob [N,K]) through top-K
// renormalisation and the softmax to the logits, with the chosen experts of
// the forward held fixed (the selection is piecewise constant). One warp per
// token recomputes p exactly as the forward does (same exp, ascending-e sum,
// IEEE divide), then, with the chosen experts e_k:
//   renorm: d = sum_k p[e_k], c = sum_k dprob_k p[e_k]/d, g_k = (dprob_k - c)/d
//   else:   g_k = dprob_k
//   s = sum_k g_k p[e_k];  dl[e] = p[e] (g[e] - s), g[e] = 0 for the others.
// Besides dl it writes the bf16 split copy dls [N, 2*Ep] (Ep = E rounded up to
// 64): dls[t,e] = hi = bf16(dl), dls[t,Ep+e] = bf16(dl - hi), zero for
// E <= e < Ep; the tensor-core contractions of the router backward read it.
constexpr int kDlWarps = 8;

// Reads the logits from `lg` and writes dl to `ld`, which may be the same
// buffer (each lane reads its entries before it writes them).
// PER: values per lane, Ep <= 32 * PER (the split copy's padded width)
template <int PER>
__global__ void __launch_bounds__(kDlWarps * 32) router_dlogits_kernel(
    const float* lg, float* ld, int N, int E, int K, int renorm,
    const int32_t* __restrict__ topk_ids, const float* __restrict__ dprob,
    uint16_t* __restrict__ dls, int Ep) {
  __shared__ float pbuf[kDlWarps][kMaxExperts];
  __shared__ float gk_s[kDlWarps][kMaxTopK];
  __shared__ int32_t id_s[kDlWarps][kMaxTopK];
  __shared__ float s_s[kDlWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kDlWarps + warp;
  if (t >= N) return;
  static_assert(PER * 32 <= kMaxExperts, "pbuf holds kMaxExperts values a token");
  const float* l = lg + (size_t)t * E;
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
      pbuf[warp][e] = v[j];
    }
  }
  __syncwarp();
  float sum = 0.0f;
  if (lane == 0) {  // ascending e; eight terms loaded ahead of their adds
    int e = 0;
    for (; e + 8 <= E; e += 8) {
      float z8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) z8[i] = pbuf[warp][e + i];
#pragma unroll
      for (int i = 0; i < 8; ++i) sum = __fadd_rn(sum, z8[i]);
    }
    for (; e < E; ++e) sum = __fadd_rn(sum, pbuf[warp][e]);
  }
  sum = __shfl_sync(0xFFFFFFFFu, sum, 0);
  __syncwarp();
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    v[j] = __fdiv_rn(v[j], sum);
    if (e < E) pbuf[warp][e] = v[j];
  }
  if (lane < K) id_s[warp][lane] = topk_ids[(size_t)t * K + lane];
  __syncwarp();
  if (lane == 0) {
    float d = 0.0f, c = 0.0f, sg = 0.0f;
    if (renorm) {
      for (int k = 0; k < K; ++k) d = __fadd_rn(d, pbuf[warp][id_s[warp][k]]);
      for (int k = 0; k < K; ++k)
        c = __fadd_rn(c, __fmul_rn(dprob[(size_t)t * K + k], __fdiv_rn(pbuf[warp][id_s[warp][k]], d)));
    }
    for (int k = 0; k < K; ++k) {
      const float dp = dprob[(size_t)t * K + k];
      const float g = renorm ? __fdiv_rn(__fsub_rn(dp, c), d) : dp;
      gk_s[warp][k] = g;
      sg = __fadd_rn(sg, __fmul_rn(g, pbuf[warp][id_s[warp][k]]));
    }
    s_s[warp] = sg;
  }
  __syncwarp();
  const float sg = s_s[warp];
  uint16_t* split = dls + (size_t)t * 2 * Ep;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    if (e >= Ep) continue;
    uint16_t hi = 0, lo = 0;
    if (e < E) {
      float g = 0.0f;
      for (int k = 0; k < K; ++k)
        if (id_s[warp][k] == e) g = gk_s[warp][k];
      const float d = __fmul_rn(v[j], __fsub_rn(g, sg));
      ld[(size_t)t * E + e] = d;
      const __nv_bfloat16 bh = __float2bfloat16_rn(d);
      hi = __bfloat16_as_ushort(bh);
      lo = __bfloat16_as_ushort(__float2bfloat16_rn(__fsub_rn(d, __bfloat162float(bh))));
    }
    split[e] = hi;
    split[Ep + e] = lo;
  }
}

// dW_r = sum of the splits' partials in split order.
__global__ void router_dwr_reduce_kernel(const float* __restrict__ part, int splits, int64_t n,
                                         float* __restrict__ dwr) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float acc = 0.0f;
  for (int z = 0; z < splits; ++z) acc = __fadd_rn(acc, part[(size_t)z * n + i]);
  dwr[i] = acc;
}

// dbias[e] = sum_t dl[t,e]: each of 256 threads sums a strided set of tokens
// in ascending order, then a fixed-order tree over the threads.
__global__ void __launch_bounds__(256) router_dbias_kernel(const float* __restrict__ dl, int N,
                                                           int E, float* __restrict__ dbias) {
  __shared__ float red[256];
  const int e = blockIdx.x;
  float acc = 0.0f;
  for (int t = threadIdx.x; t < N; t += 256) acc = __fadd_rn(acc, dl[(size_t)t * E + e]);
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] = __fadd_rn(red[threadIdx.x], red[threadIdx.x + w]);
    __syncthreads();
  }
  if (threadIdx.x == 0) dbias[e] = red[0];
}

}  // namespace

int launch_route(const RouteArgs& a, cudaStream_t s) {
  int launched = 0;
  const int C = (a.N + kTokensPerChunk - 1) / kTokensPerChunk;
  if (a.N > 0) {
    const cudaError_t e1 = launch_router_logits(a, s);
    if (e1 != cudaSuccess) return -(int)e1;
    ++launched;
    auto topk = a.E <= 32    ? router_topk_kernel<1>
                : a.E <= 64  ? router_topk_kernel<2>
                : a.E <= 128 ? router_topk_kernel<4>
                             : router_topk_kernel<8>;
    launch_pdl(topk, dim3(C), dim3(kTopkWarps * 32), 0, s, a.ws.logits, a.N, a.n_dev, a.E, a.K,
               a.renorm, a.topk_ids, a.topk_p, a.ws.chunk_counts, a.ws.chunk_lofs,
               a.ws.chunk_routes, a.ws.chunk_keys, a.keep, a.token_routes);
    ++launched;
  }
  const size_t dyn = (size_t)a.N * 8;
  cudaError_t err = cudaSuccess;
  {
    // raise the kernel's dynamic shared-memory limit once per device
    static DeviceOnce smem_set;
    err = once_per_device(smem_set, nullptr, [](int, int*) {
      cudaError_t e = cudaFuncSetAttribute(route_select_kernel<1024, 2>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kMaxTokens * 8);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(route_select_kernel<1024, 1>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxTokens * 8);
      if (e != cudaSuccess) return e;
      return cudaFuncSetAttribute(route_select_kernel<kSelSmallThreads, 1>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSelSmallThreads * kTokensPerChunk * 8);
    });
    if (err != cudaSuccess) return -(int)err;
  }
  // the narrow CTA for batches of at most 2048 tokens: an expert can hold every
  // token, and above that many keys per thread (a Zipf-skewed 8192-token batch:
  // route_align 0.168 -> 0.195 ms) cost more than the barriers save
  const bool small = a.N <= kSelSmallMaxTokens;
  const int sms = router_sm_count(&err);
  if (sms <= 0) return -(int)(err != cudaSuccess ? err : cudaErrorUnknown);
  launch_pdl(small ? route_select_kernel<kSelSmallThreads, 1>
                   : (a.E <= sms ? route_select_kernel<1024, 1> : route_select_kernel<1024, 2>),
             dim3(a.E), dim3(small ? kSelSmallThreads : 1024), dyn, s, a.ws.chunk_counts,
             a.ws.chunk_lofs, a.ws.chunk_routes, a.ws.chunk_keys, a.N, a.n_dev, a.E, a.K,
             a.cap_num, a.cap_den, a.bm, a.dropless, a.ladder, (int)a.s_max, a.keep,
             a.expert_counts, a.kept_counts, a.sorted_slot_ids, a.expert_ids, a.block_start,
             a.ntpp, a.token_routes, a.gemm_sched, a.slot_prob);
  ++launched;
  err = cudaGetLastError();
  if (err != cudaSuccess) return -(int)err;
  return launched;
}

int launch_router_backward(const RouterBwdArgs& a, cudaStream_t s) {
  if (a.N <= 0) return 0;
  int launched = 0;
  // the forward's logits, or recomputed exactly as the forward (into the dl
  // buffer)
  RouteArgs r{};
  r.N = a.N;
  r.H = a.H;
  r.E = a.E;
  r.x = a.x;
  r.wr = a.wr;
  r.bias = a.bias;
  r.ws.logits = a.dl;
  r.err = a.err;
  cudaError_t err = cudaSuccess;
  if (!a.logits) {
    err = launch_router_logits(r, s);
    if (err != cudaSuccess) return -(int)err;
    ++launched;
  }
  // W_r's split copy does not depend on dl
  int rc = launch_router_split_w(a.wr, a.H, a.E, a.wrs, s);
  if (rc < 0) return rc;
  launched += rc;
  const int ep = router_split_cols(a.E) / 2;  // E rounded up to 64
  auto dlogits = ep <= 64 ? router_dlogits_kernel<2> : ep <= 128 ? router_dlogits_kernel<4>
                                                                 : router_dlogits_kernel<8>;
  dlogits<<<(a.N + kDlWarps - 1) / kDlWarps, kDlWarps * 32, 0, s>>>(
      a.logits ? a.logits : a.dl, a.dl, a.N, a.E, a.K, a.renorm, a.topk_ids, a.dprob, a.dls, ep);
  ++launched;
  rc = launch_router_dwr_mma(a.x, a.dls, a.N, a.H, a.E, a.part, a.err, s);
  if (rc < 0) return rc;
  launched += rc;
  const int splits = router_bwd_splits(a.N, a.H, a.E);
  const int64_t n = (int64_t)a.H * a.E;
  router_dwr_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a.part, splits, n, a.dwr);
  ++launched;
  if (a.dbias) {
    router_dbias_kernel<<<a.E, 256, 0, s>>>(a.dl, a.N, a.E, a.dbias);
    ++launched;
  }
  rc = launch_router_dx_mma(a.dls, a.wrs, a.N, a.H, a.E, a.dx, a.err, s);
  if (rc < 0) return rc;
  launched += rc;
  err = cudaGetLastError();
  return err == cudaSuccess ? launched : -(int)err;
}

}  // namespace moe
