// Router backward contractions on the 5th-generation tensor cores:
//   dW_r[h,e] = sum_t x[t,h] dl[t,e]       fp32 out [H,E]
//   dx[t,h]  += sum_e dl[t,e] W_r[h,e]     bf16 in/out [N,H], summed in fp32,
//                                          rounded to bf16 once
// (dl = d loss / d logits of the router, fp32 [N,E]; W_r fp32 [H,E]; x bf16.)
//
// Precision. dl and W_r are fp32; each is carried as two bf16 parts, v = hi +
// lo with hi = bf16(v) and lo = bf16(v - hi) (v - hi is exact in fp32), which
// keeps 16 significant bits (the split of Henry, Tang and Heinecke, "Leveraging
// the bfloat16 artificial intelligence datatype for higher-precision
// computations", ARITH 2019). A product of two bf16 values is exact in the
// fp32 accumulator, so
//   dW_r = x^T hi + x^T lo                   (x is bf16 already)
//   dx  += hi hi_w + lo hi_w + hi lo_w       (lo lo_w, below 2^-16 of the
//                                             terms, is left out)
// match the fp32 sums up to accumulation order. The split copies are
// [rows, 2*Ep] bf16, hi in columns [0, Ep) and lo in [Ep, 2*Ep), where Ep is E
// rounded up to a multiple of 64 with zero padding: every 64-column block is
// one 128-byte swizzle atom, and padded experts contribute zeros.
//
// dW_r: tiles of 128 rows of h (UMMA M, read MN-major from x, h contiguous) x
// Ep experts (UMMA N, MN-major from the split dl, e contiguous), contracted
// over a split of the tokens in stages of 64; each split writes its partial
// sum, and a separate pass adds the splits in split order (deterministic).
// dx: tiles of 128 tokens (M) x 128 rows of h (N), K = Ep in stages of 64
// experts, both operands K-major; persistent CTAs walk the tiles, each tile
// of dx fetched by TMA ahead of its epilogue, which reads it back from shared
// memory, adds the accumulator and stores the rounded sum.
//
// Warp roles (192 threads): warp 0 issues the TMA copies, warp 1 owns TMEM and
// issues the MMAs (one lane), warps 2-5 drain TMEM (warp w reads lanes
// 32*(w%4)..+31). Every wait is bounded and records a bit in the error word.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "moe_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

constexpr int kRbThreads = 192;
constexpr int kRbK = 64;             // tokens (dW_r) or experts (dx) per stage
constexpr int kRbMaxStages = 4;
constexpr uint32_t kRbChunk = 8192;  // one MN-major chunk: 64 K rows x 128 bytes
constexpr int kRbAssumedSms = 152;   // sizes the dW_r token splits (workspace)

__host__ __device__ constexpr int round64(int v) { return (v + 63) / 64 * 64; }

__device__ __forceinline__ uint32_t tmem_cols_for(int n) {
  return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : 256u;
}

// ---------------------------------------------------------------- dW_r
struct DwrMmaParams {
  int N, H, E, Ep;
  int tps;                 // tokens per split, a multiple of 64
  int stages;
  uint32_t stage_bytes;    // 16 KiB of x + 2 * Ep/64 chunks of the split dl
  float* part;             // [splits, H, E]
  uint32_t* err;
};

__host__ __device__ inline uint32_t dwr_stage_bytes(int Ep) {
  return 2u * kRbChunk + 2u * (uint32_t)(Ep / 64) * kRbChunk;
}

__host__ inline int dwr_stages(int Ep) {
  // about 110 KiB per CTA lets two CTAs share an SM; never fewer than 2 stages
  int s = (int)((110u * 1024u) / dwr_stage_bytes(Ep));
  return s < 2 ? 2 : s > kRbMaxStages ? kRbMaxStages : s;
}

__global__ void __launch_bounds__(kRbThreads, 1)
    router_dwr_mma_kernel(const __grid_constant__ CUtensorMap tmX,
                          const __grid_constant__ CUtensorMap tmL, const DwrMmaParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kRbMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kRbMaxStages];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int h0 = blockIdx.x * 128;
  const int ta = blockIdx.y * p.tps;
  const int tb = min(p.N, ta + p.tps);
  const int kt_n = tb > ta ? (tb - ta + kRbK - 1) / kRbK : 0;
  const uint32_t ncols = tmem_cols_for(p.Ep);
  const uint32_t b_off = 2u * kRbChunk;                     // split dl after x
  const uint32_t lo_off = (uint32_t)(p.Ep / 64) * kRbChunk;  // lo chunks after hi

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&acc_bar), 1);
    mbar_fence_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmL);
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_base_s), ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // x is read once over the grid; the split dl by every row tile
    const uint64_t pol_x = policy_evict_first(), pol_l = policy_evict_last();
    for (int kt = 0; kt < kt_n; ++kt) {
      const int s = kt % p.stages;
      const uint32_t u = (uint32_t)(kt / p.stages);
      if (kt >= p.stages &&
          !mbar_wait_warp(smem_u32(&empty_bar[s]), (u & 1u) ^ 1u, p.err, kErrWaitEmpty))
        break;
      if (lane == 0) {
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t st = sbase + (uint32_t)s * p.stage_bytes;
        const int t = ta + kt * kRbK;
        mbar_arrive_expect_tx(fb, p.stage_bytes);
        tma_load_3d(st, &tmX, 0, t, h0 / 64, fb, pol_x);                 // 2 chunks of h
        tma_load_3d(st + b_off, &tmL, 0, t, 0, fb, pol_l);               // hi
        tma_load_3d(st + b_off + lo_off, &tmL, 0, t, p.Ep / 64, fb, pol_l);  // lo
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, p.Ep) | kIdescAMnMajor | kIdescBMnMajor;
    for (int kt = 0; kt < kt_n; ++kt) {
      const int s = kt % p.stages;
      const uint32_t u = (uint32_t)(kt / p.stages);
      if (!mbar_wait_warp(smem_u32(&full_bar[s]), u & 1u, p.err, kErrWaitFull)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t st = sbase + (uint32_t)s * p.stage_bytes;
#pragma unroll
        for (int kk = 0; kk < kRbK / 16; ++kk) {  // 16 tokens = 16 rows of 128 bytes
          const uint64_t ad = sdesc_sw128_mn(st + (uint32_t)kk * 2048u);
          umma_bf16(tmem, ad, sdesc_sw128_mn(st + b_off + (uint32_t)kk * 2048u), idesc,
                    (kt | kk) != 0);
          umma_bf16(tmem, ad, sdesc_sw128_mn(st + b_off + lo_off + (uint32_t)kk * 2048u), idesc,
                    1u);
        }
        umma_commit(smem_u32(&empty_bar[s]));
      }
      __syncwarp();
    }
    if (lane == 0) umma_commit(smem_u32(&acc_bar));  // also after an abort
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // lane = row h of the tile, columns = experts; a split with no token
    // writes zeros
    const int q = warp & 3;
    const int h = h0 + q * 32 + lane;
    float* dst = p.part + ((size_t)blockIdx.y * p.H + h) * p.E;
    const bool vec = (p.E & 3) == 0;
    if (kt_n == 0) {
      for (int e = 0; e < p.E; ++e) dst[e] = 0.0f;
    } else if (mbar_wait_warp(smem_u32(&acc_bar), 0u, p.err, kErrWaitAccum)) {
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
      for (int c = 0; c < p.Ep; c += 16) {
        uint32_t v[16];
        tmem_ld16(tl + (uint32_t)c, v);
        tmem_ld_wait();
        if (vec && c + 16 <= p.E) {
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(dst + c + j) =
                make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                            __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < p.E) dst[c + j] = __uint_as_float(v[j]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ---------------------------------------------------------------- dx
// Persistent: one CTA per SM walks the (h slice, token tile) items
// w = blockIdx.x, blockIdx.x + gridDim.x, ... (item w: rows h0 = 128 (w % h
// tiles), tokens t0 = 128 (w / h tiles)). Per item the producer loads the dx
// tile into one of three tile buffers and the Ep/64 operand stages into a
// ring of two; the MMA warp accumulates into one of two TMEM accumulators; so
// the epilogue of one item overlaps the loads and MMAs of the next ones.
struct DxMmaParams {
  int N, H, Ep;
  int h_tiles, items;
  uint16_t* dx;
  uint32_t* err;
};

constexpr uint32_t kDxOpBytes = 128u * 128u;        // one 128-row x 64-column bf16 box
constexpr uint32_t kDxStageBytes = 4u * kDxOpBytes;  // A hi, A lo, B hi, B lo
constexpr uint32_t kDxTileBytes = 2u * kDxOpBytes;   // dx: 128 tokens x 128 h
constexpr int kDxStages = 2;
constexpr int kDxTiles = 3;  // dx tiles in flight (loaded ahead of their epilogue)
constexpr uint32_t kDxSmemBytes = kDxStages * kDxStageBytes + kDxTiles * kDxTileBytes + 1024u;

__global__ void __launch_bounds__(kRbThreads, 1)
    router_dx_mma_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmD, const DxMmaParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kDxStages];
  __shared__ __align__(8) uint64_t empty_bar[kDxStages];
  __shared__ __align__(8) uint64_t dx_full[kDxTiles];
  __shared__ __align__(8) uint64_t dx_empty[kDxTiles];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t dxs0 = sbase + (uint32_t)kDxStages * kDxStageBytes;
  const int kb_n = p.Ep / kRbK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDxStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < kDxTiles; ++b) {
      mbar_init(smem_u32(&dx_full[b]), 1);
      mbar_init(smem_u32(&dx_empty[b]), 4);   // one arrival per epilogue warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 4);
    }
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_base_s), 256u);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_d = policy_evict_first(), pol_w = policy_evict_last();
    uint32_t g = 0;  // operand stages issued
    bool ok = true;
    for (int i = 0, w = blockIdx.x; ok && w < p.items; ++i, w += gridDim.x) {
      const int h0 = (w % p.h_tiles) * 128, t0 = (w / p.h_tiles) * 128;
      const int b = i % kDxTiles;
      const uint32_t u = (uint32_t)(i / kDxTiles);
      if (i >= kDxTiles &&
          !mbar_wait_warp(smem_u32(&dx_empty[b]), (u & 1u) ^ 1u, p.err, kErrWaitEmpty))
        break;
      if (lane == 0) {
        const uint32_t db = smem_u32(&dx_full[b]);
        const uint32_t dst = dxs0 + (uint32_t)b * kDxTileBytes;
        mbar_arrive_expect_tx(db, kDxTileBytes);
        tma_load_2d(dst, &tmD, h0, t0, db, pol_d);
        tma_load_2d(dst + kDxOpBytes, &tmD, h0 + 64, t0, db, pol_d);
      }
      __syncwarp();
      for (int kb = 0; kb < kb_n; ++kb, ++g) {
        const int s = (int)(g % kDxStages);
        const uint32_t us = g / kDxStages;
        if (g >= (uint32_t)kDxStages &&
            !mbar_wait_warp(smem_u32(&empty_bar[s]), (us & 1u) ^ 1u, p.err, kErrWaitEmpty)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&full_bar[s]);
          const uint32_t st = sbase + (uint32_t)s * kDxStageBytes;
          const int k = kb * kRbK;
          mbar_arrive_expect_tx(fb, kDxStageBytes);
          tma_load_2d(st, &tmA, k, t0, fb, pol_w);                           // dl hi
          tma_load_2d(st + kDxOpBytes, &tmA, p.Ep + k, t0, fb, pol_w);       // dl lo
          tma_load_2d(st + 2u * kDxOpBytes, &tmB, k, h0, fb, pol_w);         // W_r hi
          tma_load_2d(st + 3u * kDxOpBytes, &tmB, p.Ep + k, h0, fb, pol_w);  // W_r lo
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, 128);
    uint32_t g = 0;
    bool ok = true;
    for (int i = 0, w = blockIdx.x; ok && w < p.items; ++i, w += gridDim.x) {
      const int a = i & 1;
      const uint32_t u = (uint32_t)(i >> 1);
      if (i >= 2 &&
          !mbar_wait_warp(smem_u32(&acc_empty[a]), (u & 1u) ^ 1u, p.err, kErrWaitAccum))
        break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)a * 128u;
      for (int kb = 0; kb < kb_n; ++kb, ++g) {
        const int s = (int)(g % kDxStages);
        const uint32_t us = g / kDxStages;
        if (!mbar_wait_warp(smem_u32(&full_bar[s]), us & 1u, p.err, kErrWaitFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t st = sbase + (uint32_t)s * kDxStageBytes;
#pragma unroll
          for (int kk = 0; kk < kRbK / 16; ++kk) {  // 16 experts = 32 bytes of a row
            const uint32_t o = (uint32_t)kk * 32u;
            const uint64_t ahi = sdesc_sw128(st + o), alo = sdesc_sw128(st + kDxOpBytes + o);
            const uint64_t bhi = sdesc_sw128(st + 2u * kDxOpBytes + o);
            const uint64_t blo = sdesc_sw128(st + 3u * kDxOpBytes + o);
            umma_bf16(d, ahi, bhi, idesc, (kb | kk) != 0);
            umma_bf16(d, alo, bhi, idesc, 1u);
            umma_bf16(d, ahi, blo, idesc, 1u);
          }
          umma_commit(smem_u32(&empty_bar[s]));
        }
        __syncwarp();
      }
      if (lane == 0) umma_commit(smem_u32(&acc_full[a]));  // also after an abort
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // lane = token row r of the tile; 16 columns of h at a time: the old dx
    // from the 128-byte-swizzled tile (16-byte unit j of row r at
    // r*128 + ((j ^ (r%8)) * 16) within each 64-column half), plus the
    // accumulator, rounded once, stored 32 bytes per lane
    const int q = warp & 3;
    const int r = q * 32 + lane;
    for (int i = 0, w = blockIdx.x; w < p.items; ++i, w += gridDim.x) {
      const int h0 = (w % p.h_tiles) * 128, t0 = (w / p.h_tiles) * 128;
      const int a = i & 1;
      const uint32_t u = (uint32_t)(i >> 1);
      const int b = i % kDxTiles;
      const uint32_t ub = (uint32_t)(i / kDxTiles);
      if (!mbar_wait_warp(smem_u32(&acc_full[a]), u & 1u, p.err, kErrWaitAccum) ||
          !mbar_wait_warp(smem_u32(&dx_full[b]), ub & 1u, p.err, kErrWaitFull))
        break;
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)a * 128u;
      const uint8_t* tile =
          smem_raw + (dxs0 + (uint32_t)b * kDxTileBytes - smem_u32(smem_raw));
      const int t = t0 + r;
      uint16_t* out = p.dx + (size_t)t * p.H + h0;
      for (int c = 0; c < 8; ++c) {
        uint32_t v[16];
        tmem_ld16(tl + (uint32_t)(c * 16), v);
        tmem_ld_wait();
        const uint8_t* row = tile + (c >> 2) * kDxOpBytes + r * 128;
        const int j0 = (c & 3) * 2;
        const uint4 o0 = *reinterpret_cast<const uint4*>(row + ((j0 ^ (r & 7)) << 4));
        const uint4 o1 = *reinterpret_cast<const uint4*>(row + (((j0 + 1) ^ (r & 7)) << 4));
        const uint32_t wv[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
        uint32_t res[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const float lo = __fadd_rn(__uint_as_float(wv[m] << 16), __uint_as_float(v[2 * m]));
          const float hi =
              __fadd_rn(__uint_as_float(wv[m] & 0xFFFF0000u), __uint_as_float(v[2 * m + 1]));
          res[m] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
        }
        if (t < p.N) {
          *reinterpret_cast<uint4*>(out + c * 16) = make_uint4(res[0], res[1], res[2], res[3]);
          *reinterpret_cast<uint4*>(out + c * 16 + 8) = make_uint4(res[4], res[5], res[6], res[7]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&acc_empty[a]));
        mbar_arrive(smem_u32(&dx_empty[b]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256u);
  }
}

// ---------------------------------------------------------------- W_r split
// wrs[h, e] = hi(W_r[h,e]), wrs[h, Ep + e] = lo(W_r[h,e]); zero for e >= E.
__global__ void router_split_w_kernel(const float* __restrict__ wr, int H, int E, int Ep,
                                      uint16_t* __restrict__ wrs) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)H * Ep) return;
  const int h = (int)(i / Ep), e = (int)(i % Ep);
  uint16_t hi = 0, lo = 0;
  if (e < E) {
    const float v = wr[(size_t)h * E + e];
    const __nv_bfloat16 bh = __float2bfloat16_rn(v);
    hi = __bfloat16_as_ushort(bh);
    lo = __bfloat16_as_ushort(__float2bfloat16_rn(__fsub_rn(v, __bfloat162float(bh))));
  }
  wrs[(size_t)h * 2 * Ep + e] = hi;
  wrs[(size_t)h * 2 * Ep + Ep + e] = lo;
}

bool set_smem_limits(cudaError_t* err) {
  static DeviceOnce done;
  *err = once_per_device(done, nullptr, [](int, int*) {
    // dW_r asks for at most 2 stages of 80 KiB + 1 KiB (Ep = 256), dx for its
    // fixed layout; static shared memory comes on top of either
    cudaError_t e = cudaFuncSetAttribute(router_dwr_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(router_dx_mma_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDxSmemBytes);
  });
  return *err == cudaSuccess;
}

}  // namespace

int router_split_cols(int E) { return 2 * round64(E); }

int router_bwd_splits(int N, int H, int E) {
  if (N <= 0) return 0;
  const int Ep = round64(E);
  const int per_sm = dwr_stages(Ep) * dwr_stage_bytes(Ep) + 2048u <= 113u * 1024u ? 2 : 1;
  const int h_tiles = H / 128;
  int splits = per_sm * kRbAssumedSms / h_tiles;  // one wave of CTAs
  if (splits < 1) splits = 1;
  const int tps = round64((N + splits - 1) / splits);
  return (N + tps - 1) / tps;
}

int router_bwd_tokens_per_split(int N, int H, int E) {
  const int splits = router_bwd_splits(N, H, E);
  return splits > 0 ? round64((N + splits - 1) / splits) : 0;
}

int launch_router_split_w(const float* wr, int H, int E, uint16_t* wrs, cudaStream_t s) {
  const int Ep = round64(E);
  const int64_t n = (int64_t)H * Ep;
  router_split_w_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(wr, H, E, Ep, wrs);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? 1 : -(int)err;
}

int launch_router_dwr_mma(const uint16_t* x, const uint16_t* dls, int N, int H, int E,
                          float* part, uint32_t* errw, cudaStream_t s) {
  if (N <= 0) return 0;
  cudaError_t err = cudaSuccess;
  if (!set_smem_limits(&err)) return -(int)err;
  DwrMmaParams p{};
  p.N = N;
  p.H = H;
  p.E = E;
  p.Ep = round64(E);
  p.tps = router_bwd_tokens_per_split(N, H, E);
  p.stages = dwr_stages(p.Ep);
  p.stage_bytes = dwr_stage_bytes(p.Ep);
  p.part = part;
  p.err = errw;
  CUtensorMap tmX, tmL;
  if (!make_map_mn3d(&tmX, x, (uint64_t)H, (uint64_t)N, kRbK, 2) ||
      !make_map_mn3d(&tmL, dls, (uint64_t)(2 * p.Ep), (uint64_t)N, kRbK, (uint32_t)(p.Ep / 64)))
    return -1;
  const int splits = router_bwd_splits(N, H, E);
  const size_t dyn = (size_t)p.stages * p.stage_bytes + 1024;
  router_dwr_mma_kernel<<<dim3(H / 128, splits), kRbThreads, dyn, s>>>(tmX, tmL, p);
  err = cudaGetLastError();
  return err == cudaSuccess ? 1 : -(int)err;
}

int launch_router_dx_mma(const uint16_t* dls, const uint16_t* wrs, int N, int H, int E,
                         uint16_t* dx, uint32_t* errw, cudaStream_t s) {
  if (N <= 0) return 0;
  cudaError_t err = cudaSuccess;
  if (!set_smem_limits(&err)) return -(int)err;
  int sms = 0, dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess ||
      (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return -(int)err;
  DxMmaParams p{};
  p.N = N;
  p.H = H;
  p.Ep = round64(E);
  p.h_tiles = H / 128;
  p.items = p.h_tiles * ((N + 127) / 128);
  p.dx = dx;
  p.err = errw;
  CUtensorMap tmA, tmB, tmD;
  if (!make_map(&tmA, dls, (uint64_t)(2 * p.Ep), (uint64_t)N, 64, 128) ||
      !make_map(&tmB, wrs, (uint64_t)(2 * p.Ep), (uint64_t)H, 64, 128) ||
      !make_map(&tmD, dx, (uint64_t)H, (uint64_t)N, 64, 128))
    return -1;
  const int grid = p.items < sms ? p.items : sms;
  router_dx_mma_kernel<<<grid, kRbThreads, kDxSmemBytes, s>>>(tmA, tmB, tmD, p);
  err = cudaGetLastError();
  return err == cudaSuccess ? 1 : -(int)err;
}

}  // namespace moe
