// Expert weight gradients on the 5th-generation tensor cores.
//
// For each expert e, over its kept slots s (token t_s = sorted_slot_ids[s]):
//   dW2[e][h][i]  = sum_s dY[t_s, h] * aw[s, i]        aw = p' * silu(g) * u
//   dW13[e][k][h] = sum_s dPre[s, k] * x[t_s, h]        dPre = [dg | du]
// ("Permute-Free Grouped GEMM for MoE (bf16, gfx950)", section 5, the
// weight-gradient kernel: the contraction runs over the token slots, one owner
// per output tile, fp32 output). dW2 and dW13 have the packed layouts of w2
// [E,H,I] and w13 [E,2I,H], so they update the packed weights directly.
//
// Both operands have the slot as their contraction index and their feature
// dimension contiguous in memory, so both are read MN-major: stage tiles are
// 64 slots (K) x 64-feature chunks, 128 bytes per row with the 128-byte
// swizzle. One operand is slot-indexed (aw or dPre rows: TMA boxes), the other
// is token-indexed (rows of dY or x picked through sorted_slot_ids: 16-byte
// cp.async by four gather warps, padding rows zero-filled), as in the forward's
// gather-in-GEMM.
//
// The UMMA M dimension is always the output's contiguous dimension (i for dW2,
// h for dW13), so TMEM lane = output column and every epilogue store of one
// accumulator column is 32 consecutive floats. A tile is two 128-row
// accumulators x tile_n columns sharing each B stage; with tile_n = 256 they
// fill the 512 TMEM columns, so a tile's MMAs wait for the previous tile's
// epilogue (two buffers, and so overlap, only with tile_n = 128, which moves
// more operand bytes per flop and measured slower). An expert's last k-chunk
// issues only the 16-slot k-steps
// that hold kept slots (rows up to roundup(kept,16) are written by the FC2
// dgrad, zeros for padding); an expert with no kept slot gets zero tiles
// written without any MMA.
//
// Persistent CTAs with a dynamic tile scheduler (global counter, shared-memory
// tile queue, last CTA resets the counter), as in the forward GEMMs.
#include <cudaTypedefs.h>

#include "moe_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

constexpr int kWM = 128;              // UMMA M: output-contiguous features per accumulator
constexpr int kWN = 256;              // UMMA N
// slots per stage: 3 stages of 64 KB (48 slots in 4 stages, 32 in 6 measured
// slower: dropless ffn_backward 5.62 ms, against 5.85 and 6.33)
constexpr int kWK = 64;
constexpr int kWThreads = 448;
constexpr int kWEpiWarps = 8;         // warps 2-9
constexpr int kWGatherWarp0 = 10;     // warps 10-13
constexpr int kWGatherThreads = 128;
constexpr int kWMaxStages = 8;
constexpr uint32_t kWChunk = kWK * 128u;          // one 64-feature chunk of a stage
constexpr uint32_t kWABytes = 2 * kWM * kWK * 2;  // two accumulators' A, 4 chunks
constexpr uint32_t kWBBytes = kWN * kWK * 2;      // 4 chunks
constexpr uint32_t kWStageBytes = kWABytes + kWBBytes;
constexpr uint32_t kWSmemBudget = 223 * 1024;
// the epilogue's output staging: per warp one 16-column x 32-row fp32 block
constexpr uint32_t kWOutStgBytes = kWEpiWarps * 16 * 32 * 4;
constexpr uint32_t kWTmemCols = 512;
constexpr int kWTileQ = 4;

struct WgradParams {
  int E, m_total, n_total, m_tiles, n_tiles, bm, stages;
  int tile_n;            // UMMA N: 256, or 128 when n_total is not a multiple of 256
  int d_full;            // 64-column chunks of the slot-indexed operand in a full tile
  uint32_t buf_stride;   // TMEM columns of one accumulator buffer (2 x tile_n)
  int n_buf;             // accumulator buffers in flight (2 when 2 x buf_stride fits)
  int a_gather;          // 1: A from gathered token rows (dW13: x), B slot rows (dPre)
                         // 0: A slot rows (aw), B from gathered token rows (dW2: dY)
  const uint16_t* act;   // token-indexed operand [act_rows, act_ld]
  int act_ld, act_rows;
  const int32_t* sorted_slot_ids;
  const int32_t* kept_counts;
  const int32_t* block_start;
  int32_t* sched;        // [2]
  float* out;            // [E, n_total, m_total]
  uint32_t* err;
};

struct WTile {
  int e, m0, n0, kept, slot0, nacc;  // nacc: 128-row accumulators (the last M tile may hold one)
};

__device__ __forceinline__ void wtile_at(const WgradParams& p, int t, WTile& T) {
  const int per = p.m_tiles * p.n_tiles;
  T.e = t / per;
  const int r = t - T.e * per;
  T.m0 = (r % p.m_tiles) * 2 * kWM;
  T.nacc = T.m0 + kWM < p.m_total ? 2 : 1;
  T.n0 = (r / p.m_tiles) * p.tile_n;
  T.kept = max(p.kept_counts[T.e], 0);
  T.slot0 = p.block_start[T.e] * p.bm;
}

__global__ void __launch_bounds__(kWThreads, 1)
    moe_wgrad_kernel(const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
                     const __grid_constant__ CUtensorMap tmO, const WgradParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kWMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kWMaxStages];
  __shared__ __align__(8) uint64_t tmem_full_bar[2];
  __shared__ __align__(8) uint64_t tmem_empty_bar[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int32_t tile_q[kWTileQ];
  __shared__ __align__(8) uint64_t tq_full[kWTileQ];
  __shared__ __align__(8) uint64_t tq_empty[kWTileQ];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int n_tiles = p.E * p.m_tiles * p.n_tiles;
  // the slot-indexed operand: A (aw) when B is gathered, else B (dPre); an
  // A side holds 2 chunks of 64 features per accumulator
  const uint32_t d_off = p.a_gather ? kWABytes : 0u;
  const uint32_t g_off = p.a_gather ? 0u : kWABytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1 + kWGatherThreads);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tmem_full_bar[b]), 1);
      mbar_init(smem_u32(&tmem_empty_bar[b]), kWEpiWarps);
    }
    for (int i = 0; i < kWTileQ; ++i) {
      mbar_init(smem_u32(&tq_full[i]), 1);
      mbar_init(smem_u32(&tq_empty[i]), 1 + kWEpiWarps + 4);
    }
    mbar_fence_init();
    tma_prefetch_desc(&tmD);
    tma_prefetch_desc(&tmD2);
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_base_s), kWTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  auto pop_tile = [&](uint32_t& qi, uint32_t code) -> int {
    const int slot = (int)(qi % kWTileQ);
    const bool ok = mbar_wait_warp(smem_u32(&tq_full[slot]), (qi / kWTileQ) & 1u, p.err, code);
    const int t = ok ? tile_q[slot] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&tq_empty[slot]));
    ++qi;
    return t;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler + TMA producer
    const uint64_t pol = policy_evict_last();
    uint32_t gk = 0;
    for (uint32_t qi = 0;; ++qi) {
      const int slot = (int)(qi % kWTileQ);
      const bool free_ok =
          qi < (uint32_t)kWTileQ ||
          mbar_wait_warp(smem_u32(&tq_empty[slot]), ((qi / kWTileQ) - 1u) & 1u, p.err, kErrWaitEmpty);
      int t = -1;
      if (lane == 0) {
        if (free_ok) t = atomicAdd(&p.sched[0], 1);
        if (t >= n_tiles) t = -1;
        tile_q[slot] = t;
        mbar_arrive(smem_u32(&tq_full[slot]));
      }
      t = __shfl_sync(0xFFFFFFFFu, t, 0);
      if (t < 0) break;
      WTile T;
      wtile_at(p, t, T);
      const int chunks = (T.kept + kWK - 1) / kWK;
      const int dcol0 = p.a_gather ? T.n0 : T.m0;
      const int d_chunks = p.a_gather ? p.tile_n / 64 : 2 * T.nacc;
      bool ok = true;
      for (int kt = 0; kt < chunks; ++kt, ++gk) {
        const int s = (int)(gk % (uint32_t)p.stages);
        const uint32_t u = gk / (uint32_t)p.stages;
        if (gk >= (uint32_t)p.stages &&
            !mbar_wait_warp(smem_u32(&empty_bar[s]), (u & 1u) ^ 1u, p.err, kErrWaitEmpty)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&full_bar[s]);
          const uint32_t st = sbase + (uint32_t)s * kWStageBytes + d_off;
          mbar_arrive_expect_tx(fb, (uint32_t)d_chunks * kWChunk);
          // all 64-column chunks in one 3-D copy ([chunk][slot][64]); tmD2
          // holds 2 chunks, for the ragged last tile of the A side
          tma_load_3d(st, d_chunks == p.d_full ? &tmD : &tmD2, 0, T.slot0 + kt * kWK, dcol0 / 64,
                      fb, pol);
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    if (lane == 0) {
      __threadfence();
      if (atomicAdd(&p.sched[1], 1) == (int)gridDim.x - 1) {
        atomicExch(&p.sched[0], 0);
        atomicExch(&p.sched[1], 0);
        __threadfence();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    // The whole warp walks the tiles and takes the waits; lane 0 issues.
    const uint32_t idesc = idesc_bf16_f32(kWM, p.tile_n) | kIdescAMnMajor | kIdescBMnMajor;
    uint32_t gk = 0, tc = 0, qi = 0;
    for (;;) {
      const int t = pop_tile(qi, kErrWaitFull);
      if (t < 0) break;
      WTile T;
      wtile_at(p, t, T);
      if (T.kept == 0) continue;  // zero tile: the epilogue writes it without TMEM
      const uint32_t b = tc % (uint32_t)p.n_buf, bu = tc / (uint32_t)p.n_buf;
      if (bu > 0 && !mbar_wait_warp(smem_u32(&tmem_empty_bar[b]), (bu - 1u) & 1u, p.err,
                                    kErrWaitAccum))
        break;
      tc_fence_after();
      const uint32_t d = tmem + b * p.buf_stride;
      const int chunks = (T.kept + kWK - 1) / kWK;
      bool ok = true;
      for (int kt = 0; kt < chunks; ++kt, ++gk) {
        const int s = (int)(gk % (uint32_t)p.stages);
        const uint32_t u = gk / (uint32_t)p.stages;
        if (!mbar_wait_warp(smem_u32(&full_bar[s]), u & 1u, p.err, kErrWaitFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          fence_proxy_async_smem();  // gathered rows: cp.async (generic proxy) writes
          const uint32_t st = sbase + (uint32_t)s * kWStageBytes;
          const int rem = T.kept - kt * kWK;
          const int ksub = rem >= kWK ? kWK / 16 : (rem + 15) / 16;
          for (int kk = 0; kk < ksub; ++kk) {
            const uint64_t bdesc = sdesc_sw128_mn(st + kWABytes + (uint32_t)kk * 2048u, kWChunk);
            for (int a = 0; a < T.nacc; ++a)
              umma_bf16(d + (uint32_t)(a * p.tile_n),
                        sdesc_sw128_mn(st + (uint32_t)a * 2u * kWChunk + (uint32_t)kk * 2048u, kWChunk), bdesc,
                        idesc, (kt | kk) != 0);
          }
          umma_commit(smem_u32(&empty_bar[s]));
        }
        __syncwarp();
      }
      if (lane == 0) umma_commit(smem_u32(&tmem_full_bar[b]));  // also after an abort
      __syncwarp();
      ++tc;
      if (!ok) break;
    }
  } else if (warp < 2 + kWEpiWarps) {
    // ------------------------------------------------------------ epilogue
    // warp w reads TMEM lanes 32*(w%4)..+31 (output rows m0+32q..+31) and the
    // 16-column chunks c0 = 16*half, +32, ...
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    // this warp's output staging block [16 columns][32 rows] fp32; each
    // 16-column chunk goes out as one TMA store of a 32 x 16 box (dW rows
    // e*n_total + n, m contiguous), so the epilogue's writes leave through the
    // TMA engine rather than the load/store pipe the row gather uses
    const uint32_t ostg = sbase + (uint32_t)p.stages * kWStageBytes + (uint32_t)(warp - 2) * 2048u;
    uint32_t tc = 0, qi = 0;
    for (;;) {
      const int t = pop_tile(qi, kErrWaitAccum);
      if (t < 0) break;
      WTile T;
      wtile_at(p, t, T);
      float* dst = p.out + ((size_t)T.e * p.n_total + T.n0) * p.m_total + T.m0 + q * 32 + lane;
      if (T.kept == 0) {
        for (int a = 0; a < T.nacc; ++a)
          for (int c = half * 16; c < p.tile_n; c += 32)
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[(size_t)(c + j) * p.m_total + a * kWM] = 0.0f;
        continue;
      }
      const uint32_t b = tc % (uint32_t)p.n_buf, bu = tc / (uint32_t)p.n_buf;
      const bool w =
          mbar_wait_warp(smem_u32(&tmem_full_bar[b]), bu & 1u, p.err, kErrWaitAccum);
      ++tc;
      if (!w) break;
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + b * p.buf_stride;
      for (int a = 0; a < T.nacc; ++a) {
        for (int c = half * 16; c < p.tile_n; c += 32) {
          uint32_t v[16];
          tmem_ld16(tl + (uint32_t)(a * p.tile_n + c), v);
          tmem_ld_wait();
          // the warp's previous block has left the staging buffer
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(ostg + (uint32_t)(j * 128 + lane * 4)),
                         "f"(__uint_as_float(v[j]))
                         : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmO, ostg, T.m0 + a * kWM + q * 32, T.e * p.n_total + T.n0 + c);
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive(smem_u32(&tmem_empty_bar[b]));
    }
    if (lane == 0) bulk_wait_all();  // the last stores have read their staging and landed
  } else {
    // ------------------------------------------------------------ token-row gather
    // Stage row r (slot slot0 + 64kt + r) of 64-feature chunk c holds
    // act[t, col0 + 64c .. +63] for t = sorted_slot_ids[slot]: 16-byte unit j
    // at c*8192 + r*128 + ((j ^ (r%8)) * 16). Slots past the kept count and
    // sentinel tokens are zero-filled. One warp instruction copies one chunk
    // (128 bytes) of four consecutive rows, 512 contiguous bytes of shared
    // memory (lane l: row 4i + l/8, unit l%8); with four chunks warp g takes
    // chunk g of all 64 rows (16 instructions a stage), with two chunk g%2 of
    // rows 32*(g/2) .. +31 (8). (Copying a whole 512-byte token row per
    // instruction into four chunks 8 KB apart issued 1.5x slower.) Lane l
    // holds the tokens of stage rows l and l + 32, loaded one stage ahead and
    // broadcast with a shuffle. The full barrier receives each thread's
    // arrival when its copies complete (cp.async.mbarrier.arrive.noinc); the
    // UMMA thread fences them against its async-proxy reads. Waits end in a
    // warp vote, so a warp leaves together when one runs out.
    const int gw = warp - kWGatherWarp0;
    const int jj = lane & 7, rsub = lane >> 3;
    uint32_t gk = 0, qi = 0;
    bool ok = true;
    while (ok) {
      const int t = pop_tile(qi, kErrWaitFull);
      if (t < 0) break;
      WTile T;
      wtile_at(p, t, T);
      const int g_chunks = p.a_gather ? 2 * T.nacc : p.tile_n / 64;  // 4 or 2
      const int cw = g_chunks == 4 ? gw : (gw & 1);
      const int row_lo = g_chunks == 4 ? 0 : (kWK / 2) * (gw >> 1);
      const int n_ins = (g_chunks == 4 ? kWK : kWK / 2) / 4;
      const int gcol0 = (p.a_gather ? T.m0 : T.n0) + cw * 64 + jj * 8;
      const int chunks = (T.kept + kWK - 1) / kWK;
      auto token_of = [&](int kt, int r) -> int {
        const int ks = kt * kWK + r;
        return (r < kWK && kt < chunks && ks < T.kept) ? p.sorted_slot_ids[T.slot0 + ks] : -1;
      };
      int nxt0 = token_of(0, lane), nxt1 = token_of(0, lane + 32);
      for (int kt = 0; kt < chunks; ++kt, ++gk) {
        const int cur0 = nxt0, cur1 = nxt1;
        nxt0 = token_of(kt + 1, lane);
        nxt1 = token_of(kt + 1, lane + 32);
        const int s = (int)(gk % (uint32_t)p.stages);
        const uint32_t u = gk / (uint32_t)p.stages;
        if (gk >= (uint32_t)p.stages &&
            !mbar_wait_warp(smem_u32(&empty_bar[s]), (u & 1u) ^ 1u, p.err, kErrWaitEmpty)) {
          ok = false;
          break;
        }
        const uint32_t g = sbase + (uint32_t)s * kWStageBytes + g_off + (uint32_t)cw * kWChunk;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i < n_ins) {
            const int r0 = row_lo + 4 * i;  // the instruction's first row (warp-uniform)
            const int r = r0 + rsub;
            const int tok = __shfl_sync(0xFFFFFFFFu, r0 < 32 ? cur0 : cur1, r & 31);
            const bool valid = (unsigned)tok < (unsigned)p.act_rows;
            const uint16_t* src = p.act + (size_t)(valid ? tok : 0) * p.act_ld + gcol0;
            cp_async_16(g + (uint32_t)r * 128u + ((uint32_t)(jj ^ (r & 7)) << 4), src,
                        valid ? 16u : 0u);
          }
        }
        cp_async_mbar_arrive_noinc(smem_u32(&full_bar[s]));
      }
    }
    cp_async_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kWTmemCols);
  }
}

int wgrad_sms(cudaError_t* err) {
  static DeviceOnce sms;
  int n = 0;
  *err = once_per_device(sms, &n, [](int dev, int* v) {
    cudaError_t e = cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(moe_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kWSmemBudget);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
  });
  return *err == cudaSuccess ? n : 0;
}

}  // namespace

int launch_wgrad(const WgradArgs& a, cudaStream_t s) {
  if (a.E <= 0) return 0;
  WgradParams p{};
  p.E = a.E;
  p.bm = a.bm;
  p.sorted_slot_ids = a.sorted_slot_ids;
  p.kept_counts = a.kept_counts;
  p.block_start = a.block_start;
  p.sched = a.sched;
  p.out = a.out;
  p.err = a.err;
  CUtensorMap tmD, tmD2, tmO;
  const int tile_n = ((a.dw13 ? 2 * a.I : a.H) % kWN == 0) ? kWN : 128;
  if (a.dw13) {
    // M = h (x gathered), N = k over 2I (dPre rows)
    p.a_gather = 1;
    p.m_total = a.H;
    p.n_total = 2 * a.I;
    p.act = static_cast<const uint16_t*>(a.x);
    p.act_ld = a.H;
    p.d_full = tile_n / 64;
    if (!make_map_mn3d(&tmD, a.slot_mat, (uint64_t)(2 * a.I), (uint64_t)a.s_max, kWK, p.d_full) ||
        !make_map_mn3d(&tmD2, a.slot_mat, (uint64_t)(2 * a.I), (uint64_t)a.s_max, kWK, 2))
      return -1;
  } else {
    // M = i (aw rows), N = h (dY gathered)
    p.a_gather = 0;
    p.m_total = a.I;
    p.n_total = a.H;
    p.act = static_cast<const uint16_t*>(a.dy);
    p.act_ld = a.H;
    p.d_full = 4;  // two accumulators of 128 rows
    if (!make_map_mn3d(&tmD, a.slot_mat, (uint64_t)a.I, (uint64_t)a.s_max, kWK, 4) ||
        !make_map_mn3d(&tmD2, a.slot_mat, (uint64_t)a.I, (uint64_t)a.s_max, kWK, 2))
      return -1;
  }
  p.act_rows = a.N;
  p.tile_n = tile_n;
  if (p.m_total % kWM != 0 || p.n_total % p.tile_n != 0) return -1;
  p.m_tiles = (p.m_total + 2 * kWM - 1) / (2 * kWM);
  p.n_tiles = p.n_total / p.tile_n;
  p.buf_stride = (uint32_t)(2 * p.tile_n);
  p.n_buf = 2 * p.buf_stride <= kWTmemCols ? 2 : 1;
  // dW as a 2-D fp32 matrix [E * n_total rows, m_total], stored in 32 x 16 boxes
  if (!make_map_plain(&tmO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.out, (uint64_t)p.m_total,
                      (uint64_t)p.E * p.n_total, 32, 16))
    return -1;
  p.stages = (int)((kWSmemBudget - 1024u - kWOutStgBytes) / kWStageBytes);
  if (p.stages > kWMaxStages) p.stages = kWMaxStages;
  const size_t dyn = (size_t)p.stages * kWStageBytes + kWOutStgBytes + 1024;
  cudaError_t err = cudaSuccess;
  const int sms = wgrad_sms(&err);
  if (sms <= 0) return -(int)(err != cudaSuccess ? err : cudaErrorUnknown);
  const int64_t tiles = (int64_t)p.E * p.m_tiles * p.n_tiles;
  const int grid = (int)(tiles < sms ? tiles : sms);
  moe_wgrad_kernel<<<grid, kWThreads, dyn, s>>>(tmD, tmD2, tmO, p);
  err = cudaGetLastError();
  return err == cudaSuccess ? 1 : -(int)err;
}

}  // namespace moe
