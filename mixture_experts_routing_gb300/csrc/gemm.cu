// Expert grouped GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Both GEMMs are computed "weights as M": D[f, s] = W[e][f, :] . A[s, :] for the
// weight rows f of one 128-row tile and the token slots s of one tile (UMMA
// M = 128, N = slots rounded up to 16, K = 16 per instruction). A slot tile
// never holds more than 256 slots, so a tile of an expert with few kept routes
// costs one MMA per k-step, with N as small as 16.
//
//  FC1 (gather-in-GEMM, "Permute-Free Grouped GEMM for MoE (bf16, gfx950)",
//  section 2 Core idea and section 3 End-to-end flow): the B operand rows are
//  x[sorted_slot_ids[s], :], copied row by row (16-byte cp.async, 128 threads)
//  straight into the 128-byte-swizzled operand buffer; no permuted copy of x is
//  written. (A TMA tile::gather4 of the same rows measured 2x slower overall:
//  one 512-byte gather per ~80 cycles per SM.) Two
//  accumulators per CTA, gate rows and up rows of the same 128 features; the
//  epilogue reads both from TMEM and writes h = silu(gate) * up (SwiGLU as the
//  FC1 epilogue rather than a separate pass).
//  FC2 (route space, same section 3): B rows are h[s, :] for a contiguous slot
//  range, fetched by tiled TMA loads; up to two 128-row output tiles per CTA
//  share one B stage.
//
// The grouping comes from device-side vectors only (kept_counts, block_start:
// "[4/5] feat: capture the FFN experts at bucketed padded shapes", What this
// adds): the grid is the static bound E x feature tiles x slot tiles and a CTA
// whose slot tile lies past its expert's kept count exits at once, so nothing
// is read back to the host and the launch is graph-capturable.
//
// Warp roles (192 threads): warp 0 = TMA producer (weight tiles; FC2's B
// tiles), warp 1 = TMEM allocator and single-thread UMMA issuer, warps 2-5 =
// FC1's B-row gatherers during the main loop, then the epilogue (warp w reads
// TMEM lanes 32*(w%4) .. 32*(w%4)+31). Operand stages form a ring guarded by
// full/empty mbarriers; UMMA completion is signalled with tcgen05.commit.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;           // contraction elements per stage (128 B of bf16)
constexpr int kTileM = 128;       // weight rows per accumulator (UMMA M)
constexpr int kMaxTileN = 256;    // slots per tile (UMMA N)
constexpr int kMaxStages = 8;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kATileBytes = kTileM * kBK * 2;  // 16 KiB
constexpr uint32_t kSmemBudget = 225 * 1024;
constexpr int kGatherThreads = 128;  // warps 2-5
constexpr int kGatherDepth = 2;      // cp.async groups in flight per gather thread

struct GemmParams {
  int fc1;
  int n_acc;
  int k_tiles;
  int a_rows_per_expert;
  int a_second_off;
  int f_rows;
  int f_tiles;
  int n_tok_tiles;
  int tile_n;
  int bm;
  int out_ld;
  int stages;
  uint32_t stage_bytes;
  uint32_t b_off;
  const uint16_t* act;   // FC1: x [act_rows, act_ld] for the row gather
  int act_ld;
  int act_rows;
  const int32_t* sorted_slot_ids;
  const int32_t* kept_counts;
  const int32_t* block_start;
  uint16_t* out;
  uint32_t* err;
};

__device__ __forceinline__ uint16_t f32_to_bf16(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t accum_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int32_t rows_s[kMaxTileN];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int idx = blockIdx.x;
  const int jt = idx % p.n_tok_tiles;
  idx /= p.n_tok_tiles;
  const int f = idx % p.f_tiles;
  const int e = idx / p.f_tiles;
  const int rows = min(p.tile_n, p.kept_counts[e] - jt * p.tile_n);
  if (rows <= 0) return;  // uniform over the CTA: nothing allocated or armed yet
  const int n_eff = (rows + 15) & ~15;
  const int slot0 = p.block_start[e] * p.bm + jt * p.tile_n;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), p.fc1 ? 1 + kGatherThreads : 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&accum_bar), 1);
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    if (!p.fc1) tma_prefetch_desc(&tmB);
  }
  if (warp >= 2 && p.fc1)
    for (int i = threadIdx.x - 64; i < n_eff; i += kGatherThreads)
      rows_s[i] = p.sorted_slot_ids[slot0 + i];
  if (warp == 1) tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    // Lane 0 arms the stage barrier and loads the weight tiles; for FC2 every
    // lane then issues its share of the B-operand tile loads.
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    const int a_row0 = e * p.a_rows_per_expert + f * p.f_rows;
    const uint32_t tx = (uint32_t)p.n_acc * kATileBytes + (p.fc1 ? 0u : (uint32_t)n_eff * 128u);
    for (int kt = 0; kt < p.k_tiles; ++kt) {
      const int s = kt % p.stages;
      const uint32_t u = (uint32_t)(kt / p.stages);
      int ok = 1;
      if (lane == 0 && kt >= p.stages)
        ok = mbar_wait(smem_u32(&empty_bar[s]), (u & 1u) ^ 1u, p.err, kErrWaitEmpty);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      const uint32_t fb = smem_u32(&full_bar[s]);
      const uint32_t st = sbase + (uint32_t)s * p.stage_bytes;
      const int kx = kt * kBK;
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, tx);
        tma_load_2d(st, &tmA, kx, a_row0, fb, pol_w);
        if (p.n_acc == 2) tma_load_2d(st + kATileBytes, &tmA, kx, a_row0 + p.a_second_off, fb, pol_w);
      }
      __syncwarp();
      if (!p.fc1) {
        const uint32_t b = st + p.b_off;
        for (int q = lane * 16; q < n_eff; q += 512)
          tma_load_2d(b + (uint32_t)q * 128u, &tmB, kx, slot0 + q, fb, pol_x);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, n_eff);
      for (int kt = 0; kt < p.k_tiles; ++kt) {
        const int s = kt % p.stages;
        const uint32_t u = (uint32_t)(kt / p.stages);
        if (!mbar_wait(smem_u32(&full_bar[s]), u & 1u, p.err, kErrWaitFull)) break;
        tc_fence_after();
        const uint32_t st = sbase + (uint32_t)s * p.stage_bytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint32_t acc = (kt | kk) != 0;
          const uint64_t bdesc = sdesc_sw128(st + p.b_off + (uint32_t)kk * 32u);
          umma_bf16(tmem, sdesc_sw128(st + (uint32_t)kk * 32u), bdesc, idesc, acc);
          if (p.n_acc == 2)
            umma_bf16(tmem + 256u, sdesc_sw128(st + kATileBytes + (uint32_t)kk * 32u), bdesc, idesc,
                      acc);
        }
        umma_commit(smem_u32(&empty_bar[s]));
      }
      umma_commit(smem_u32(&accum_bar));
    }
  } else {
    if (p.fc1) {
      // FC1 B operand: row r of the stage holds x[rows_s[r], kx .. kx+63],
      // 16-byte chunk c at r*128 + ((c ^ (r%8)) * 16) (the 128-byte swizzle
      // the UMMA descriptor expects); sentinel rows are zero-filled. Each
      // thread keeps kGatherDepth copy groups in flight, then makes a stage's
      // writes visible to the tensor core's async proxy and arrives.
      const int gt = threadIdx.x - 64;
      const int nchunks = n_eff * 8;
      int kt = 0;
      for (; kt < p.k_tiles; ++kt) {
        const int s = kt % p.stages;
        const uint32_t u = (uint32_t)(kt / p.stages);
        if (kt >= p.stages &&
            !mbar_wait(smem_u32(&empty_bar[s]), (u & 1u) ^ 1u, p.err, kErrWaitEmpty))
          break;
        const uint32_t b = sbase + (uint32_t)s * p.stage_bytes + p.b_off;
        const int kx = kt * kBK;
        for (int j = gt; j < nchunks; j += kGatherThreads) {
          const int r = j >> 3, c = j & 7;
          const int tok = rows_s[r];
          const bool valid = (unsigned)tok < (unsigned)p.act_rows;
          const uint16_t* src = p.act + (size_t)(valid ? tok : 0) * p.act_ld + kx + c * 8;
          cp_async_16(b + (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4), src,
                      valid ? 16u : 0u);
        }
        cp_async_commit();
        if (kt >= kGatherDepth) {
          cp_async_wait<kGatherDepth>();
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&full_bar[(kt - kGatherDepth) % p.stages]));
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      for (int j = kt > kGatherDepth ? kt - kGatherDepth : 0; j < kt; ++j)
        mbar_arrive(smem_u32(&full_bar[j % p.stages]));
    }
    const int q = warp & 3;
    if (mbar_wait(smem_u32(&accum_bar), 0u, p.err, kErrWaitAccum)) {
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
      if (p.fc1) {
        const int feat = f * kTileM + q * 32 + lane;
        for (int c0 = 0; c0 < n_eff; c0 += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(tl + (uint32_t)c0, g);
          tmem_ld16(tl + 256u + (uint32_t)c0, u);
          tmem_ld_wait();
          uint16_t* o = p.out + (size_t)(slot0 + c0) * p.out_ld + feat;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gv = __uint_as_float(g[i]);
            const float uv = __uint_as_float(u[i]);
            const float a = gv / (1.0f + __expf(-gv)) * uv;
            o[(size_t)i * p.out_ld] = f32_to_bf16(a);
          }
        }
      } else {
        const int feat = f * p.f_rows + q * 32 + lane;
        for (int c0 = 0; c0 < n_eff; c0 += 16) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tl + (uint32_t)c0, v0);
          if (p.n_acc == 2) tmem_ld16(tl + 256u + (uint32_t)c0, v1);
          tmem_ld_wait();
          uint16_t* o = p.out + (size_t)(slot0 + c0) * p.out_ld + feat;
#pragma unroll
          for (int i = 0; i < 16; ++i) o[(size_t)i * p.out_ld] = f32_to_bf16(__uint_as_float(v0[i]));
          if (p.n_acc == 2) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              o[(size_t)i * p.out_ld + kTileM] = f32_to_bf16(__uint_as_float(v1[i]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// 2-D bf16 tensor [rows, cols] row-major, 128-byte swizzled boxes of
// box_cols x box_rows; out-of-bounds elements read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_gemm(const GemmArgs& a, cudaStream_t s) {
  if (a.cpad <= 0 || a.N <= 0) return 0;
  GemmParams p{};
  p.fc1 = a.fc1;
  p.bm = a.bm;
  p.sorted_slot_ids = a.sorted_slot_ids;
  p.kept_counts = a.kept_counts;
  p.block_start = a.block_start;
  p.out = static_cast<uint16_t*>(a.out);
  p.err = a.err;
  p.act = static_cast<const uint16_t*>(a.act);
  p.act_ld = a.fc1 ? a.H : a.I;
  p.act_rows = a.fc1 ? a.N : 0;
  const int64_t S = (int64_t)a.E * a.cpad;
  CUtensorMap tmA, tmB;
  if (a.fc1) {
    p.n_acc = 2;
    p.k_tiles = a.H / kBK;
    p.a_rows_per_expert = 2 * a.I;
    p.a_second_off = a.I;
    p.f_rows = kTileM;
    p.f_tiles = a.I / kTileM;
    p.out_ld = a.I;
    if (!make_map(&tmA, a.w, (uint64_t)a.H, (uint64_t)a.E * 2 * a.I, kBK, kTileM)) return -1;
    tmB = tmA;  // unused: FC1 gathers its B rows with cp.async
  } else {
    p.n_acc = (a.H % (2 * kTileM) == 0) ? 2 : 1;
    p.k_tiles = a.I / kBK;
    p.a_rows_per_expert = a.H;
    p.a_second_off = kTileM;
    p.f_rows = kTileM * p.n_acc;
    p.f_tiles = a.H / p.f_rows;
    p.out_ld = a.H;
    if (!make_map(&tmA, a.w, (uint64_t)a.I, (uint64_t)a.E * a.H, kBK, kTileM)) return -1;
    if (!make_map(&tmB, a.act, (uint64_t)a.I, (uint64_t)S, kBK, 16)) return -1;
  }
  p.n_tok_tiles = (int)((a.cpad + kMaxTileN - 1) / kMaxTileN);
  const int64_t per = (a.cpad + p.n_tok_tiles - 1) / p.n_tok_tiles;
  p.tile_n = (int)((per + 15) / 16 * 16);
  p.b_off = (uint32_t)p.n_acc * kATileBytes;
  p.stage_bytes = p.b_off + (((uint32_t)p.tile_n * 128u + 1023u) & ~1023u);
  p.stages = (int)((kSmemBudget - 1024u) / p.stage_bytes);
  if (p.stages > kMaxStages) p.stages = kMaxStages;
  if (p.stages < 2) return -1;
  const size_t dyn = (size_t)p.stages * p.stage_bytes + 1024;
  cudaError_t err = cudaSuccess;
  {
    // raise the kernel's dynamic shared-memory limit once per device
    static int set_for[64] = {};
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return -(int)err;
    if (dev < 0 || dev >= 64 || !set_for[dev]) {
      err = cudaFuncSetAttribute(moe_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBudget);
      if (err != cudaSuccess) return -(int)err;
      if (dev >= 0 && dev < 64) set_for[dev] = 1;
    }
  }
  const int64_t grid = (int64_t)a.E * p.f_tiles * p.n_tok_tiles;
  moe_gemm_kernel<<<(unsigned)grid, kThreads, dyn, s>>>(tmA, tmB, p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return -(int)err;
  return 1;
}

}  // namespace moe
