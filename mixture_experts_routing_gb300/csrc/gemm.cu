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
//  one 512-byte gather per ~80 cycles per SM.) Two accumulators per tile, gate
//  rows and up rows of the same 128 features; the epilogue reads both from TMEM
//  and writes h = silu(gate) * up (SwiGLU as the FC1 epilogue rather than a
//  separate pass).
//  FC2 (route space, same section 3): B rows are h[s, :] for a contiguous slot
//  range, fetched by tiled TMA loads; up to two 128-row output tiles share one
//  B stage.
//
// The grouping comes from device-side vectors only (kept_counts, block_start:
// "[4/5] feat: capture the FFN experts at bucketed padded shapes", What this
// adds): the tile list is the static bound E x feature tiles x slot tiles and a
// tile past its expert's kept count is skipped, so nothing is read back to the
// host and the launch is graph-capturable.
//
// Persistent: one CTA per SM takes tiles from a global counter (dynamic
// scheduling: tiles of a skewed routing differ a lot in size) and publishes
// each tile id to its other warps through a small shared-memory queue. The
// operand ring runs across tile boundaries, so the weight stream keeps going
// while the epilogue of the previous tile drains TMEM and stores. The last CTA
// to finish resets the counter, so the next launch finds it at zero.
// Warp roles (448 threads): warp 0 = TMA producer (weight tiles; FC2's B
// tiles), warp 1 = TMEM allocator and single-thread UMMA issuer, warps 2-9 =
// epilogue (warp w reads TMEM lanes 32*(w%4) .. +31; two warps per lane
// quarter take alternate 16-column chunks, halving the time TMEM stays
// occupied), warps 10-13 = FC1's B-row gatherers. Stages are guarded by
// full/empty mbarriers, the accumulator by tmem_full / tmem_empty; UMMA
// completion is signalled with tcgen05.commit.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace moe {
namespace {

constexpr int kBK = 64;           // contraction elements per stage (128 B of bf16)
constexpr int kTileM = 128;       // weight rows per accumulator (UMMA M)
constexpr int kMaxTileN = 256;    // slots per tile (UMMA N), at most
constexpr int kMxMaxTileN = 224;  // the same for the MX modes (TMEM also holds the scales)
constexpr int kMaxStages = 8;
// Rows per TMA box of a slot-indexed B operand (one CTA; one CTA of a pair):
// whole large boxes for the bulk of a tile's rows, small ones (a multiple of
// which every tile's row count is) for the rest. Fewer, larger boxes took the
// Qwen3-30B-shaped FC2 from 0.135 to 0.132 ms (pair: 0.132 -> 0.128 ms);
// large boxes alone, reading past a tile's rows, cost the DeepSeek-V3-shaped
// FC2 6 % (slot tiles of at most 160 rows).
constexpr int kBBoxRows = 64;
constexpr int kBBoxRowsPair = 32;
constexpr int kBBoxRowsSmall = 16;
constexpr int kBBoxRowsPairSmall = 8;
constexpr int kThreads = 448;
constexpr int kEpiWarps = 8;         // warps 2-9
constexpr int kGatherWarp0 = 10;     // warps 10-13
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kATileBytes = kTileM * kBK * 2;  // 16 KiB
// dynamic shared memory opt-in; with the kernel's 2.25 KB of static shared
// memory the CTA stays under the 227 KB per-block limit
constexpr uint32_t kSmemBudget = 224 * 1024;
constexpr int kGatherThreads = 128;  // warps 10-13
constexpr int kStageRowElems = 32;   // epilogue staging row: 32 features (bf16)
constexpr uint32_t kEpiStageBytes = kEpiWarps * 8u * kStageRowElems * 2u;  // per warp 8 rows
constexpr int kTileQ = 4;            // depth of the tile-id queue
constexpr uint32_t kPsBytes = kEpiWarps * 16 * 4;  // FC2 dgrad: 16 p' values per epilogue warp
constexpr uint32_t kPreBufBytes = kEpiWarps * 2048;  // FC2 dgrad: a warp's next 16 x 2 x 32
                                                      // pre-activations (bf16)
constexpr uint32_t kXsBytes = kEpiWarps * 128 * 4;  // FC1 FP8: the token scales of a warp's
                                                    // (up to 8) chunks of 16 slots

struct GemmParams {
  int n_acc;             // accumulators per tile: FC1 gate + up; otherwise two 128-feature
                         // tiles (the last feature tile may hold one: Tile::nacc)
  int pair_feats;        // the two accumulators are feature tiles (not gate/up)
  int m_total;           // features of the output (ragged last tile when pair_feats)
  int max_tn;            // slots per tile, at most (128 or 256)
  uint32_t acc_off;      // TMEM columns between a tile's two accumulators
  uint32_t buf_stride;   // TMEM columns of one accumulator buffer
  int k_tiles;
  int a_rows_per_expert;
  int a_second_off;
  int f_rows;
  int f_tiles;
  int E;
  int bm;
  int out_ld;
  int stages;
  uint32_t stage_bytes;
  uint32_t b_off;
  uint32_t epi_off;      // offset of the epilogue staging buffer from the aligned smem base
  uint32_t ps_off;       // FC2 dgrad: offset of the epilogue warps' p' slots
  int n_buf;             // accumulators in flight: 2 when a tile uses 256 TMEM columns, else 1
  const uint16_t* act;   // FC1: x [act_rows, act_ld] for the row gather
  int act_ld;
  int act_rows;
  const int32_t* sorted_slot_ids;
  const int32_t* kept_counts;
  const int32_t* block_start;
  int32_t* sched;        // [2]: next tile to hand out, CTAs finished
  uint16_t* out;
  uint16_t* out2;        // FC1: pre-activations [S,2I] or null; FC2 dgrad: p'*a [S,I]
  const uint16_t* aux;   // FC2 dgrad: pre-activations [S,2I]
  const float* slot_prob;     // p' of each slot's route, 0 for padding (FC1 with
                              // prob_in_act, FC2 dgrad)
  int activation;             // 0 SwiGLU, 1 GeGLU
  int prob_in_act;            // FC1: h = act(g) u p'
  const float* w_scale;       // FP8: scale of each A (weight) row: FC1 [E*2I], FC2 [E*H]
  const float* x_scale;       // FP8: scale of each B row: FC1 token [N], FC2 slot [S]
  uint32_t xs_off;            // FP8: offset of the epilogue warps' B-row scale slices
  float* part;                // FC2 dgrad: dprob partials [S, I/32]
  int inter;                  // I
  uint32_t* err;
  const uint8_t* sfa;         // MX: E8M0 scales of the weight rows, 512-byte atoms
  const uint8_t* sfb;         // MX: E8M0 scales of the B rows, [rows, sfb_ld]
  int sfb_ld;                 // MX: scale bytes per B row (K / 32)
  uint32_t sf_off;            // MX: offset in a stage of its scale atoms (2 of A, 2 of B)
  uint32_t sf_tmem;           // MX: first TMEM column of the scale ring (16 per stage)
  int f_cta;                  // pair mode: features of a pair tile that each CTA holds
};

struct Tile {
  int e, f, rows, n_eff, slot0, nacc;
};

// Dense tile list: expert e owns tiles [tpre[e], tpre[e+1]); each of its
// ntt = ceil(kept/256) slot tiles holds ttn[e] slots (kept split evenly,
// rounded up to 16, at most max_tn), times f_tiles feature tiles. Built once
// per CTA.
__device__ __forceinline__ void build_tile_list(const GemmParams& p, int32_t* tpre, int32_t* ttn,
                                                int lane) {
  int run = 0;
  for (int e0 = 0; e0 < p.E; e0 += 32) {
    const int e = e0 + lane;
    int tiles = 0;
    if (e < p.E) {
      const int kept = max(p.kept_counts[e], 0);
      const int ntt = (kept + p.max_tn - 1) / p.max_tn;
      ttn[e] = ntt ? ((kept + ntt - 1) / ntt + 15) & ~15 : 0;
      tiles = ntt * p.f_tiles;
    }
    int incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += u;
    }
    if (e < p.E) tpre[e] = run + incl - tiles;
    run += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  if (lane == 0) tpre[p.E] = run;
}

// Decodes tile index t (slot tile fastest, then feature tile, within expert).
__device__ __forceinline__ void tile_at(const GemmParams& p, const int32_t* tpre,
                                        const int32_t* ttn, int t, Tile& T) {
  int lo = 0, hi = p.E - 1;  // last e with tpre[e] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tpre[mid] <= t) lo = mid; else hi = mid - 1;
  }
  T.e = lo;
  const int local = t - tpre[lo];
  const int tn = ttn[lo];
  const int kept = p.kept_counts[lo];
  const int ntt = (kept + p.max_tn - 1) / p.max_tn;
  const int jt = local % ntt;
  T.f = local / ntt;
  T.rows = min(tn, kept - jt * tn);
  T.n_eff = (T.rows + 15) & ~15;
  T.slot0 = p.block_start[lo] * p.bm + jt * tn;
  T.nacc = (p.pair_feats && T.f * p.f_rows + kTileM >= p.m_total) ? 1 : p.n_acc;
}

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Writes a 16-slot x 32-feature block to a bf16 row-major matrix: lane l holds
// feature l of slot j in value_of(j) (evaluated as the block is written, so
// the 16 values need not be live together); dst points at (slot 0, feature 0),
// ld is the row stride in elements. Staged through this warp's 512-byte
// buffer, eight rows at a time, so that each row goes out as four 16-byte
// stores.
template <class F>
__device__ __forceinline__ void store_rows16_of(uint32_t stg_u, int lane, F value_of,
                                                uint16_t* dst, int ld) {
#pragma unroll
  for (int h8 = 0; h8 < 2; ++h8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t at = stg_u + (uint32_t)(i * kStageRowElems + lane) * 2u;
      asm volatile("st.shared.b16 [%0], %1;" ::"r"(at),
                   "h"((unsigned short)bf16_bits(value_of(h8 * 8 + i)))
                   : "memory");
    }
    __syncwarp();
    const int row = lane >> 2, part = lane & 3;  // 8 rows x 4 chunks of 16 bytes
    uint4 val;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                 : "r"(stg_u + (uint32_t)(row * kStageRowElems + part * 8) * 2u)
                 : "memory");
    *reinterpret_cast<uint4*>(dst + (size_t)(h8 * 8 + row) * ld + part * 8) = val;
    __syncwarp();
  }
}

// The same with the 16 values in registers: v[j] is slot j's.
__device__ __forceinline__ void store_rows16(uint32_t stg_u, int lane, const float (&v)[16],
                                             uint16_t* dst, int ld) {
  store_rows16_of(stg_u, lane, [&](int j) { return v[j]; }, dst, ld);
}

// Gated activation act(gate) of the FFN and its derivative ("Permute-Free
// Grouped GEMM for MoE (bf16, gfx950)", section 3 act(gate)*up; section 8:
// silu and gelu): 0 = silu(v) = v sigma(v); 1 = gelu(v) = v Phi(v) (the erf
// form); act_grad: sigma(v)(1 + v(1 - sigma(v))), Phi(v) + v phi(v).
template <int act>
__device__ __forceinline__ float act_fwd(float v) {
  if (act == 1) return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
  return __fdividef(v, 1.0f + __expf(-v));
}

// The factor both share: act(v) = v c(v) with c = sigma (silu) or Phi (gelu),
// and act'(v) from c: c (1 + v (1 - c)) for silu, c + v phi(v) for gelu. The
// backward evaluates c once per element and derives both from it.
template <int act>
__device__ __forceinline__ float act_core(float v) {
  if (act == 1) return 0.5f * (1.0f + erff(v * 0.70710678118654752f));
  return __fdividef(1.0f, 1.0f + __expf(-v));
}

template <int act>
__device__ __forceinline__ float act_grad_core(float v, float c) {
  if (act == 1) return c + v * (__expf(-0.5f * v * v) * 0.39894228040143268f);
  return c * (1.0f + v * (1.0f - c));
}

// p' of slot c0 + lane of the tile for lanes 0..15 (0 past the kept rows).
__device__ __forceinline__ float load_slot_prob(const GemmParams& p, const Tile& T, int c0, int lane) {
  return (lane < 16 && c0 + lane < T.rows) ? p.slot_prob[T.slot0 + c0 + lane] : 0.0f;
}

// The 32-feature partial sums of the dprob terms: dp[j] (slot j's term of
// this lane's feature) summed over the warp's 32 lanes for each of the 16
// slots, halving the values held per lane at each exchange (afterwards lanes
// 2m and 2m+1 hold slot m), written to part[slot, feat0/32].
__device__ __forceinline__ void dprob_part16(const GemmParams& p, const Tile& T, int c0, int feat0,
                                             int lane, float (&dp)[16]) {
  const size_t row0 = (size_t)(T.slot0 + c0);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const bool hi = lane & 16;
    const float send = hi ? dp[j] : dp[j + 8];
    dp[j] = (hi ? dp[j + 8] : dp[j]) + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool hi = lane & 8;
    const float send = hi ? dp[j] : dp[j + 4];
    dp[j] = (hi ? dp[j + 4] : dp[j]) + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const bool hi = lane & 4;
    const float send = hi ? dp[j] : dp[j + 2];
    dp[j] = (hi ? dp[j + 2] : dp[j]) + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
  }
  {
    const bool hi = lane & 2;
    const float send = hi ? dp[0] : dp[1];
    dp[0] = (hi ? dp[1] : dp[0]) + __shfl_xor_sync(0xFFFFFFFFu, send, 2);
  }
  dp[0] += __shfl_xor_sync(0xFFFFFFFFu, dp[0], 1);
  const int m = lane >> 1;
  if ((lane & 1) == 0 && c0 + m < T.rows)
    p.part[(row0 + m) * (size_t)(p.inter / 32) + feat0 / 32] = dp[0];
}

// Epilogue of the FC2 dgrad for 16 slots (registers) x 32 features (lanes).
// dA0[s,i] = dY[t_s] . W_down[e][i,:] arrives in v; with g, u the saved
// pre-activations (gu) and p' the slot's routing probability (ps):
//   a = act(g) u,  dprob part = sum_i a dA0,  dA = p' dA0,
//   dg = dA u act'(g),  du = dA act(g),  aw = p' a.
// dg and du go to dPre (gate columns, then up columns), aw to out2, and the
// 32-feature partial sum of a dA0 of each slot to part[s, feat0/32]. Padding
// slots get zeros (their dA0, g, u and p' are 0).
template <int act>
__device__ __forceinline__ void swiglu_backward_chunk(const GemmParams& p, const Tile& T, int c0,
                                                      int feat0, int lane, uint32_t stg_u,
                                                      uint32_t stg2_u, const uint32_t (&v)[16],
                                                      const uint32_t (&gu)[16], const float* ps) {
  const int I = p.inter;
  const int ld2 = 2 * I;
  const size_t row0 = (size_t)(T.slot0 + c0);
  // One pass over each half of 8 slots: act's factor c (sigma or Phi) once
  // per element, all three outputs staged as bf16 in the warp's three
  // 512-byte buffers (dg in stg_u, du and aw in stg2_u), then each lane
  // copies 16 bytes of each output row. (One pass per output, recomputing c,
  // made this epilogue instruction-bound: ~1 us a chunk, ~24 us a tile.)
  const uint32_t st_dg = stg_u, st_du = stg2_u, st_aw = stg2_u + 512u;
  float dp[16];
#pragma unroll
  for (int h8 = 0; h8 < 2; ++h8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = h8 * 8 + i;
      const float g = __uint_as_float(gu[j] << 16), u = __uint_as_float(gu[j] & 0xFFFF0000u);
      const float da0 = __uint_as_float(v[j]), pj = ps[c0 + j];
      const float c = act_core<act>(g);
      const float a = g * c;  // act(g)
      const float au = a * u;
      dp[j] = au * da0;
      const float dA = pj * da0;
      const uint32_t at = (uint32_t)(i * kStageRowElems + lane) * 2u;
      asm volatile("st.shared.b16 [%0], %1;" ::"r"(st_dg + at),
                   "h"((unsigned short)bf16_bits(dA * u * act_grad_core<act>(g, c)))
                   : "memory");
      asm volatile("st.shared.b16 [%0], %1;" ::"r"(st_du + at),
                   "h"((unsigned short)bf16_bits(dA * a))
                   : "memory");
      asm volatile("st.shared.b16 [%0], %1;" ::"r"(st_aw + at),
                   "h"((unsigned short)bf16_bits(pj * au))
                   : "memory");
    }
    __syncwarp();
    const int row = lane >> 2, part = lane & 3;  // 8 rows x 4 chunks of 16 bytes
    const uint32_t rd = (uint32_t)(row * kStageRowElems + part * 8) * 2u;
    const size_t r = row0 + (size_t)(h8 * 8 + row);
    auto copy16 = [&](uint32_t src, uint16_t* dst) {
      uint4 val;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                   : "r"(src)
                   : "memory");
      *reinterpret_cast<uint4*>(dst) = val;
    };
    copy16(st_dg + rd, p.out + r * ld2 + feat0 + part * 8);
    copy16(st_du + rd, p.out + r * ld2 + I + feat0 + part * 8);
    copy16(st_aw + rd, p.out2 + r * I + feat0 + part * 8);
    __syncwarp();
  }
  dprob_part16(p, T, c0, feat0, lane, dp);
}

// One instantiation per GemmMode (and per activation for the modes that apply
// one), so each carries only its own code path.
//
// kPair = 1: the CTAs run as pairs (clusters of two) on one tile. Each CTA
// loads its own 128 rows of every accumulator's weights and half of the
// tile's B rows (slots [r*N/2, (r+1)*N/2) for CTA r), and holds its 128
// accumulator rows in its TMEM; the even CTA issues the pair's M = 256 MMAs
// (tcgen05 cta_group::2), which read both CTAs' shared memory. So a stage
// holds half the B rows a one-CTA tile would, and each CTA's epilogue works on
// its own features. Roles beyond the one-CTA ones: the even CTA's scheduler
// publishes each tile to both CTAs; the odd CTA's warp 0 is only its producer
// and its warp 1 relays "stage full" to the even CTA's barrier; the MMA
// commits multicast their arrivals to both CTAs; the odd CTA's epilogue warps
// release the accumulator on the even CTA's barrier.
template <int kMode, int kAct, int kPair>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB2, const GemmParams p) {
  constexpr bool kP = kPair != 0;
  constexpr bool kGatherB = kMode == kModeFc1 || kMode == kModeDgrad2 || kMode == kModeFc1Fp8 ||
                            kMode == kModeFc1Mx;
  constexpr bool kMx = kMode == kModeFc1Mx || kMode == kModeFc2Mx;
  // warps 10-13 copy B rows (gathered modes) and, in the MX modes, the B rows'
  // scale bytes
  constexpr bool kGatherWarps = kGatherB || kMx;
  constexpr bool kFc1 = kMode == kModeFc1 || kMode == kModeFc1Fp8 || kMode == kModeFc1Mx;
  constexpr bool kFp8 = kMode == kModeFc1Fp8 || kMode == kModeFc2Fp8;
  constexpr bool kAMn = kMode == kModeDgrad2 || kMode == kModeDgrad1;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t tmem_full_bar[2];
  __shared__ __align__(8) uint64_t tmem_empty_bar[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int32_t tpre[kMaxExperts + 1];
  __shared__ int32_t ttn[kMaxExperts];
  __shared__ int32_t tile_q[kTileQ];
  __shared__ __align__(8) uint64_t tq_full[kTileQ];
  __shared__ __align__(8) uint64_t tq_empty[kTileQ];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  const uint32_t crank = kP ? cluster_ctarank() : 0u;
  const bool lead = crank == 0u;  // the CTA that schedules and issues the MMAs

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      // pair mode, even CTA: one more arrival per phase, the odd CTA's relay
      mbar_init(smem_u32(&full_bar[s]),
                (kGatherWarps ? 1 + kGatherThreads : 1) + (kP && lead ? 1 : 0));
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tmem_full_bar[b]), 1);
      // one arrive per epilogue warp (pair mode: of both CTAs, on the even one's)
      mbar_init(smem_u32(&tmem_empty_bar[b]), kEpiWarps * (kP ? 2 : 1));
    }
    for (int i = 0; i < kTileQ; ++i) {
      mbar_init(smem_u32(&tq_full[i]), 1);
      // consumers: the UMMA thread, the epilogue warps, the 4 gather warps (FC1);
      // pair mode adds the odd CTA's producer, relay, epilogue and gather warps
      mbar_init(smem_u32(&tq_empty[i]), 1 + kEpiWarps + (kGatherWarps ? 4 : 0) +
                                            (kP ? 2 + kEpiWarps + (kGatherWarps ? 4 : 0) : 0));
    }
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    if (!kGatherB) {
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmB2);
    }
    if (kAMn) tma_prefetch_desc(&tmA2);
  }
  if (warp == 1) {
    if constexpr (kP)
      tmem_alloc_pair(smem_u32(&tmem_base_s), kTmemCols);
    else
      tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
  }
  // the setup above touches no global memory; the tile list reads the counts
  // the previous kernel wrote
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 0) build_tile_list(p, tpre, ttn, lane);
  tc_fence_before();
  __syncthreads();
  // pair mode: both CTAs' barriers are initialised before either signals the other
  if constexpr (kP) cluster_sync_all();
  const int n_tiles = tpre[p.E];
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  // pair mode: a barrier of this CTA at the same offset in the even CTA
  auto at_lead = [&](const void* local) -> uint32_t {
    return kP ? mapa_shared(smem_u32(local), 0u) : smem_u32(local);
  };
  // waits on barriers that the other CTA of a pair signals take cluster scope
  auto wait_warp = [&](uint32_t bar, uint32_t parity, uint32_t code) -> bool {
    if constexpr (kP)
      return mbar_wait_cluster_warp(bar, parity, p.err, code);
    else
      return mbar_wait_warp(bar, parity, p.err, code);
  };

  // Pops the next tile id (lane 0 waits, the warp gets the value); -1 ends.
  auto pop_tile = [&](uint32_t& qi, uint32_t code) -> int {
    const int slot = (int)(qi % kTileQ);
    const bool ok = wait_warp(smem_u32(&tq_full[slot]), (qi / kTileQ) & 1u, code);
    const int t = ok ? tile_q[slot] : -1;
    __syncwarp();
    if (lane == 0) {
      if (kP && !lead)
        mbar_arrive_remote_relaxed(at_lead(&tq_empty[slot]));
      else
        mbar_arrive(smem_u32(&tq_empty[slot]));
    }
    ++qi;
    return t;
  };
  // this CTA's first feature of tile T, and its share of the tile's B rows
  auto feat_base = [&](const Tile& T) -> int { return T.f * p.f_rows + (int)crank * p.f_cta; };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    // Also the scheduler: takes the next non-empty tile from the global counter
    // and publishes it to the other roles.
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    uint32_t gk = 0;  // k-steps issued by this CTA, across tiles
    uint32_t pq = 0;  // pair mode, odd CTA: tiles popped
    for (uint32_t qi = 0;; ++qi) {
      int t = -1;
      if (kP && !lead) {
        t = pop_tile(pq, kErrWaitFull);  // the odd CTA takes the even CTA's tile
      } else {
        const int slot = (int)(qi % kTileQ);
        const bool free_ok =
            qi < (uint32_t)kTileQ ||
            wait_warp(smem_u32(&tq_empty[slot]), ((qi / kTileQ) - 1u) & 1u, kErrWaitEmpty);
        if (lane == 0) {
          if (free_ok) t = atomicAdd(&p.sched[0], 1);
          if (t >= n_tiles) t = -1;
          tile_q[slot] = t;
          if constexpr (kP) {  // publish to the odd CTA too
            st_shared_remote_u32(mapa_shared(smem_u32(&tile_q[slot]), 1u), (uint32_t)t);
            mbar_arrive_remote(mapa_shared(smem_u32(&tq_full[slot]), 1u));
          }
          mbar_arrive(smem_u32(&tq_full[slot]));
        }
        t = __shfl_sync(0xFFFFFFFFu, t, 0);
      }
      if (t < 0) break;
      Tile T;
      tile_at(p, tpre, ttn, t, T);
      // K-major A: rows e*a_rows_per_expert + f*f_rows, k along the row.
      // MN-major A: the weight matrix read transposed; its rows are k
      // (e*a_rows_per_expert + k) and the tile's features are 64-wide column
      // chunks, all of them fetched by one 3-D copy ([chunk][row][64]; one copy
      // instead of one per chunk took the FC1 dgrad from 1.93 to 1.70 ms on
      // the dropless shape).
      const int fb0 = feat_base(T);
      const int a_row0 = T.e * p.a_rows_per_expert + (kAMn ? 0 : fb0);
      const int a_col0 = fb0;
      // pair mode: this CTA's B rows (half of the tile's)
      const int b_rows = kP ? T.n_eff / 2 : T.n_eff;
      const int b_row0 = T.slot0 + (int)crank * b_rows;
      constexpr int kBox = kP ? kBBoxRowsPair : kBBoxRows;
      constexpr int kBoxS = kP ? kBBoxRowsPairSmall : kBBoxRowsSmall;
      const int b_big = b_rows / kBox * kBox;  // rows in whole large boxes
      const uint32_t tx = (uint32_t)T.nacc * kATileBytes +
                          (kGatherB ? 0u : (uint32_t)b_rows * 128u) +
                          (kMx ? (uint32_t)T.nacc * 512u : 0u);
      bool ok = true;
      for (int kt = 0; kt < p.k_tiles; ++kt, ++gk) {
        const int s = (int)(gk % (uint32_t)p.stages);
        const uint32_t u = gk / (uint32_t)p.stages;
        if (gk >= (uint32_t)p.stages &&
            !mbar_wait_warp(smem_u32(&empty_bar[s]), (u & 1u) ^ 1u, p.err, kErrWaitEmpty)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t st = sbase + (uint32_t)s * p.stage_bytes;
        const int kx = kt * kBK;
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, tx);
          if (kAMn) {
            // every chunk of the tile's accumulators in one copy: [chunk][row][64]
            if (T.nacc == 2)
              tma_load_3d(st, &tmA, 0, a_row0 + kx, a_col0 / 64, fb, pol_w);
            else
              tma_load_3d(st, &tmA2, 0, a_row0 + kx, a_col0 / 64, fb, pol_w);
          } else {
            tma_load_2d(st, &tmA, kx, a_row0, fb, pol_w);
            if (T.nacc == 2)
              tma_load_2d(st + kATileBytes, &tmA, kx, a_row0 + p.a_second_off, fb, pol_w);
          }
          if constexpr (kMx) {
            // the weight rows' scale atom of this k tile, one per accumulator
            for (int a2 = 0; a2 < T.nacc; ++a2) {
              const int row = a_row0 + a2 * p.a_second_off;
              bulk_load(st + p.sf_off + 512u * (uint32_t)a2,
                        p.sfa + ((size_t)(row / kTileM) * p.k_tiles + kt) * 512u, 512u, fb);
            }
          }
        }
        __syncwarp();
        if (!kGatherB) {
          const uint32_t b = st + p.b_off;
          for (int q = lane * kBox; q < b_big; q += 32 * kBox)
            tma_load_2d(b + (uint32_t)q * 128u, &tmB, kx, b_row0 + q, fb, pol_x);
          for (int q = b_big + lane * kBoxS; q < b_rows; q += 32 * kBoxS)
            tma_load_2d(b + (uint32_t)q * 128u, &tmB2, kx, b_row0 + q, fb, pol_x);
        }
      }
      if (!ok) break;
    }
    if (lane == 0) {
      // every CTA has made its last fetch before counting itself finished, so
      // the last one to finish may reset the counter for the next launch
      __threadfence();
      if (atomicAdd(&p.sched[1], 1) == (int)gridDim.x - 1) {
        atomicExch(&p.sched[0], 0);
        atomicExch(&p.sched[1], 0);
        __threadfence();
      }
    }
  } else if (kP && !lead && warp == 1) {
    // ---------------------------------------------------------------- pair relay
    // The odd CTA issues no MMAs: this warp tells the even CTA's MMA thread
    // when each of this CTA's stages is full (its TMA bytes and its gathered
    // rows have landed), ordering the gathered rows' generic-proxy writes
    // before the tensor core's reads.
    uint32_t gk = 0, qi = 0;
    for (bool ok = true; ok;) {
      const int t = pop_tile(qi, kErrWaitFull);
      if (t < 0) break;
      for (int kt = 0; kt < p.k_tiles; ++kt, ++gk) {
        const int s = (int)(gk % (uint32_t)p.stages);
        const uint32_t u = gk / (uint32_t)p.stages;
        if (!mbar_wait_warp(smem_u32(&full_bar[s]), u & 1u, p.err, kErrWaitFull)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          if (kGatherWarps) fence_proxy_async_smem();
          mbar_arrive_remote_relaxed(at_lead(&full_bar[s]));
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- UMMA issuer
    // The whole warp walks the tiles and takes the waits; lane 0 issues.
    // Pair mode (even CTA): the MMAs are the pair's (M = 256), the waits take
    // cluster scope, and the commits arrive on both CTAs' barriers.
    uint32_t gk = 0, tc = 0, qi = 0;
    for (;;) {
      const int t = pop_tile(qi, kErrWaitFull);
      if (t < 0) break;
      Tile T;
      tile_at(p, tpre, ttn, t, T);
      // accumulator buffer: two in flight when one tile uses 256 columns
      const uint32_t ab = tc % (uint32_t)p.n_buf, au = tc / (uint32_t)p.n_buf;
      if (au > 0 && !wait_warp(smem_u32(&tmem_empty_bar[ab]), (au - 1) & 1u, kErrWaitAccum))
        break;
      tc_fence_after();
      const uint32_t dacc = tmem + ab * p.buf_stride;
      const uint32_t idesc =
          kFp8 ? idesc_e4m3_f32(kTileM, T.n_eff)
               : (idesc_bf16_f32(kP ? 2 * kTileM : kTileM, T.n_eff) | (kAMn ? kIdescAMnMajor : 0u));
      // one UMMA k-step (16 elements) advances 32 bytes along a K-major row,
      // or 16 rows of 128 bytes in an MN-major tile
      constexpr uint32_t a_kstep = kAMn ? 2048u : 32u;
      bool ok = true;
      for (int kt = 0; kt < p.k_tiles; ++kt, ++gk) {
        const int s = (int)(gk % (uint32_t)p.stages);
        const uint32_t u = gk / (uint32_t)p.stages;
        if (!wait_warp(smem_u32(&full_bar[s]), u & 1u, kErrWaitFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          // B rows written by cp.async (generic proxy) are read by the tensor core
          if (kGatherWarps) fence_proxy_async_smem();
          const uint32_t st = sbase + (uint32_t)s * p.stage_bytes;
          if constexpr (kMx) {
            // this stage's scales into its TMEM columns: A atoms at +0 / +4, B
            // atoms (128 rows each) at +8 / +12; the copies run before this
            // thread's MMAs below
            const uint32_t sft = tmem + p.sf_tmem + 16u * (uint32_t)s;
            for (int a2 = 0; a2 < T.nacc; ++a2)
              tmem_cp_32x128b_x4(sft + 4u * (uint32_t)a2,
                                 sdesc_rows16(st + p.sf_off + 512u * (uint32_t)a2));
            for (int g = 0; g * kTileM < T.n_eff; ++g)
              tmem_cp_32x128b_x4(sft + 8u + 4u * (uint32_t)g,
                                 sdesc_rows16(st + p.sf_off + 1024u + 512u * (uint32_t)g));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // one 32-value scale block per k-step
              const uint32_t acc = (kt | kk) != 0;
              const uint32_t id = idesc_mx_e4m3(kTileM, T.n_eff, kk, kk);
              const uint64_t bdesc = sdesc_sw128(st + p.b_off + (uint32_t)kk * 32u);
              const uint32_t a0 = st + (uint32_t)kk * 32u;
              umma_mx(dacc, sdesc_sw128(a0), bdesc, id, sft, sft + 8u, acc);
              if (T.nacc == 2)
                umma_mx(dacc + p.acc_off, sdesc_sw128(a0 + kATileBytes), bdesc, id, sft + 4u,
                        sft + 8u, acc);
            }
          }
#pragma unroll
          for (int kk = 0; kk < (kMx ? 0 : kBK / 16); ++kk) {
            const uint32_t acc = (kt | kk) != 0;
            const uint64_t bdesc = sdesc_sw128(st + p.b_off + (uint32_t)kk * 32u);
            const uint32_t a0 = st + (uint32_t)kk * a_kstep;
            if constexpr (kFp8) {  // 32 E4M3 values = the same 32 bytes per k-step
              umma_fp8(dacc, sdesc_sw128(a0), bdesc, idesc, acc);
              if (T.nacc == 2) umma_fp8(dacc + p.acc_off, sdesc_sw128(a0 + kATileBytes), bdesc, idesc, acc);
            } else if constexpr (kP) {
              umma_bf16_pair(dacc, kAMn ? sdesc_sw128_mn(a0) : sdesc_sw128(a0), bdesc, idesc, acc);
              if (T.nacc == 2) {
                const uint32_t a1 = a0 + kATileBytes;
                umma_bf16_pair(dacc + p.acc_off, kAMn ? sdesc_sw128_mn(a1) : sdesc_sw128(a1),
                               bdesc, idesc, acc);
              }
            } else {
              umma_bf16(dacc, kAMn ? sdesc_sw128_mn(a0) : sdesc_sw128(a0), bdesc, idesc, acc);
              if (T.nacc == 2) {
                const uint32_t a1 = a0 + kATileBytes;
                umma_bf16(dacc + p.acc_off, kAMn ? sdesc_sw128_mn(a1) : sdesc_sw128(a1), bdesc,
                          idesc, acc);
              }
            }
          }
          if constexpr (kP)
            umma_commit_pair(smem_u32(&empty_bar[s]), 3);
          else
            umma_commit(smem_u32(&empty_bar[s]));
        }
        __syncwarp();
      }
      if (lane == 0) {  // also after an abort
        if constexpr (kP)
          umma_commit_pair(smem_u32(&tmem_full_bar[ab]), 3);
        else
          umma_commit(smem_u32(&tmem_full_bar[ab]));
      }
      __syncwarp();
      ++tc;
      if (!ok) break;
    }
  } else if (warp < 2 + kEpiWarps) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;  // which of the two warps of this lane quarter
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t stg_u = sbase + p.epi_off + (uint32_t)(warp - 2) * 8u * kStageRowElems * 2u;
    // FC2 dgrad: this warp's 16 p' values of the current chunk
    float* ps_w = reinterpret_cast<float*>(smem_raw + (sbase - smem_u32(smem_raw)) + p.ps_off) +
                  (warp - 2) * 16;
    // FC2 dgrad: the next chunk's pre-activations wait in this warp's 2 KB of
    // shared memory (row r: gate features at r*128, up at r*128 + 64),
    // fetched with 16-byte cp.async copies, instead of in 16 registers
    // filled by 2-byte loads (with gelu, whose backward keeps Phi of 16
    // values live, the register form spilled past the 128 registers)
    const uint32_t pre_u = sbase + p.xs_off + (uint32_t)(warp - 2) * 2048u;
    // FC2 dgrad: this warp's two more 512-byte output staging buffers
    const uint32_t stg2_u = sbase + p.xs_off + kPreBufBytes + (uint32_t)(warp - 2) * 1024u;
    auto prefetch_preact = [&](const Tile& T, int c, int f0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int pi = lane + 32 * k;  // 16 rows x (4 gate + 4 up) 16-byte pieces
        const int r = pi >> 3, gsel = (pi >> 2) & 1, qq = pi & 3;
        const bool ok = c + r < T.rows;
        const uint16_t* src = p.aux + (size_t)(T.slot0 + (ok ? c + r : 0)) * (2 * p.inter) +
                              (gsel ? p.inter : 0) + f0 + qq * 8;
        cp_async_16(pre_u + (uint32_t)(r * 128 + gsel * 64 + qq * 16), src, ok ? 16u : 0u);
      }
      cp_async_commit();
    };
    auto read_preact = [&](uint32_t (&gu)[16]) {
      cp_async_wait_all();
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        uint16_t g, u;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(g) : "r"(pre_u + (uint32_t)(j * 128 + lane * 2)));
        asm volatile("ld.shared.u16 %0, [%1];"
                     : "=h"(u)
                     : "r"(pre_u + (uint32_t)(j * 128 + 64 + lane * 2)));
        gu[j] = (uint32_t)g | ((uint32_t)u << 16);
      }
      __syncwarp();  // every lane has its values before the buffer is refilled
    };
    uint32_t tc = 0, qi = 0;
    for (;;) {
      const int t = pop_tile(qi, kErrWaitAccum);
      if (t < 0) break;
      Tile T;
      tile_at(p, tpre, ttn, t, T);
      const uint32_t ab = tc % (uint32_t)p.n_buf, au = tc / (uint32_t)p.n_buf;
      const int fbt = feat_base(T);
      const int feat0 = fbt + q * 32;  // first feature of this lane quarter
      // accumulators whose features this CTA writes: all of the tile's, except
      // in a pair whose last feature tile is ragged (the odd CTA's 128-row
      // halves past the last feature are computed but not stored)
      int na = T.nacc;
      if constexpr (kP) {
        if (p.pair_feats)
          na = (fbt >= p.m_total) ? 0 : (fbt + kTileM >= p.m_total ? min(T.nacc, 1) : T.nacc);
        else
          na = fbt < p.m_total ? T.nacc : 0;
      }
      const int nch = na > 0 ? (T.n_eff - half * 16 + 31) / 32 : 0;  // this warp's 16-slot chunks
      float p_next = 0.0f;
      float wsg = 1.0f, wsu = 1.0f;
      if constexpr (kFp8) {
        // before the accumulator is ready: this lane's row scale of each
        // accumulator (FC1: gate and up rows; FC2: the two 128-row halves of
        // the feature tile), and the B-row scale of every slot of the warp's
        // chunks (slot c0 + j of chunk m at xs_w[16m + j]) into the warp's
        // own slice; the previous tile's readers of the slice passed the
        // warp barrier that ends each chunk's stores
        if constexpr (kMode == kModeFc1Fp8) {
          const int rg = T.e * 2 * p.inter + feat0 + lane;
          wsg = p.w_scale[rg];
          wsu = p.w_scale[rg + p.inter];
        } else {
          const int rg = T.e * p.m_total + feat0 + lane;
          wsg = p.w_scale[rg];
          if (T.nacc == 2) wsu = p.w_scale[rg + kTileM];
        }
        float* xs_w = reinterpret_cast<float*>(smem_raw + (sbase - smem_u32(smem_raw)) + p.xs_off) +
                      (warp - 2) * 128;
        for (int i = lane; i < 16 * nch; i += 32) {
          const int c = half * 16 + 32 * (i >> 4) + (i & 15);
          float v = 0.0f;
          if (c < T.rows) {
            if constexpr (kMode == kModeFc1Fp8) {
              const int tok = p.sorted_slot_ids[T.slot0 + c];
              if ((unsigned)tok < (unsigned)p.act_rows) v = p.x_scale[tok];
            } else {
              v = p.x_scale[T.slot0 + c];
            }
          }
          xs_w[i] = v;
        }
        __syncwarp();
      }
      if (kMode == kModeDgrad2 && nch > 0) {
        // before the accumulator is ready: the first chunk's pre-activations
        // and p' (lane j < 16 holds slot j's)
        prefetch_preact(T, half * 16, feat0);
        p_next = load_slot_prob(p, T, half * 16, lane);
      }
      // the warp's vote: the warp-collective TMEM loads below are reached by
      // all lanes or by none
      const bool w = wait_warp(smem_u32(&tmem_full_bar[ab]), au & 1u, kErrWaitAccum);
      ++tc;
      if (!w) break;
      tc_fence_after();
      const uint32_t ta = tl + ab * p.buf_stride;
      if constexpr (kMode == kModeDgrad2) {
        // chunks of accumulator 0, then of accumulator 1; the next chunk's
        // operands load under this chunk's math
        const int total = na * nch;
        for (int it = 0; it < total; ++it) {
          const int a = it / nch, c0 = half * 16 + 32 * (it - a * nch);
          uint32_t gu[16];  // gate in the low half, up in the high half of each word
          read_preact(gu);
          const float p_cur = p_next;
          if (it + 1 < total) {
            const int a2 = (it + 1) / nch, c2 = half * 16 + 32 * (it + 1 - a2 * nch);
            prefetch_preact(T, c2, feat0 + a2 * kTileM);
            p_next = load_slot_prob(p, T, c2, lane);
          }
          uint32_t v[16];
          tmem_ld16(ta + (uint32_t)a * p.acc_off + (uint32_t)c0, v);
          tmem_ld_wait();
          if (lane < 16) ps_w[lane] = p_cur;
          __syncwarp();
          swiglu_backward_chunk<kAct>(p, T, c0, feat0 + a * kTileM, lane, stg_u, stg2_u, v, gu,
                                      ps_w - c0);
        }
      } else {
        for (int c0 = half * 16; c0 < (na > 0 ? T.n_eff : 0); c0 += 32) {
          uint32_t v0[16], v1[16];
          tmem_ld16(ta + (uint32_t)c0, v0);
          if (T.nacc == 2) tmem_ld16(ta + p.acc_off + (uint32_t)c0, v1);
          tmem_ld_wait();
          const size_t row0 = (size_t)(T.slot0 + c0);  // slot of register 0
          if constexpr (kFc1) {
            // p' of the chunk's slots (lane j < 16 holds slot j's) when the
            // routing probability multiplies the activation
            const float pl = p.prob_in_act ? load_slot_prob(p, T, c0, lane) : 1.0f;
            const float* xs_c =
                reinterpret_cast<const float*>(smem_raw + (sbase - smem_u32(smem_raw)) + p.xs_off) +
                (warp - 2) * 128 + 16 * ((c0 - half * 16) >> 5);
            float hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float g = __uint_as_float(v0[i]), u = __uint_as_float(v1[i]);
              if constexpr (kFp8) {  // dequantise: row scale x token scale
                g *= wsg * xs_c[i];
                u *= wsu * xs_c[i];
              }
              hv[i] = act_fwd<kAct>(g) * u;
              if (p.prob_in_act) hv[i] *= __shfl_sync(0xFFFFFFFFu, pl, i);
            }
            store_rows16(stg_u, lane, hv, p.out + row0 * p.out_ld + feat0, p.out_ld);
            if (p.out2) {  // pre-activations for the backward: gate, then up
              float gv[16], uv[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                gv[i] = __uint_as_float(v0[i]);
                uv[i] = __uint_as_float(v1[i]);
              }
              const int ld2 = 2 * p.inter;
              store_rows16(stg_u, lane, gv, p.out2 + row0 * ld2 + feat0, ld2);
              store_rows16(stg_u, lane, uv, p.out2 + row0 * ld2 + p.inter + feat0, ld2);
            }
          } else {
            const float* xs_c =
                reinterpret_cast<const float*>(smem_raw + (sbase - smem_u32(smem_raw)) + p.xs_off) +
                (warp - 2) * 128 + 16 * ((c0 - half * 16) >> 5);
            for (int seg = 0; seg < na; ++seg) {
              float ov[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                ov[i] = __uint_as_float(seg == 0 ? v0[i] : v1[i]);
                if constexpr (kFp8) ov[i] *= (seg == 0 ? wsg : wsu) * xs_c[i];
              }
              store_rows16(stg_u, lane, ov, p.out + row0 * p.out_ld + feat0 + seg * kTileM,
                           p.out_ld);
            }
          }
        }
      }
      tc_fence_before();
      if (lane == 0) {
        if (kP && !lead)
          mbar_arrive_remote_relaxed(at_lead(&tmem_empty_bar[ab]));
        else
          mbar_arrive(smem_u32(&tmem_empty_bar[ab]));
      }
    }
  } else if (kGatherWarps) {
    // ---------------------------------------------------------------- B row gather
    // Row r of a stage holds act[sorted_slot_ids[slot0 + r], kx .. kx+63]:
    // 16-byte chunk c at r*128 + ((c ^ (r%8)) * 16), the 128-byte swizzle the
    // UMMA descriptor expects; sentinel rows are zero-filled. Thread gt copies
    // chunk c = gt%8 of rows r = gt/8 + 16i (i < n_eff/16) of every stage; it
    // looks its rows' token offsets up once per tile, so each copy is one
    // address add and one cp.async. A thread does not wait for its copies: the
    // stage's full barrier receives its arrival when they complete
    // (cp.async.mbarrier.arrive.noinc), so the gather runs as many stages ahead
    // as the ring holds; the UMMA thread fences the generic-proxy writes
    // against its async-proxy operand reads after the barrier. Waits end in a
    // warp vote, so a warp leaves together when one runs out.
    const int gt = threadIdx.x - kGatherWarp0 * 32;
    const int c = gt & 7, rb = gt >> 3;
    const uint32_t dst0 = (uint32_t)rb * 128u + ((uint32_t)(c ^ (rb & 7)) << 4);
    uint32_t gk = 0, qi = 0;
    bool ok = true;
    while (ok) {
      const int t = pop_tile(qi, kErrWaitFull);
      if (t < 0) break;
      Tile T;
      tile_at(p, tpre, ttn, t, T);
      // this CTA's B rows: all of the tile's, or in a pair the half
      // [crank*N/2, (crank+1)*N/2), in 16-row passes
      const int g_rows = kP ? T.n_eff / 2 : T.n_eff;
      const int g_off = kP ? (int)crank * g_rows : 0;
      const int n_i = (g_rows - rb + 15) >> 4;  // rows rb + 16i below g_rows
      // MX: the scale rows this thread copies (rows gt and gt + 128 of the
      // tile), looked up once per tile; -1 for a row past the tile's routes or
      // a sentinel token (zero scale bytes)
      int sf_row[2] = {-1, -1};
      if constexpr (kMx) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int r = gt + j * kGatherThreads;
          if (r < T.rows) {
            if constexpr (kMode == kModeFc1Mx) {
              const int tok = p.sorted_slot_ids[T.slot0 + r];
              sf_row[j] = (unsigned)tok < (unsigned)p.act_rows ? tok : -1;
            } else {
              sf_row[j] = T.slot0 + r;
            }
          }
        }
      }
      uint32_t off[16];
      uint32_t vmask = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        off[i] = 0;
        if (kGatherB && i < n_i) {
          const int tok = p.sorted_slot_ids[T.slot0 + g_off + rb + 16 * i];
          if ((unsigned)tok < (unsigned)p.act_rows) {
            // MX: the token itself (its scale row); otherwise its element offset
            off[i] = kMx ? (uint32_t)tok : (uint32_t)tok * (uint32_t)p.act_ld + (uint32_t)(c * 8);
            vmask |= 1u << i;
          }
        }
      }
      for (int kt = 0; kt < p.k_tiles; ++kt, ++gk) {
        const int s = (int)(gk % (uint32_t)p.stages);
        const uint32_t u = gk / (uint32_t)p.stages;
        if (gk >= (uint32_t)p.stages &&
            !mbar_wait_warp(smem_u32(&empty_bar[s]), (u & 1u) ^ 1u, p.err, kErrWaitEmpty)) {
          ok = false;
          break;
        }
        const uint32_t stb = sbase + (uint32_t)s * p.stage_bytes;
        if constexpr (kGatherB) {
          const uint32_t b = stb + p.b_off + dst0;
          const uint16_t* src = p.act + kt * kBK;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (i < n_i) {
              const uint32_t eo = kMx ? off[i] * (uint32_t)p.act_ld + (uint32_t)(c * 8) : off[i];
              cp_async_16(b + (uint32_t)i * 2048u, src + eo, ((vmask >> i) & 1u) << 4);
            }
          }
        }
        if constexpr (kMx) {
          // the B rows' scale bytes of this k tile (4 blocks of 32) into the
          // stage's B atoms: row r at (r/128)*512 + (r%32)*16 + ((r%128)/32)*4;
          // every gather thread copies at most two rows, so a stage's scales
          // take one 4-byte copy per thread
          const uint32_t sfb_s = stb + p.sf_off + 1024u;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int r = gt + j * kGatherThreads;
            if (r < T.n_eff) {
              const uint32_t d = sfb_s + (uint32_t)((r >> 7) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4);
              const int row = sf_row[j] < 0 ? 0 : sf_row[j];
              cp_async_4(d, p.sfb + (size_t)row * p.sfb_ld + kt * 4, sf_row[j] < 0 ? 0u : 4u);
            }
          }
        }
        cp_async_mbar_arrive_noinc(smem_u32(&full_bar[s]));
      }
    }
    cp_async_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  // pair mode: neither CTA leaves (or frees its TMEM) while the other may still
  // signal its barriers or have MMAs write its accumulators
  if constexpr (kP) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kP)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

template <int kMode, int kAct, int kPair = 0>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(moe_gemm_kernel<kMode, kAct, kPair>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
}

// Whether a GEMM runs as CTA pairs (cta_group::2 tiles): the bf16 forward
// GEMMs with a short contraction, where each tile's fixed costs weigh most and
// halving the B rows each CTA stages pays (Qwen3-30B-shaped layer, H = 2048,
// I = 768: FC1 0.217 -> 0.211 ms, FC2 0.136 -> 0.134 ms). With longer
// contractions pairs measured slower (DeepSeek-V3-shaped FC1 2.39 -> 2.40,
// FC2 1.26 -> 1.29 ms; the dropless layer's forward 2.63 -> 2.76 ms, its
// dgrads as pairs 7.03 -> 7.08 ms).
bool pair_mode(int mode, int H, int I) {
  return (mode == kModeFc1 && H <= 2048) || (mode == kModeFc2 && I <= 1024);
}

// SM count of the current device, with every instantiation's shared-memory
// opt-in set up once per device.
int device_sms(cudaError_t* err) {
  static DeviceOnce sms;
  int n = 0;
  *err = once_per_device(sms, &n, [](int dev, int* v) {
    cudaError_t e = cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if ((e = set_smem_attr<kModeFc1, 0>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc1, 1>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc1Fp8, 0>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc1Fp8, 1>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc2, 0>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc2Fp8, 0>()) != cudaSuccess ||
        (e = set_smem_attr<kModeDgrad2, 0>()) != cudaSuccess ||
        (e = set_smem_attr<kModeDgrad2, 1>()) != cudaSuccess ||
        (e = set_smem_attr<kModeDgrad1, 0>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc1Mx, 0>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc1Mx, 1>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc2Mx, 0>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc1, 0, 1>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc1, 1, 1>()) != cudaSuccess ||
        (e = set_smem_attr<kModeFc2, 0, 1>()) != cudaSuccess)
      cudaGetLastError();  // reported here; do not leave it for a later launch to report
    return e;
  });
  return *err == cudaSuccess ? n : 0;
}

}  // namespace

int launch_gemm(const GemmArgs& a, cudaStream_t s) {
  if (a.max_rows <= 0 || a.N <= 0) return 0;
  GemmParams p{};
  const bool gather_b = a.mode == kModeFc1 || a.mode == kModeDgrad2 || a.mode == kModeFc1Fp8 ||
                        a.mode == kModeFc1Mx;
  const bool mx = a.mode == kModeFc1Mx || a.mode == kModeFc2Mx;
  p.bm = a.bm;
  p.sorted_slot_ids = a.sorted_slot_ids;
  p.kept_counts = a.kept_counts;
  p.block_start = a.block_start;
  p.out = static_cast<uint16_t*>(a.out);
  p.out2 = static_cast<uint16_t*>(a.out2);
  p.aux = static_cast<const uint16_t*>(a.aux);
  p.slot_prob = a.slot_prob;
  p.activation = a.activation;
  p.w_scale = a.w_scale;
  p.x_scale = a.x_scale;
  p.prob_in_act = a.prob_in_act;
  p.part = a.part;
  p.inter = a.I;
  p.err = a.err;
  p.act = static_cast<const uint16_t*>(a.act);
  p.act_rows = gather_b ? a.N : 0;
  const int64_t S = a.s_max;
  const uint64_t E = (uint64_t)a.E;
  CUtensorMap tmA{}, tmB{}, tmA2{}, tmB2{};
  // a slot-indexed B operand [S, cols]: large and small boxes
  auto make_b = [&](const void* base, uint64_t cols) -> bool {
    return make_map(&tmB, base, cols, (uint64_t)S, kBK, kBBoxRows) &&
           make_map(&tmB2, base, cols, (uint64_t)S, kBK, kBBoxRowsSmall);
  };
  // MX: the scale ring needs TMEM columns beside the two accumulators, so a
  // slot tile holds at most 224 slots (2 x 224 + 4 stages x 16 <= 512)
  p.max_tn = mx ? kMxMaxTileN : kMaxTileN;
  p.sfa = a.w_sf;
  p.sfb = a.b_sf;
  switch (a.mode) {
    case kModeFc1:  // A = w13 rows [E*2I, H] (gate and up accumulators); B gathered from x
      p.n_acc = 2;
      p.pair_feats = 0;
      p.m_total = a.I;
      p.k_tiles = a.H / kBK;
      p.a_rows_per_expert = 2 * a.I;
      p.a_second_off = a.I;
      p.f_rows = kTileM;
      p.f_tiles = a.I / kTileM;
      p.out_ld = a.I;
      p.act_ld = a.H;
      if (!make_map(&tmA, a.w, (uint64_t)a.H, E * 2 * a.I, kBK, kTileM)) return -1;
      tmB = tmA;  // unused: B rows are gathered with cp.async
      tmA2 = tmA;
      break;
    case kModeFc1Fp8:  // A = quantised w13 rows [E*2I, H] bytes; B gathered from quantised x
      // bytes addressed as pairs: a 64-element (16-bit) box row is 128 E4M3
      // values, the same 128-byte swizzled rows as bf16
      p.n_acc = 2;
      p.pair_feats = 0;
      p.m_total = a.I;
      p.k_tiles = a.H / (2 * kBK);
      p.a_rows_per_expert = 2 * a.I;
      p.a_second_off = a.I;
      p.f_rows = kTileM;
      p.f_tiles = a.I / kTileM;
      p.out_ld = a.I;
      p.act_ld = a.H / 2;
      if (!make_map(&tmA, a.w, (uint64_t)(a.H / 2), E * 2 * a.I, kBK, kTileM)) return -1;
      tmB = tmA;
      tmA2 = tmA;
      break;
    case kModeFc1Mx:  // as kModeFc1Fp8; the block scales travel with the operands
      p.n_acc = 2;
      p.pair_feats = 0;
      p.m_total = a.I;
      p.k_tiles = a.H / (2 * kBK);
      p.a_rows_per_expert = 2 * a.I;
      p.a_second_off = a.I;
      p.f_rows = kTileM;
      p.f_tiles = a.I / kTileM;
      p.out_ld = a.I;
      p.act_ld = a.H / 2;
      p.sfb_ld = a.H / 32;
      if (!a.w_sf || !a.b_sf) return -1;
      if (!make_map(&tmA, a.w, (uint64_t)(a.H / 2), E * 2 * a.I, kBK, kTileM)) return -1;
      tmB = tmA;
      tmA2 = tmA;
      break;
    case kModeFc2Mx:  // as kModeFc2Fp8; the h rows' scale bytes gathered by warps 10-13
      p.n_acc = 2;
      p.pair_feats = 1;
      p.m_total = a.H;
      p.k_tiles = a.I / (2 * kBK);
      p.a_rows_per_expert = a.H;
      p.a_second_off = kTileM;
      p.f_rows = 2 * kTileM;
      p.f_tiles = (a.H + 2 * kTileM - 1) / (2 * kTileM);
      p.out_ld = a.H;
      p.act_ld = a.I / 2;
      p.sfb_ld = a.I / 32;
      if (!a.w_sf || !a.b_sf) return -1;
      if (!make_map(&tmA, a.w, (uint64_t)(a.I / 2), E * a.H, kBK, kTileM)) return -1;
      if (!make_b(a.act, (uint64_t)(a.I / 2))) return -1;
      tmA2 = tmA;
      break;
    case kModeFc2:  // A = w2 rows [E*H, I], two 128-row feature tiles; B = h [S, I]
      p.n_acc = 2;
      p.pair_feats = 1;
      p.m_total = a.H;
      p.k_tiles = a.I / kBK;
      p.a_rows_per_expert = a.H;
      p.a_second_off = kTileM;
      p.f_rows = 2 * kTileM;
      p.f_tiles = (a.H + 2 * kTileM - 1) / (2 * kTileM);
      p.out_ld = a.H;
      p.act_ld = a.I;
      if (!make_map(&tmA, a.w, (uint64_t)a.I, E * a.H, kBK, kTileM)) return -1;
      if (!make_b(a.act, (uint64_t)a.I)) return -1;
      tmA2 = tmA;
      break;
    case kModeFc2Fp8:  // FC2 on E4M3 bytes: w2q rows [E*H, I], hq [S, I], addressed as pairs
      p.n_acc = 2;
      p.pair_feats = 1;
      p.m_total = a.H;
      p.k_tiles = a.I / (2 * kBK);
      p.a_rows_per_expert = a.H;
      p.a_second_off = kTileM;
      p.f_rows = 2 * kTileM;
      p.f_tiles = (a.H + 2 * kTileM - 1) / (2 * kTileM);
      p.out_ld = a.H;
      p.act_ld = a.I / 2;
      if (!make_map(&tmA, a.w, (uint64_t)(a.I / 2), E * a.H, kBK, kTileM)) return -1;
      if (!make_b(a.act, (uint64_t)(a.I / 2))) return -1;
      tmA2 = tmA;
      break;
    case kModeDgrad2:  // A[i, h] = w2[e][h][i] (MN-major, K = H); B gathered from dY [N, H]
      // two 128-feature accumulators share each gathered dY stage (the last
      // tile holds one when I is not a multiple of 256). One tile in TMEM, so
      // the SwiGLU-backward epilogue does not overlap the next tile's MMAs;
      // halving the gathered bytes per flop still measured faster (dropless
      // ffn_backward 7.02 -> 6.93 ms) than one accumulator with two tiles in
      // flight.
      p.n_acc = 2;
      p.pair_feats = 1;
      p.m_total = a.I;
      p.k_tiles = a.H / kBK;
      p.a_rows_per_expert = a.H;
      p.f_rows = 2 * kTileM;
      p.f_tiles = (a.I + 2 * kTileM - 1) / (2 * kTileM);
      p.out_ld = 2 * a.I;
      p.act_ld = a.H;
      if (!make_map_mn3d(&tmA, a.w, (uint64_t)a.I, E * a.H, kBK, 4)) return -1;
      if (!make_map_mn3d(&tmA2, a.w, (uint64_t)a.I, E * a.H, kBK, 2)) return -1;
      tmB = tmA;
      break;
    case kModeDgrad1:  // A[h, k] = w13[e][k][h] (MN-major, K = 2I); B = dPre [S, 2I]
      p.n_acc = 2;
      p.pair_feats = 1;
      p.m_total = a.H;
      p.k_tiles = 2 * a.I / kBK;
      p.a_rows_per_expert = 2 * a.I;
      p.f_rows = 2 * kTileM;
      p.f_tiles = (a.H + 2 * kTileM - 1) / (2 * kTileM);
      p.out_ld = a.H;
      p.act_ld = 2 * a.I;
      if (!make_map_mn3d(&tmA, a.w, (uint64_t)a.H, E * 2 * a.I, kBK, 4)) return -1;
      if (!make_map_mn3d(&tmA2, a.w, (uint64_t)a.H, E * 2 * a.I, kBK, 2)) return -1;
      if (!make_b(a.act, (uint64_t)(2 * a.I))) return -1;
      break;
    default:
      return -1;
  }
  p.E = a.E;
  const bool pair = pair_mode(a.mode, a.H, a.I);
  if (pair) {
    // a pair tile covers twice the features, each CTA f_cta of them; the B
    // rows of a slot tile are split between the CTAs, fetched in 32-row boxes
    p.f_cta = p.f_rows;
    p.f_rows = 2 * p.f_rows;
    p.f_tiles = (p.m_total + p.f_rows - 1) / p.f_rows;
    if (!gather_b &&
        !(make_map(&tmB, a.act, (uint64_t)p.act_ld, (uint64_t)S, kBK, kBBoxRowsPair) &&
          make_map(&tmB2, a.act, (uint64_t)p.act_ld, (uint64_t)S, kBK, kBBoxRowsPairSmall)))
      return -1;
  }
  // stage size for the largest slot tile any expert can have
  const int64_t rows_cap = a.max_rows < p.max_tn ? a.max_rows : p.max_tn;
  const int tile_cap = (int)((rows_cap + 15) / 16 * 16);
  const int b_rows_cap = pair ? tile_cap / 2 : tile_cap;  // B rows of a stage in one CTA
  const int64_t grid_bound =
      (int64_t)p.f_tiles * ((a.max_total + p.max_tn - 1) / p.max_tn + a.E) * (pair ? 2 : 1);
  p.b_off = (uint32_t)p.n_acc * kATileBytes;
  p.sf_off = p.b_off + (((uint32_t)b_rows_cap * 128u + 1023u) & ~1023u);
  p.stage_bytes = p.sf_off + (mx ? 2048u : 0u);  // MX: 2 A and 2 B scale atoms
  // the FP8 modes' epilogue keeps its B-row scales in shared memory, the FC2
  // dgrad its next pre-activations and two more output staging buffers (the
  // same region)
  const uint32_t xs_bytes = (a.mode == kModeFc1Fp8 || a.mode == kModeFc2Fp8) ? kXsBytes
                            : a.mode == kModeDgrad2 ? kPreBufBytes + kEpiWarps * 1024u
                                                    : 0u;
  p.stages = (int)((kSmemBudget - 1024u - kEpiStageBytes - kPsBytes - xs_bytes) / p.stage_bytes);
  if (p.stages > kMaxStages) p.stages = kMaxStages;
  p.sf_tmem = (uint32_t)(2 * p.max_tn);
  if (mx && p.stages > (int)((kTmemCols - p.sf_tmem) / 16)) p.stages = (int)((kTmemCols - p.sf_tmem) / 16);
  if (p.stages < 2) return -1;
  p.epi_off = (uint32_t)p.stages * p.stage_bytes;
  p.ps_off = p.epi_off + kEpiStageBytes;
  p.xs_off = p.ps_off + kPsBytes;
  p.acc_off = (uint32_t)p.max_tn;
  p.buf_stride = (uint32_t)(p.n_acc * p.max_tn);
  p.n_buf = 2 * p.buf_stride <= kTmemCols ? 2 : 1;
  const size_t dyn = (size_t)p.xs_off + xs_bytes + 1024;
  cudaError_t err = cudaSuccess;
  const int sms = device_sms(&err);
  if (sms <= 0) return -(int)(err != cudaSuccess ? err : cudaErrorUnknown);
  int grid = (int)(grid_bound < sms ? grid_bound : sms);
  if (pair) grid &= ~1;  // whole pairs
  if (grid <= 0) return -1;
  p.sched = a.sched;
  const bool gelu = a.activation == 1;
  // a mode's kernel, as CTA pairs or single CTAs
#define MOE_LAUNCH_GEMM(MODE, ACT)                                                                  \
  (pair ? launch_pdl_pairs(moe_gemm_kernel<MODE, ACT, 1>, dim3(grid), dim3(kThreads), dyn, s, tmA, \
                           tmB, tmA2, tmB2, p)                                                     \
        : launch_pdl(moe_gemm_kernel<MODE, ACT, 0>, dim3(grid), dim3(kThreads), dyn, s, tmA, tmB,  \
                     tmA2, tmB2, p))
#define MOE_LAUNCH_GEMM1(MODE, ACT)                                                                 \
  launch_pdl(moe_gemm_kernel<MODE, ACT, 0>, dim3(grid), dim3(kThreads), dyn, s, tmA, tmB, tmA2, \
             tmB2, p)
  switch (a.mode) {
    case kModeFc1:
      if (gelu) MOE_LAUNCH_GEMM(kModeFc1, 1); else MOE_LAUNCH_GEMM(kModeFc1, 0);
      break;
    case kModeFc2: MOE_LAUNCH_GEMM(kModeFc2, 0); break;
    case kModeDgrad2:
      if (gelu) MOE_LAUNCH_GEMM1(kModeDgrad2, 1); else MOE_LAUNCH_GEMM1(kModeDgrad2, 0);
      break;
    case kModeDgrad1: MOE_LAUNCH_GEMM1(kModeDgrad1, 0); break;
    case kModeFc1Fp8:
      if (gelu) MOE_LAUNCH_GEMM1(kModeFc1Fp8, 1); else MOE_LAUNCH_GEMM1(kModeFc1Fp8, 0);
      break;
    case kModeFc2Fp8: MOE_LAUNCH_GEMM1(kModeFc2Fp8, 0); break;
    case kModeFc1Mx:
      if (gelu) MOE_LAUNCH_GEMM1(kModeFc1Mx, 1); else MOE_LAUNCH_GEMM1(kModeFc1Mx, 0);
      break;
    case kModeFc2Mx: MOE_LAUNCH_GEMM1(kModeFc2Mx, 0); break;
    default: return -1;
  }
#undef MOE_LAUNCH_GEMM
#undef MOE_LAUNCH_GEMM1
  err = cudaGetLastError();
  if (err != cudaSuccess) return -(int)err;
  return 1;
}

}  // namespace moe
