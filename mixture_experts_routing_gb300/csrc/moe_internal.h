// Internal launch interface between the C ABI (moe_abi.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace moe {

constexpr int kMaxDevices = 64;

// One-time, per-device set-up (shared-memory opt-ins, SM counts): `fn(dev,
// &v)` runs for the current device under a lock until it succeeds with v > 0;
// later calls read v without locking. Safe when several host threads make
// their first call on a device at the same time.
struct DeviceOnce {
  std::mutex mu;
  std::atomic<int> value[kMaxDevices];
};

template <class Fn>
inline cudaError_t once_per_device(DeviceOnce& o, int* value, Fn fn) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int v = o.value[dev].load(std::memory_order_acquire);
  if (v <= 0) {
    std::lock_guard<std::mutex> lock(o.mu);
    v = o.value[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
      err = fn(dev, &v);
      if (err != cudaSuccess) return err;
      if (v <= 0) v = 1;
      o.value[dev].store(v, std::memory_order_release);
    }
  }
  if (value) *value = v;
  return cudaSuccess;
}

// Launch of a forward-path kernel with programmatic stream serialization: it
// may start (setup, then griddep_wait) while the previous kernel in the
// stream finishes, which hides the launch gap between the six kernels of a
// forward. Captured into CUDA graphs as programmatic edges.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same launch with the CTAs in clusters of two (CTA pairs).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_pairs(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

constexpr int kTokensPerChunk = 32;   // tokens per router CTA = one scan chunk
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 16;
constexpr int kMaxTokens = 24576;     // select kernel stages one expert's routes in smem

struct RouteWs {
  float* logits;          // [N,E]
  int32_t* chunk_counts;  // [C,E] routes of expert e in chunk c
  int32_t* chunk_lofs;    // [C,E] offset of expert e's routes in chunk c's sorted list
  int32_t* chunk_routes;  // [N*K] per chunk: route indices sorted by expert, token order kept
  uint32_t* chunk_keys;   // [N*K] the renormalised probability bits of those routes
};

constexpr int kMaxLadder = 16;

struct Ladder {  // dropless padding rungs: multiples num[j]/den of the expected rows
  int len, den;
  int num[kMaxLadder];
};

struct RouteArgs {
  int N, H, E, K, renorm, bm;   // N: the static token bound (buffers, grids)
  const int32_t* n_dev;         // live token count on the device, or null for N
  uint32_t* err;                // device error word (bounded waits)
  int cap_num, cap_den;         // capacity factor (the capacity follows the live count)
  int dropless;          // 1: keep every route, extents from the ladder
  Ladder ladder;
  int64_t s_max;         // slots the caller allocated (static bound)
  const uint16_t* x;
  const float* wr;
  const float* bias;
  int32_t* topk_ids;
  float* topk_p;
  uint8_t* keep;
  int32_t* expert_counts;
  int32_t* kept_counts;
  int32_t* sorted_slot_ids;
  int32_t* expert_ids;
  int32_t* block_start;
  int32_t* ntpp;
  int32_t* token_routes;
  int32_t* gemm_sched;
  float* slot_prob;      // [S] p' of each slot's route, 0 for padding
  RouteWs ws;
};

// Returns the number of kernels launched (>= 0) or a negative cudaError_t.
int launch_route(const RouteArgs& a, cudaStream_t s);

enum GemmMode {
  kModeFc1 = 0,     // FC1: B = rows of x gathered by slot, SwiGLU epilogue
  kModeFc2 = 1,     // FC2: B = h rows by slot (TMA), plain epilogue
  kModeDgrad2 = 2,  // dgrad of FC2: A = w2 read MN-major, B = rows of dY gathered by
                    // slot, SwiGLU-backward epilogue
  kModeDgrad1 = 3,  // dgrad of FC1: A = w13 read MN-major, B = dPre rows by slot (TMA)
  kModeFc1Fp8 = 4,  // FC1 in FP8 (E4M3): A = quantised w13 rows, B = rows of quantised x
                    // gathered by slot; epilogue applies the row and token scales
  kModeFc2Fp8 = 5,  // FC2 in FP8: A = quantised w2 rows, B = quantised h rows (TMA);
                    // epilogue applies the w2 row and h slot-row scales
  kModeFc1Mx = 6,   // FC1 on MX (block-scaled E4M3) operands: B rows of x gathered with
                    // their scale bytes; the tensor cores apply the block scales
  kModeFc2Mx = 7,   // FC2 on MX operands: B = h rows (TMA), their scale bytes gathered
};

struct GemmArgs {
  int mode;              // GemmMode
  int N, H, E, I, bm;
  int64_t max_rows;      // upper bound of kept routes per expert
  int64_t max_total;     // upper bound of kept routes over all experts
  int64_t s_max;         // rows of the slot-space buffers (h, o)
  const void* act;       // FC1: x [N,H]; FC2: h [S,I]; dgrad2: dY [N,H]; dgrad1: dPre [S,2I]
  const void* w;         // FC1, dgrad1: w13 [E,2I,H]; FC2, dgrad2: w2 [E,H,I]
  void* out;             // FC1: h [S,I]; FC2: o [S,H]; dgrad2: dPre [S,2I]; dgrad1: dXr [S,H]
  void* out2;            // FC1: pre-activations [S,2I] or null; dgrad2: p'*a [S,I]
  const void* aux;       // dgrad2: pre-activations [S,2I]
  const float* slot_prob;     // FC1 (prob_in_act), dgrad2: p' of each slot's route (0 padding)
  int activation;             // FC1, dgrad2: 0 SwiGLU, 1 GeGLU
  int prob_in_act;            // FC1: multiply the activation by the slot's p'
  const float* w_scale;       // FP8: scale of each weight row (FC1 [E*2I], FC2 [E*H])
  const float* x_scale;       // FP8: scale of each B row (FC1: token [N]; FC2: slot [S])
  float* part;                // dgrad2: dprob partials [S, I/32]
  const uint8_t* w_sf;        // MX: E8M0 scales of the weight rows in 512-byte atoms
  const uint8_t* b_sf;        // MX: E8M0 scales of the B rows, [rows, K/32]
  int64_t act_rows;      // rows of act (N when gathered, else S)
  const int32_t* sorted_slot_ids;
  const int32_t* kept_counts;
  const int32_t* block_start;
  int32_t* sched;        // [2]: next tile, finished CTAs (this GEMM's pair of gemm_sched)
  uint32_t* err;
};

int launch_gemm(const GemmArgs& a, cudaStream_t s);

struct WgradArgs {
  int dw13;              // 1: dW13 [E,2I,H] from dPre and x; 0: dW2 [E,H,I] from aw and dY
  int N, H, E, I, bm;
  int64_t s_max;
  const void* slot_mat;  // dW13: dPre [S,2I]; dW2: aw [S,I]
  const void* x;         // [N,H]
  const void* dy;        // [N,H]
  const int32_t* sorted_slot_ids;
  const int32_t* kept_counts;
  const int32_t* block_start;
  int32_t* sched;        // [2]
  float* out;
  uint32_t* err;
};

int launch_wgrad(const WgradArgs& a, cudaStream_t s);

// Router backward (route.cu, router_mma.cu): logits recomputed into dl,
// dl = d loss / d logits from dprob (fp32, plus its bf16 hi/lo split copy dls),
// then dW_r on the tensor cores (split over tokens, partials in part), dbias,
// and dx += dl . W_r^T on the tensor cores (W_r's split copy in wrs; bf16
// in/out).
struct RouterBwdArgs {
  int N, H, E, K, renorm;
  uint32_t* err;                // device error word (bounded waits)
  const float* logits;          // the forward's logits [N,E], or null to recompute them
  const uint16_t* x;
  const float* wr;
  const float* bias;
  const int32_t* topk_ids;
  const float* dprob;
  float* dl;        // [N,E] workspace
  uint16_t* dls;    // [N, router_split_cols(E)] workspace: bf16 hi | lo of dl
  uint16_t* wrs;    // [H, router_split_cols(E)] workspace: bf16 hi | lo of W_r
  float* part;      // [splits,H,E] workspace
  float* dwr;       // [H,E]
  float* dbias;     // [E] or null
  uint16_t* dx;     // [N,H] bf16, accumulated
};
int launch_router_backward(const RouterBwdArgs& a, cudaStream_t s);
// router_mma.cu: columns of a split copy (2 * E rounded up to 64), the token
// splits of dW_r (a function of the shape only), and the launches
int router_split_cols(int E);
int router_bwd_splits(int N, int H, int E);
int launch_router_split_w(const float* wr, int H, int E, uint16_t* wrs, cudaStream_t s);
int launch_router_dwr_mma(const uint16_t* x, const uint16_t* dls, int N, int H, int E,
                          float* part, uint32_t* err, cudaStream_t s);
int launch_router_dx_mma(const uint16_t* dls, const uint16_t* wrs, int N, int H, int E,
                         uint16_t* dx, uint32_t* err, cudaStream_t s);

// Backward helpers (combine.cu).
// dX[t] = sum_k dXr[token_routes[t,k]] (fp32, k order) and
// dprob[t,k] = sum_j part[token_routes[t,k], j] (j order; 0 for a dropped route).
int launch_combine_bwd(const uint16_t* dxr, const float* part, int n_part,
                       const int32_t* token_routes, int N, int H, int K, uint16_t* dx,
                       float* dprob, cudaStream_t s);

struct CombineArgs {
  int N, H, K;
  const int32_t* n_dev;  // live token count (null: N); rows past it are written as 0
  const uint16_t* o;
  const int32_t* token_routes;
  const float* topk_p;
  uint16_t* y;
};

int launch_combine(const CombineArgs& a, cudaStream_t s);

// Row-wise E4M3 quantisation of a bf16 [rows, cols] matrix (cols a multiple
// of 8, rows 16-byte aligned): codes q [rows, cols], scales [rows]. With
// rows_dev, rows at or past *rows_dev (read on the device) are left as they are.
int launch_quantize_rows_fp8(const uint16_t* m, int64_t rows, const int32_t* rows_dev, int cols,
                             uint8_t* q, float* scale, cudaStream_t s);

// MX (block-scaled) E4M3 quantisation of a bf16 [rows, cols] matrix along its
// rows (cols a multiple of 32; with atoms, rows and cols multiples of 128):
// codes q [rows, cols] and one E8M0 scale byte per 32 values, plain
// [rows, cols/32] or, with atoms, in the 512-byte atoms the MX GEMMs copy to
// tensor memory. With rows_dev, rows at or past *rows_dev are left as they are.
int launch_quantize_mx_fp8(const uint16_t* m, int64_t rows, const int32_t* rows_dev, int cols,
                           uint8_t* q, uint8_t* scale, int atoms, cudaStream_t s);

// The library's launch counter (moe_launch_count): read, and adjusted by the
// graph ladder (captured launches are not executions; a replay is).
uint64_t launch_counter();
void add_launches(int64_t n);

// out[e*out_es + out_off + c*R + r] = in[e*in_es + r*C + c], bf16.
int launch_transpose(const uint16_t* in, uint16_t* out, int E, int R, int C, int64_t in_es,
                     int64_t out_es, int64_t out_off, cudaStream_t s);

}  // namespace moe
