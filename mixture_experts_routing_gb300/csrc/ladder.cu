// Graph bucket ladder: captured CUDA graphs of the layer forward at a ladder
// of token-count buckets, for batches whose size changes from call to call
// ("[4/5] feat: capture the FFN experts at bucketed padded shapes", What this
// adds). A batch of n tokens replays the first bucket >= n; it runs eagerly
// when n is above the top bucket or that bucket exceeds max_pad_ratio * n.
// Capture goes from the top bucket down, after one warm-up call at the top
// size.
//
// A bucket's graph is the three forward calls (route_align, ffn_forward,
// combine) captured with n_tokens = the bucket and n_valid pointing at one
// device int32: every kernel reads the live count when it runs, so the replay
// of a bucket computes exactly what an eager call on the first n tokens
// computes (capacity, ladder extents and layout follow n). Before a replay the
// live count is written by a one-thread kernel on the same stream.
#include <cuda_runtime.h>

#include <new>
#include <vector>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

__global__ void set_count_kernel(int32_t* p, int32_t v) { *p = v; }

int forward_calls(const moe_config_t* cfg, const moe_layer_buffers_t* b, cudaStream_t s) {
  int rc = moe_route_align(cfg, b->x, b->w_router, b->bias, &b->routes, b->route_workspace,
                           b->route_workspace_bytes, s);
  if (rc != MOE_OK) return rc;
  rc = moe_ffn_forward(cfg, &b->routes, b->x, b->w13, b->w2, b->h, b->o, s);
  if (rc != MOE_OK) return rc;
  return moe_combine(cfg, &b->routes, b->o, b->y, s);
}

}  // namespace

struct moe_ladder {
  moe_config_t top;
  std::vector<int32_t> ladder_num;  // the dropless rungs the configs point at
  std::vector<int32_t> buckets;
  float max_pad_ratio = 0.0f;
  moe_layer_buffers_t bufs{};
  std::vector<cudaGraphExec_t> execs;  // one per bucket, same order as buckets
  std::vector<int64_t> kernels;        // kernels in each bucket's graph
};

extern "C" {

int moe_ladder_pick(const int32_t* buckets, int n_buckets, int32_t n, float max_pad_ratio) {
  if (!buckets || n_buckets <= 0 || n < 0) return -1;
  for (int b = 0; b < n_buckets; ++b) {
    if (buckets[b] < n) continue;
    // a replay costs the bucket's full size, so a batch far below it goes eager
    if (max_pad_ratio > 0.0f && n > 0 && (double)buckets[b] > (double)max_pad_ratio * n)
      return -1;
    return b;
  }
  return -1;
}

int moe_ladder_create(const moe_config_t* top, const int32_t* buckets, int n_buckets,
                      float max_pad_ratio, const moe_layer_buffers_t* bufs, moe_ladder_t** out) {
  if (!top || !buckets || n_buckets <= 0 || !bufs || !out || !bufs->n_valid || top->n_valid)
    return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  for (int b = 0; b < n_buckets; ++b)
    if (buckets[b] <= 0 || (b > 0 && buckets[b] <= buckets[b - 1])) return MOE_ERR_INVALID_ARG;
  if (buckets[n_buckets - 1] != top->n_tokens) return MOE_ERR_INVALID_ARG;
  if (moe_max_slots(top) < 0) return MOE_ERR_INVALID_ARG;
  moe_ladder* L = new (std::nothrow) moe_ladder();
  if (!L) return MOE_ERR_INVALID_ARG;
  L->top = *top;
  if (top->ladder_len > 0 && top->ladder_num) {
    L->ladder_num.assign(top->ladder_num, top->ladder_num + top->ladder_len);
    L->top.ladder_num = L->ladder_num.data();
  }
  L->buckets.assign(buckets, buckets + n_buckets);
  L->max_pad_ratio = max_pad_ratio;
  L->bufs = *bufs;
  cudaStream_t cs = nullptr;
  int rc = MOE_OK;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) rc = MOE_ERR_CUDA;
  // one warm-up call at the top size first: every lazily set kernel attribute and
  // looked-up symbol is in place before any capture
  if (rc == MOE_OK) rc = forward_calls(&L->top, &L->bufs, cs);
  if (rc == MOE_OK && cudaStreamSynchronize(cs) != cudaSuccess) rc = MOE_ERR_CUDA;
  L->execs.assign(n_buckets, nullptr);
  L->kernels.assign(n_buckets, 0);
  for (int b = n_buckets - 1; b >= 0 && rc == MOE_OK; --b) {  // largest first
    moe_config_t cfg = L->top;
    cfg.n_tokens = L->buckets[b];
    cfg.n_valid = L->bufs.n_valid;
    cudaGraph_t g = nullptr;
    const uint64_t before = moe::launch_counter();
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      rc = MOE_ERR_CUDA;
      break;
    }
    const int crc = forward_calls(&cfg, &L->bufs, cs);
    const cudaError_t ce = cudaStreamEndCapture(cs, &g);
    // captured launches are not executions: count them when a replay runs
    L->kernels[b] = (int64_t)(moe::launch_counter() - before);
    moe::add_launches(-L->kernels[b]);
    if (crc != MOE_OK || ce != cudaSuccess) {
      rc = crc != MOE_OK ? crc : MOE_ERR_CUDA;
      if (g) cudaGraphDestroy(g);
      break;
    }
    const cudaError_t ie = cudaGraphInstantiate(&L->execs[b], g, 0);
    cudaGraphDestroy(g);
    if (ie != cudaSuccess) rc = MOE_ERR_CUDA;
  }
  if (cs) cudaStreamDestroy(cs);
  if (rc != MOE_OK) {
    cudaGetLastError();
    moe_ladder_destroy(L);
    return rc;
  }
  *out = L;
  return MOE_OK;
}

int moe_ladder_forward(moe_ladder_t* L, int32_t n, cudaStream_t stream, int* bucket) {
  if (!L || n < 0 || n > L->top.n_tokens) return MOE_ERR_INVALID_ARG;
  const int b = moe_ladder_pick(L->buckets.data(), (int)L->buckets.size(), n, L->max_pad_ratio);
  if (bucket) *bucket = b;
  if (b < 0) {  // eager on exactly n tokens
    moe_config_t cfg = L->top;
    cfg.n_tokens = n;
    cfg.n_valid = nullptr;
    return forward_calls(&cfg, &L->bufs, stream);
  }
  set_count_kernel<<<1, 1, 0, stream>>>(L->bufs.n_valid, n);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaGraphLaunch(L->execs[b], stream) != cudaSuccess) return MOE_ERR_CUDA;
  moe::add_launches(1 + L->kernels[b]);
  return MOE_OK;
}

int moe_ladder_destroy(moe_ladder_t* L) {
  if (!L) return MOE_OK;
  for (cudaGraphExec_t e : L->execs)
    if (e) cudaGraphExecDestroy(e);
  delete L;
  return MOE_OK;
}

}  // extern "C"
