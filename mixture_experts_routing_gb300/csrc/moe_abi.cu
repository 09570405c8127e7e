// C ABI of the library (declared in include/moe.h): argument checks, workspace
// carving, and the launch sequence of each entry point. No allocation, no
// host synchronisation, no device-to-host reads (except moe_device_error, which
// is documented as a synchronising diagnostic).
#include <atomic>
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

std::atomic<uint64_t> g_launches{0};

// Device error word: kernels OR flags into it instead of trapping.
__device__ uint32_t g_moe_error_word;

uint32_t* error_word_ptr() {
  static std::mutex mu;
  static uint32_t* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t roundup(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// Fields valid and shape inside what the kernels implement.
int check_cfg(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->n_tokens < 0 || c->hidden <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->inter <= 0 ||
      c->cap_den <= 0 || c->cap_num < 0 || (c->renorm != 0 && c->renorm != 1) ||
      c->top_k > c->n_experts)
    return MOE_ERR_INVALID_ARG;
  if (c->block_m != 16 && c->block_m != 32 && c->block_m != 64 && c->block_m != 128)
    return MOE_ERR_INVALID_ARG;
  if ((c->activation != MOE_ACT_SWIGLU && c->activation != MOE_ACT_GEGLU) ||
      (c->prob_in_act != 0 && c->prob_in_act != 1))
    return MOE_ERR_INVALID_ARG;
  if (c->cap_num == 0) {  // dropless: the ladder must be well formed
    if (c->ladder_len < 0 || c->ladder_len > moe::kMaxLadder) return MOE_ERR_INVALID_ARG;
    if (c->ladder_len > 0) {
      if (!c->ladder_num || c->ladder_den <= 0) return MOE_ERR_INVALID_ARG;
      for (int j = 0; j < c->ladder_len; ++j)
        if (c->ladder_num[j] <= 0 || (j > 0 && c->ladder_num[j] <= c->ladder_num[j - 1]))
          return MOE_ERR_INVALID_ARG;
    }
  }
  if (c->hidden % 128 != 0 || c->inter % 128 != 0 || c->n_experts > moe::kMaxExperts ||
      c->top_k > moe::kMaxTopK || c->n_tokens > moe::kMaxTokens)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  int64_t S = 0;
  if (c->cap_num == 0) {
    const int64_t R = (int64_t)c->n_tokens * c->top_k;
    int64_t top = 0;
    if (c->ladder_len > 0) {
      const int64_t num = (int64_t)c->ladder_num[c->ladder_len - 1] * R;
      const int64_t den = (int64_t)c->ladder_den * c->n_experts;
      top = roundup((num + den - 1) / den, c->block_m);
    }
    S = roundup(R + (int64_t)c->n_experts * (top + c->block_m), c->block_m);
  } else {
    const int64_t cap =
        ((int64_t)c->n_tokens * c->top_k * c->cap_num + (int64_t)c->n_experts * c->cap_den - 1) /
        ((int64_t)c->n_experts * c->cap_den);
    S = (int64_t)c->n_experts * roundup(cap, c->block_m);
  }
  if (S > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

bool dropless_of(const moe_config_t* c) { return c->cap_num == 0; }

int64_t cap_of(const moe_config_t* c) {
  if (dropless_of(c)) return c->n_tokens;
  return ((int64_t)c->n_tokens * c->top_k * c->cap_num + (int64_t)c->n_experts * c->cap_den - 1) /
         ((int64_t)c->n_experts * c->cap_den);
}

int64_t cpad_of(const moe_config_t* c) { return roundup(cap_of(c), c->block_m); }

// Slot rows of the route list and of the slot-space buffers.
int64_t slots_of(const moe_config_t* c) {
  if (!dropless_of(c)) return (int64_t)c->n_experts * cpad_of(c);
  const int64_t R = (int64_t)c->n_tokens * c->top_k;
  int64_t top = 0;
  if (c->ladder_len > 0) {
    const int64_t num = (int64_t)c->ladder_num[c->ladder_len - 1] * R;
    const int64_t den = (int64_t)c->ladder_den * c->n_experts;
    top = roundup((num + den - 1) / den, c->block_m);
  }
  return roundup(R + (int64_t)c->n_experts * (top + c->block_m), c->block_m);
}

struct WsLayout {
  size_t logits, chunk_counts, chunk_lofs, chunk_routes, chunk_keys, total;
};

WsLayout ws_layout(const moe_config_t* c) {
  WsLayout w{};
  const int64_t N = c->n_tokens, E = c->n_experts, K = c->top_k;
  const int64_t C = (N + moe::kTokensPerChunk - 1) / moe::kTokensPerChunk;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  w.logits = take((size_t)(N * E) * 4);
  w.chunk_counts = take((size_t)(C * E) * 4);
  w.chunk_lofs = take((size_t)(C * E) * 4);
  w.chunk_routes = take((size_t)(N * K) * 4);
  w.chunk_keys = take((size_t)(N * K) * 4);
  w.total = off;
  return w;
}

// Backward scratch: the backward GEMMs' tile counters, the
// dprob partials, dPre = [dg | du], aw = p' a and the per-slot input gradient.
struct BwdLayout {
  size_t sched, part, dpre, aw, dxr, total;
};

BwdLayout bwd_layout(const moe_config_t* c) {
  BwdLayout w{};
  const int64_t S = c->n_tokens > 0 ? slots_of(c) : 0;
  const int64_t H = c->hidden, I = c->inter;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  w.sched = take(8 * 4);
  w.part = take((size_t)(S * (I / 32)) * 4);
  w.dpre = take((size_t)(S * 2 * I) * 2);
  w.aw = take((size_t)(S * I) * 2);
  w.dxr = take((size_t)(S * H) * 2);
  w.total = off;
  return w;
}

bool routes_complete(const moe_routes_t* r) {
  return r && r->topk_ids && r->topk_p && r->keep && r->expert_counts && r->kept_counts &&
         r->sorted_slot_ids && r->expert_ids && r->block_start && r->num_tokens_post_padded &&
         r->token_routes && r->gemm_sched && r->slot_prob;
}

int finish(int launched) {
  if (launched < 0) return MOE_ERR_CUDA;
  g_launches.fetch_add((uint64_t)launched, std::memory_order_relaxed);
  return MOE_OK;
}

}  // namespace

namespace moe {
uint64_t launch_counter() { return g_launches.load(std::memory_order_relaxed); }
void add_launches(int64_t n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace moe

extern "C" {

int64_t moe_capacity(const moe_config_t* cfg) {
  const int rc = check_cfg(cfg);
  return rc != MOE_OK ? rc : cap_of(cfg);
}

int64_t moe_max_slots(const moe_config_t* cfg) {
  const int rc = check_cfg(cfg);
  return rc != MOE_OK ? rc : slots_of(cfg);
}

int64_t moe_max_blocks(const moe_config_t* cfg) {
  const int rc = check_cfg(cfg);
  return rc != MOE_OK ? rc : slots_of(cfg) / cfg->block_m;
}

int64_t moe_route_workspace_bytes(const moe_config_t* cfg) {
  const int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  return (int64_t)ws_layout(cfg).total;
}

int moe_route_align(const moe_config_t* cfg, const void* x, const float* w_router,
                    const float* bias, const moe_routes_t* out, void* workspace, size_t ws_bytes,
                    cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!routes_complete(out)) return MOE_ERR_INVALID_ARG;
  if (cfg->n_tokens > 0 && (!x || !w_router || !aligned16(x))) return MOE_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(cfg);
  if (!workspace || ws_bytes < w.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  moe::RouteArgs a{};
  a.err = error_word_ptr();
  if (!a.err) return MOE_ERR_CUDA;
  a.N = cfg->n_tokens;
  a.H = cfg->hidden;
  a.E = cfg->n_experts;
  a.K = cfg->top_k;
  a.renorm = cfg->renorm;
  a.bm = cfg->block_m;
  a.n_dev = cfg->n_valid;
  a.cap_num = cfg->cap_num;
  a.cap_den = cfg->cap_den;
  a.dropless = dropless_of(cfg);
  a.ladder.len = a.dropless ? cfg->ladder_len : 0;
  a.ladder.den = cfg->ladder_den > 0 ? cfg->ladder_den : 1;
  for (int j = 0; j < a.ladder.len; ++j) a.ladder.num[j] = cfg->ladder_num[j];
  a.s_max = slots_of(cfg);
  a.x = static_cast<const uint16_t*>(x);
  a.wr = w_router;
  a.bias = bias;
  a.topk_ids = out->topk_ids;
  a.topk_p = out->topk_p;
  a.keep = out->keep;
  a.expert_counts = out->expert_counts;
  a.kept_counts = out->kept_counts;
  a.sorted_slot_ids = out->sorted_slot_ids;
  a.expert_ids = out->expert_ids;
  a.block_start = out->block_start;
  a.ntpp = out->num_tokens_post_padded;
  a.token_routes = out->token_routes;
  a.gemm_sched = out->gemm_sched;
  a.slot_prob = out->slot_prob;
  a.ws.logits = reinterpret_cast<float*>(ws + w.logits);
  a.ws.chunk_counts = reinterpret_cast<int32_t*>(ws + w.chunk_counts);
  a.ws.chunk_lofs = reinterpret_cast<int32_t*>(ws + w.chunk_lofs);
  a.ws.chunk_routes = reinterpret_cast<int32_t*>(ws + w.chunk_routes);
  a.ws.chunk_keys = reinterpret_cast<uint32_t*>(ws + w.chunk_keys);
  return finish(moe::launch_route(a, stream));
}

// Shape fields and routing pointers common to every expert-GEMM launch.
static void gemm_base(const moe_config_t* cfg, const moe_routes_t* routes, uint32_t* err,
                      moe::GemmArgs& a) {
  a.N = cfg->n_tokens;
  a.H = cfg->hidden;
  a.E = cfg->n_experts;
  a.I = cfg->inter;
  a.bm = cfg->block_m;
  a.max_rows = dropless_of(cfg) ? cfg->n_tokens : cap_of(cfg);
  if (a.max_rows > cfg->n_tokens) a.max_rows = cfg->n_tokens;
  a.max_total = (int64_t)cfg->n_tokens * cfg->top_k;
  a.s_max = slots_of(cfg);
  a.sorted_slot_ids = routes->sorted_slot_ids;
  a.kept_counts = routes->kept_counts;
  a.block_start = routes->block_start;
  a.err = err;
}

static bool gemm_routes_ok(const moe_routes_t* routes) {
  return routes && routes->sorted_slot_ids && routes->kept_counts && routes->block_start &&
         routes->gemm_sched && routes->slot_prob;
}

// One forward expert GEMM: mode kModeFc1/kModeFc2, or their FP8 forms with
// the weight-row and activation-row scales.
static int fc_forward(const moe_config_t* cfg, const moe_routes_t* routes, int mode,
                      const void* act, const void* w, void* out, void* preact,
                      const float* w_scale, const float* x_scale, cudaStream_t stream,
                      const void* w_sf = nullptr, const void* b_sf = nullptr) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!gemm_routes_ok(routes)) return MOE_ERR_INVALID_ARG;
  const bool fp8 = mode == moe::kModeFc1Fp8 || mode == moe::kModeFc2Fp8;
  const bool mx = mode == moe::kModeFc1Mx || mode == moe::kModeFc2Mx;
  const bool fc1 = mode == moe::kModeFc1 || mode == moe::kModeFc1Fp8 || mode == moe::kModeFc1Mx;
  if (fp8 && (!w_scale || !x_scale)) return MOE_ERR_INVALID_ARG;
  if (mx && (!w_sf || !b_sf || !aligned16(w_sf) || !aligned16(b_sf))) return MOE_ERR_INVALID_ARG;
  if (cfg->n_tokens == 0) return MOE_OK;
  if (!act || !w || !out || !aligned16(act) || !aligned16(w) || !aligned16(out) ||
      !aligned16(preact))
    return MOE_ERR_INVALID_ARG;
  uint32_t* err = error_word_ptr();
  if (!err) return MOE_ERR_CUDA;
  moe::GemmArgs a{};
  gemm_base(cfg, routes, err, a);
  a.mode = mode;
  a.act = act;
  a.w = w;
  a.out = out;
  a.out2 = fc1 ? preact : nullptr;
  a.activation = cfg->activation;
  a.prob_in_act = fc1 ? cfg->prob_in_act : 0;
  a.slot_prob = routes->slot_prob;
  a.w_scale = w_scale;
  a.x_scale = x_scale;
  a.w_sf = static_cast<const uint8_t*>(w_sf);
  a.b_sf = static_cast<const uint8_t*>(b_sf);
  a.act_rows = fc1 ? cfg->n_tokens : a.s_max;
  a.sched = routes->gemm_sched + (fc1 ? 0 : 2);
  return finish(moe::launch_gemm(a, stream));
}

int moe_fc1_forward(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                    const void* w13, void* h, cudaStream_t stream) {
  return fc_forward(cfg, routes, moe::kModeFc1, x, w13, h, nullptr, nullptr, nullptr, stream);
}

int moe_fc2_forward(const moe_config_t* cfg, const moe_routes_t* routes, const void* h,
                    const void* w2, void* o, cudaStream_t stream) {
  return fc_forward(cfg, routes, moe::kModeFc2, h, w2, o, nullptr, nullptr, nullptr, stream);
}

int moe_quantize_rows_fp8(const void* m, int64_t rows, const int32_t* rows_dev, int cols, void* q,
                          float* scale, cudaStream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 8 != 0 || rows > (int64_t)INT32_MAX)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!m || !q || !scale || !aligned16(m) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return finish(moe::launch_quantize_rows_fp8(static_cast<const uint16_t*>(m), rows, rows_dev, cols,
                                              static_cast<uint8_t*>(q), scale, stream));
}

int moe_fc1_forward_fp8(const moe_config_t* cfg, const moe_routes_t* routes, const void* xq,
                        const float* x_scale, const void* w13q, const float* w13_scale, void* h,
                        cudaStream_t stream) {
  return fc_forward(cfg, routes, moe::kModeFc1Fp8, xq, w13q, h, nullptr, w13_scale, x_scale,
                    stream);
}

int moe_fc2_forward_fp8(const moe_config_t* cfg, const moe_routes_t* routes, const void* hq,
                        const float* h_scale, const void* w2q, const float* w2_scale, void* o,
                        cudaStream_t stream) {
  return fc_forward(cfg, routes, moe::kModeFc2Fp8, hq, w2q, o, nullptr, w2_scale, h_scale, stream);
}

int moe_ffn_forward_fp8(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                        const void* w13q, const float* w13_scale, const void* w2q,
                        const float* w2_scale, void* xq, float* x_scale, void* h, void* hq,
                        float* h_scale, void* o, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!gemm_routes_ok(routes) || !routes->num_tokens_post_padded) return MOE_ERR_INVALID_ARG;
  if (cfg->n_tokens == 0) return MOE_OK;
  if (!x || !xq || !x_scale || !h || !hq || !h_scale || !aligned16(x) || !aligned16(xq) ||
      !aligned16(h) || !aligned16(hq))
    return MOE_ERR_INVALID_ARG;
  // x rows past a device-side live count are quantised too: FC1 gathers only
  // live rows, so they are never read
  rc = finish(moe::launch_quantize_rows_fp8(static_cast<const uint16_t*>(x), cfg->n_tokens, nullptr,
                                            cfg->hidden, static_cast<uint8_t*>(xq), x_scale,
                                            stream));
  if (rc != MOE_OK) return rc;
  rc = moe_fc1_forward_fp8(cfg, routes, xq, x_scale, w13q, w13_scale, h, stream);
  if (rc != MOE_OK) return rc;
  // only the slots below the padded extent hold routes
  rc = finish(moe::launch_quantize_rows_fp8(static_cast<const uint16_t*>(h), slots_of(cfg),
                                            routes->num_tokens_post_padded, cfg->inter,
                                            static_cast<uint8_t*>(hq), h_scale, stream));
  if (rc != MOE_OK) return rc;
  return moe_fc2_forward_fp8(cfg, routes, hq, h_scale, w2q, w2_scale, o, stream);
}

int moe_quantize_mx_fp8(const void* m, int64_t rows, const int32_t* rows_dev, int cols, void* q,
                        void* scale, cudaStream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 32 != 0 || rows > (int64_t)INT32_MAX)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!m || !q || !scale || !aligned16(m) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return finish(moe::launch_quantize_mx_fp8(static_cast<const uint16_t*>(m), rows, rows_dev, cols,
                                            static_cast<uint8_t*>(q),
                                            static_cast<uint8_t*>(scale), 0, stream));
}

int moe_quantize_mx_fp8_weights(const void* m, int64_t rows, int cols, void* q, void* scale_atoms,
                                cudaStream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 128 != 0 || rows % 128 != 0 || rows > (int64_t)INT32_MAX)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!m || !q || !scale_atoms || !aligned16(m) || !aligned16(q) || !aligned16(scale_atoms))
    return MOE_ERR_INVALID_ARG;
  return finish(moe::launch_quantize_mx_fp8(static_cast<const uint16_t*>(m), rows, nullptr, cols,
                                            static_cast<uint8_t*>(q),
                                            static_cast<uint8_t*>(scale_atoms), 1, stream));
}

int moe_fc1_forward_mx(const moe_config_t* cfg, const moe_routes_t* routes, const void* xq,
                       const void* x_sf, const void* w13q, const void* w13_sf, void* h,
                       cudaStream_t stream) {
  return fc_forward(cfg, routes, moe::kModeFc1Mx, xq, w13q, h, nullptr, nullptr, nullptr, stream,
                    w13_sf, x_sf);
}

int moe_fc2_forward_mx(const moe_config_t* cfg, const moe_routes_t* routes, const void* hq,
                       const void* h_sf, const void* w2q, const void* w2_sf, void* o,
                       cudaStream_t stream) {
  return fc_forward(cfg, routes, moe::kModeFc2Mx, hq, w2q, o, nullptr, nullptr, nullptr, stream,
                    w2_sf, h_sf);
}

int moe_ffn_forward_mx(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                       const void* w13q, const void* w13_sf, const void* w2q, const void* w2_sf,
                       void* xq, void* x_sf, void* h, void* hq, void* h_sf, void* o,
                       cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!gemm_routes_ok(routes) || !routes->num_tokens_post_padded) return MOE_ERR_INVALID_ARG;
  if (cfg->n_tokens == 0) return MOE_OK;
  if (!x || !xq || !x_sf || !h || !hq || !h_sf || !aligned16(x) || !aligned16(xq) ||
      !aligned16(x_sf) || !aligned16(h) || !aligned16(hq) || !aligned16(h_sf))
    return MOE_ERR_INVALID_ARG;
  rc = finish(moe::launch_quantize_mx_fp8(static_cast<const uint16_t*>(x), cfg->n_tokens, nullptr,
                                          cfg->hidden, static_cast<uint8_t*>(xq),
                                          static_cast<uint8_t*>(x_sf), 0, stream));
  if (rc != MOE_OK) return rc;
  rc = moe_fc1_forward_mx(cfg, routes, xq, x_sf, w13q, w13_sf, h, stream);
  if (rc != MOE_OK) return rc;
  // only the slots below the padded extent hold routes
  rc = finish(moe::launch_quantize_mx_fp8(static_cast<const uint16_t*>(h), slots_of(cfg),
                                          routes->num_tokens_post_padded, cfg->inter,
                                          static_cast<uint8_t*>(hq), static_cast<uint8_t*>(h_sf), 0,
                                          stream));
  if (rc != MOE_OK) return rc;
  return moe_fc2_forward_mx(cfg, routes, hq, h_sf, w2q, w2_sf, o, stream);
}

int moe_ffn_forward(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                    const void* w13, const void* w2, void* h, void* o, cudaStream_t stream) {
  const int rc = moe_fc1_forward(cfg, routes, x, w13, h, stream);
  if (rc != MOE_OK) return rc;
  return moe_fc2_forward(cfg, routes, h, w2, o, stream);
}

int moe_ffn_forward_train(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                          const void* w13, const void* w2, void* h, void* o, void* preact,
                          cudaStream_t stream) {
  if (cfg && cfg->n_tokens > 0 && !preact) return MOE_ERR_INVALID_ARG;
  const int rc =
      fc_forward(cfg, routes, moe::kModeFc1, x, w13, h, preact, nullptr, nullptr, stream);
  if (rc != MOE_OK) return rc;
  return moe_fc2_forward(cfg, routes, h, w2, o, stream);
}

int moe_combine(const moe_config_t* cfg, const moe_routes_t* routes, const void* o, void* y,
                cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!routes || !routes->token_routes || !routes->topk_p) return MOE_ERR_INVALID_ARG;
  if (cfg->n_tokens == 0) return MOE_OK;
  if (!o || !y || !aligned16(o) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  moe::CombineArgs a{};
  a.N = cfg->n_tokens;
  a.H = cfg->hidden;
  a.K = cfg->top_k;
  a.o = static_cast<const uint16_t*>(o);
  a.token_routes = routes->token_routes;
  a.topk_p = cfg->prob_in_act ? nullptr : routes->topk_p;  // unit weights: p' is in h
  a.n_dev = cfg->n_valid;
  a.y = static_cast<uint16_t*>(y);
  return finish(moe::launch_combine(a, stream));
}

int moe_pack_w13(const moe_config_t* cfg, const void* w_gate, const void* w_up, void* w13,
                 cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!w_gate || !w_up || !w13) return MOE_ERR_INVALID_ARG;
  const int E = cfg->n_experts, H = cfg->hidden, I = cfg->inter;
  const int64_t in_es = (int64_t)H * I, out_es = 2 * (int64_t)H * I;
  int l1 = moe::launch_transpose(static_cast<const uint16_t*>(w_gate), static_cast<uint16_t*>(w13),
                                 E, H, I, in_es, out_es, 0, stream);
  if (l1 < 0) return MOE_ERR_CUDA;
  int l2 = moe::launch_transpose(static_cast<const uint16_t*>(w_up), static_cast<uint16_t*>(w13), E,
                                 H, I, in_es, out_es, (int64_t)I * H, stream);
  if (l2 < 0) return MOE_ERR_CUDA;
  return finish(l1 + l2);
}

int moe_pack_w2(const moe_config_t* cfg, const void* w_down, void* w2, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (!w_down || !w2) return MOE_ERR_INVALID_ARG;
  const int E = cfg->n_experts, H = cfg->hidden, I = cfg->inter;
  return finish(moe::launch_transpose(static_cast<const uint16_t*>(w_down), static_cast<uint16_t*>(w2),
                                      E, I, H, (int64_t)I * H, (int64_t)I * H, 0, stream));
}

int64_t moe_backward_workspace_bytes(const moe_config_t* cfg) {
  const int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  return (int64_t)bwd_layout(cfg).total;
}

int moe_ffn_backward(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                     const void* w13, const void* w2, const void* preact, const void* dy,
                     void* dx, float* dw13, float* dw2, float* dprob, void* workspace,
                     size_t ws_bytes, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (cfg->n_valid) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!routes_complete(routes)) return MOE_ERR_INVALID_ARG;
  if (!dw13 || !dw2 || !aligned16(dw13) || !aligned16(dw2)) return MOE_ERR_INVALID_ARG;
  const BwdLayout L = bwd_layout(cfg);
  if (!workspace || ws_bytes < L.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  if (cfg->n_tokens > 0 &&
      (!x || !w13 || !w2 || !preact || !dy || !dx || !dprob || !aligned16(x) ||
       !aligned16(w13) || !aligned16(w2) || !aligned16(preact) || !aligned16(dy) ||
       !aligned16(dx)))
    return MOE_ERR_INVALID_ARG;
  uint32_t* err = error_word_ptr();
  if (!err) return MOE_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* sched = reinterpret_cast<int32_t*>(ws + L.sched);
  float* part = reinterpret_cast<float*>(ws + L.part);
  void* dpre = ws + L.dpre;
  void* aw = ws + L.aw;
  void* dxr = ws + L.dxr;
  const int N = cfg->n_tokens, H = cfg->hidden, E = cfg->n_experts, I = cfg->inter,
            K = cfg->top_k;
  const int64_t S = slots_of(cfg);
  int launched = 0;
  auto add = [&](int l) {
    if (l < 0) return false;
    launched += l;
    return true;
  };
  // 1. the backward GEMMs' tile counters start at zero
  if (cudaMemsetAsync(sched, 0, 8 * sizeof(int32_t), stream) != cudaSuccess) return finish(-1);
  if (N > 0) {
    // 2. FC2 dgrad with the SwiGLU backward: dPre, aw = p' a, dprob partials
    moe::GemmArgs g{};
    gemm_base(cfg, routes, err, g);
    g.mode = moe::kModeDgrad2;
    g.act = dy;
    g.w = w2;
    g.out = dpre;
    g.out2 = aw;
    g.aux = preact;
    g.slot_prob = routes->slot_prob;
    g.activation = cfg->activation;
    g.part = part;
    g.act_rows = N;
    g.sched = sched + 0;
    if (!add(moe::launch_gemm(g, stream))) return finish(-1);
    // 3. FC1 dgrad: dXr[s] = dg W_gate^T + du W_up^T
    moe::GemmArgs d{};
    gemm_base(cfg, routes, err, d);
    d.mode = moe::kModeDgrad1;
    d.act = dpre;
    d.w = w13;
    d.out = dxr;
    d.act_rows = S;
    d.sched = sched + 2;
    if (!add(moe::launch_gemm(d, stream))) return finish(-1);
    // 4. per-token reduction: dX (unit weights) and dprob
    if (!add(moe::launch_combine_bwd(static_cast<const uint16_t*>(dxr), part, I / 32,
                                     routes->token_routes, N, H, K, static_cast<uint16_t*>(dx),
                                     dprob, stream)))
      return finish(-1);
  }
  // 5. weight gradients (zero for an expert without kept slots, and for N = 0)
  moe::WgradArgs wg{};
  wg.N = N;
  wg.H = H;
  wg.E = E;
  wg.I = I;
  wg.bm = cfg->block_m;
  wg.s_max = S > 0 ? S : 1;
  wg.x = x;
  wg.dy = dy;
  wg.sorted_slot_ids = routes->sorted_slot_ids;
  wg.kept_counts = routes->kept_counts;
  wg.block_start = routes->block_start;
  wg.err = err;
  if (N > 0) {
    wg.dw13 = 0;
    wg.slot_mat = aw;
    wg.sched = sched + 4;
    wg.out = dw2;
    if (!add(moe::launch_wgrad(wg, stream))) return finish(-1);
    wg.dw13 = 1;
    wg.slot_mat = dpre;
    wg.sched = sched + 6;
    wg.out = dw13;
    if (!add(moe::launch_wgrad(wg, stream))) return finish(-1);
  } else {
    const size_t n13 = (size_t)E * 2 * I * H * 4, n2 = (size_t)E * H * I * 4;
    if (cudaMemsetAsync(dw13, 0, n13, stream) != cudaSuccess ||
        cudaMemsetAsync(dw2, 0, n2, stream) != cudaSuccess)
      return finish(-1);
  }
  return finish(launched);
}

// Router-backward workspace: dl [N,E] f32, its split copy [N,C] bf16, W_r's
// split copy [H,C] bf16 (C = moe::router_split_cols(E)), the dW_r partials
// [splits,H,E] f32; each region 256-byte aligned.
struct RouterBwdLayout {
  size_t dl, dls, wrs, part, total;
};

static RouterBwdLayout router_bwd_layout(const moe_config_t* c) {
  const int64_t N = c->n_tokens, H = c->hidden, E = c->n_experts;
  const int64_t C = moe::router_split_cols((int)E);
  const int64_t splits = N > 0 ? moe::router_bwd_splits((int)N, (int)H, (int)E) : 0;
  RouterBwdLayout L{};
  L.dl = 0;
  L.dls = L.dl + (size_t)roundup(N * E * 4, 256);
  L.wrs = L.dls + (size_t)roundup(N * C * 2, 256);
  L.part = L.wrs + (size_t)roundup(H * C * 2, 256);
  L.total = L.part + (size_t)roundup(splits * H * E * 4, 256);
  return L;
}

int64_t moe_router_backward_workspace_bytes(const moe_config_t* cfg) {
  const int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  return (int64_t)router_bwd_layout(cfg).total;
}

const float* moe_route_workspace_logits(const moe_config_t* cfg, const void* workspace) {
  if (check_cfg(cfg) != MOE_OK || !workspace) return nullptr;
  return reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) +
                                        ws_layout(cfg).logits);
}

int moe_router_backward(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                        const float* w_router, const float* bias, const float* logits,
                        const float* dprob, void* dx, float* dw_router, float* dbias,
                        void* workspace, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (cfg->n_valid) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!routes || !routes->topk_ids || !w_router || !dw_router) return MOE_ERR_INVALID_ARG;
  const RouterBwdLayout L = router_bwd_layout(cfg);
  if (cfg->n_tokens > 0 && (!workspace || ws_bytes < L.total || !aligned16(workspace)))
    return MOE_ERR_WORKSPACE;
  if (cfg->n_tokens > 0 && (!x || !dprob || !dx || !aligned16(x) || !aligned16(dx)))
    return MOE_ERR_INVALID_ARG;
  if (cfg->n_tokens == 0) {  // no token: zero gradients
    if (cudaMemsetAsync(dw_router, 0, (size_t)cfg->hidden * cfg->n_experts * 4, stream) !=
            cudaSuccess ||
        (dbias && cudaMemsetAsync(dbias, 0, (size_t)cfg->n_experts * 4, stream) != cudaSuccess))
      return finish(-1);
    return MOE_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  moe::RouterBwdArgs a{};
  a.err = error_word_ptr();
  if (!a.err) return MOE_ERR_CUDA;
  a.N = cfg->n_tokens;
  a.H = cfg->hidden;
  a.E = cfg->n_experts;
  a.K = cfg->top_k;
  a.renorm = cfg->renorm;
  a.x = static_cast<const uint16_t*>(x);
  a.wr = w_router;
  a.bias = bias;
  a.topk_ids = routes->topk_ids;
  a.dprob = dprob;
  a.logits = logits;
  a.dl = reinterpret_cast<float*>(ws + L.dl);
  a.dls = reinterpret_cast<uint16_t*>(ws + L.dls);
  a.wrs = reinterpret_cast<uint16_t*>(ws + L.wrs);
  a.part = reinterpret_cast<float*>(ws + L.part);
  a.dwr = dw_router;
  a.dbias = dbias;
  a.dx = static_cast<uint16_t*>(dx);
  return finish(moe::launch_router_backward(a, stream));
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA launch or driver error";
    case MOE_ERR_DEVICE: return "device-side error recorded";
    default: return "unknown status";
  }
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_device_error(uint32_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  uint32_t v = 0, zero = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, g_moe_error_word, sizeof v) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_moe_error_word, &zero, sizeof zero) != cudaSuccess) return MOE_ERR_CUDA;
  *out = v;
  return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// moe_route_align_noalloc: moe_route_align with a scratch array built into the
// library, for callers that cannot allocate device memory (see moe.h).
namespace {

static __device__ __align__(256) uint8_t g_route_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of g_route_scratch on the current device, looked up once per
// device (the host-side name is only a stand-in, not a device address).
uint8_t* route_scratch_ptr() {
  static std::mutex mu;
  static uint8_t* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return nullptr;
    ptrs[dev] = static_cast<uint8_t*>(p);
  }
  return ptrs[dev];
}

}  // namespace

extern "C" int moe_route_align_noalloc(const moe_config_t* cfg, const void* x,
                                       const float* w_router, const float* bias,
                                       const moe_routes_t* out, cudaStream_t stream) {
  const int rc = check_cfg(cfg);
  if (rc != MOE_OK) return rc;
  if (ws_layout(cfg).total > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  uint8_t* scratch = route_scratch_ptr();
  if (!scratch) return MOE_ERR_CUDA;
  return moe_route_align(cfg, x, w_router, bias, out, scratch, MOE_NOALLOC_SCRATCH_BYTES, stream);
}
