/*
 * Plain, slow CPU oracle of the capacity-bounded MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this file; the library path never does. It shares
 * no code, header or constant table with the CUDA library.
 *
 * Steps, in the order the pages give them:
 *   1. router: logits -> softmax -> top-K -> renormalise
 *      (router precedes dispatch: "Permute-Free Grouped GEMM for MoE (bf16,
 *      gfx950)", section 1 "Motivation"; the captured region "starts after
 *      routing": "feat(cuda-graphs): capture fixed-capacity MoE execution",
 *      "What does this PR do?")
 *   2. source capacity ceil(N*K*F/E) ("feat(cuda-graphs) ...", "Design notes")
 *   3. drop-and-pad: each expert keeps at most `capacity` routes, chosen by
 *      routing probability; unused slots carry no probability (same section)
 *   4. route-list layout: expert-sorted, block-padded sorted_slot_ids with
 *      sentinel N, expert_ids (-1 for blocks without a kept route),
 *      block_start, num_tokens_post_padded, token_routes ("Permute-Free ...",
 *      section 4 "Data structures")
 *   5. expert FFN on kept routes: FC1 on the gathered row, the gated
 *      activation act(gate)*up (silu or gelu; optionally times p'), FC2
 *      ("Permute-Free ...", section 3 "End-to-end flow")
 *   6. gather-combine: each token sums its kept routes weighted by routing
 *      probability ("Permute-Free ...", section 2 "Core idea")
 * Dropless, bucketed variant and backward (second half of the file):
 *   7. dropless layout: per-expert extents from a ladder of multiples of the
 *      expected rows ("[4/5] feat: capture the FFN experts at bucketed padded
 *      shapes", What this adds)
 *   8. expert-path backward given dY: FC2 data gradient, SwiGLU backward with
 *      the activation recomputed from gate and up, routing-weight gradient,
 *      FC1 data gradient reduced per token, weight gradients in slot order
 *      ("Permute-Free ...", sections 3, 5 and 6)
 *
 * Floating point: fp32 throughout, as the library's contract states (fp32
 * accumulation). Every output element is produced by one thread in a fixed
 * order, so results do not depend on the OpenMP thread count. Build with
 * -ffp-contract=off so that no a*b+c is fused except where fmaf() is written.
 *
 * Parity pins (tests/test_oracle_pins.py, tests/test_oracle_backward_pins.py):
 * capacity worked values, invariants of both layouts, hand-worked layouts,
 * brute-force selection by rank counting, a dense fp64 reference on tiny
 * inputs, exp against the C library, top-K against a stable sort, reductions
 * to a plain SwiGLU MLP (E=1,K=1) and to a dense softmax mixture (K=E),
 * central finite differences of an fp64 forward for every backward output.
 * tests/test_oracle_mutations.py plants mistakes here and checks a pin fails.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static float bits_to_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* fp32 exp used by the router softmax.                                      */
/* Cody-Waite argument reduction v = n*ln2 + r with n = rint(v*log2(e)), the */
/* constant ln 2 split in two fp32 parts (hi = ln 2 rounded to fp32, lo = the */
/* remainder rounded to fp32), then the degree-7 Taylor polynomial of e^r in  */
/* Horner form with fma, then scaling by 2^n through the exponent bits.       */
/* Domain used by the softmax: v <= 0. v < -87 returns +0.                    */
/* ------------------------------------------------------------------------ */
float oracle_exp(float v) {
  if (v < -87.0f) return 0.0f;
  const float log2e = (float)(1.0 / M_LN2);
  const float ln2_hi = (float)M_LN2;
  const float ln2_lo = (float)(M_LN2 - (double)ln2_hi);
  float n = rintf(v * log2e);
  float r = fmaf(-n, ln2_hi, v);
  r = fmaf(-n, ln2_lo, r);
  /* 1/k! for k = 7 .. 0, each rounded from double to fp32 */
  float p = (float)(1.0 / 5040.0);
  p = fmaf(p, r, (float)(1.0 / 720.0));
  p = fmaf(p, r, (float)(1.0 / 120.0));
  p = fmaf(p, r, (float)(1.0 / 24.0));
  p = fmaf(p, r, (float)(1.0 / 6.0));
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  int ni = (int)n;
  float scale = bits_to_f32((uint32_t)(ni + 127) << 23);
  return p * scale;
}

/* ------------------------------------------------------------------------ */
/* Step 1: router.                                                           */
/* logits l[t,e] = (sum over h ascending of x[t,h]*Wr[h,e], one fp32 fma per */
/*   term) + b[e];                                                           */
/* p = softmax(l): m = max_e l, z_e = exp(l_e - m), s = sum of z_e in        */
/*   ascending e, p_e = z_e / s;                                             */
/* top-K: K times take the largest p_e not yet taken, ties to the lower e;   */
/* renormalise (renorm=1): d = sum of the K chosen p in pick order,          */
/*   p'_k = p_k / d; renorm=0 keeps p'_k = p_k.                              */
/* probs_out (optional, [N,E]) receives p; logits_out (optional) receives l. */
/* ------------------------------------------------------------------------ */
int oracle_router(int N, int H, int E, int K, int renorm, const uint16_t* x, const float* wr,
                  const float* bias, int32_t* topk_ids, float* topk_p, float* probs_out,
                  float* logits_out) {
  if (N < 0 || H <= 0 || E <= 0 || K <= 0 || K > E) return -1;
  int bad = 0;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < N; ++t) {
    float* l = (float*)malloc(sizeof(float) * (size_t)E);
    float* p = (float*)malloc(sizeof(float) * (size_t)E);
    char* taken = (char*)calloc((size_t)E, 1);
    if (!l || !p || !taken) {
#pragma omp atomic write
      bad = 1;
      free(l); free(p); free(taken);
      continue;
    }
    for (int e = 0; e < E; ++e) {
      float acc = 0.0f;
      for (int h = 0; h < H; ++h) acc = fmaf(bf16_to_f32(x[(size_t)t * H + h]), wr[(size_t)h * E + e], acc);
      l[e] = acc + (bias ? bias[e] : 0.0f);
    }
    float m = l[0];
    for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
    float s = 0.0f;
    for (int e = 0; e < E; ++e) {
      p[e] = oracle_exp(l[e] - m);
      s = s + p[e];
    }
    for (int e = 0; e < E; ++e) p[e] = p[e] / s;
    if (probs_out) memcpy(probs_out + (size_t)t * E, p, sizeof(float) * (size_t)E);
    if (logits_out) memcpy(logits_out + (size_t)t * E, l, sizeof(float) * (size_t)E);
    float d = 0.0f;
    for (int k = 0; k < K; ++k) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || p[e] > p[best]) best = e; /* strict '>' keeps the lower e on ties */
      }
      taken[best] = 1;
      topk_ids[(size_t)t * K + k] = best;
      topk_p[(size_t)t * K + k] = p[best];
      d = d + p[best];
    }
    if (renorm)
      for (int k = 0; k < K; ++k) topk_p[(size_t)t * K + k] = topk_p[(size_t)t * K + k] / d;
    free(l); free(p); free(taken);
  }
  return bad ? -2 : 0;
}

/* ------------------------------------------------------------------------ */
/* Step 2: source capacity ceil(N*K*F/E) with F = cap_num/cap_den, in exact  */
/* integer arithmetic.                                                       */
/* ------------------------------------------------------------------------ */
int64_t oracle_capacity(int64_t N, int64_t K, int64_t E, int64_t cap_num, int64_t cap_den) {
  if (E <= 0 || cap_den <= 0 || N < 0 || K < 0 || cap_num < 0) return -1;
  int64_t num = N * K * cap_num;
  int64_t den = E * cap_den;
  return (num + den - 1) / den;
}

/* ------------------------------------------------------------------------ */
/* Steps 3 and 4: drop-and-pad selection, then the route-list layout.        */
/* For each expert e: the routes (t,k) with topk_ids[t,k] == e, ordered by   */
/* (p' descending, t ascending); the first `cap` are kept, the rest dropped. */
/* Layout with Cpad = roundup(cap, bm): expert e owns slots                  */
/* [e*Cpad, (e+1)*Cpad); its kept tokens fill the first slots in ascending t; */
/* the other slots hold the sentinel N.                                      */
/* ------------------------------------------------------------------------ */
typedef struct {
  float p;
  int32_t t;
  int32_t r; /* route index t*K + k */
} route_key;

static int cmp_prob_desc_token_asc(const void* a, const void* b) {
  const route_key* x = (const route_key*)a;
  const route_key* y = (const route_key*)b;
  if (x->p > y->p) return -1;
  if (x->p < y->p) return 1;
  return (x->t > y->t) - (x->t < y->t);
}

static int cmp_token_asc(const void* a, const void* b) {
  const route_key* x = (const route_key*)a;
  const route_key* y = (const route_key*)b;
  return (x->t > y->t) - (x->t < y->t);
}

int oracle_select_layout(int N, int E, int K, int64_t cap, int bm, const int32_t* topk_ids,
                         const float* topk_p, uint8_t* keep, int32_t* expert_counts,
                         int32_t* kept_counts, int32_t* sorted_slot_ids, int32_t* expert_ids,
                         int32_t* block_start, int32_t* num_tokens_post_padded,
                         int32_t* token_routes) {
  if (N < 0 || E <= 0 || K <= 0 || cap < 0 || bm <= 0) return -1;
  const int64_t cpad = (cap + bm - 1) / bm * bm;
  const int64_t R = (int64_t)N * K;
  for (int64_t r = 0; r < R; ++r) { keep[r] = 0; token_routes[r] = -1; }
  for (int64_t s = 0; s < (int64_t)E * cpad; ++s) sorted_slot_ids[s] = N;
  route_key* buf = (route_key*)malloc(sizeof(route_key) * (size_t)(R > 0 ? R : 1));
  if (!buf) return -2;
  for (int e = 0; e < E; ++e) {
    int64_t n = 0;
    for (int64_t r = 0; r < R; ++r)
      if (topk_ids[r] == e) { buf[n].p = topk_p[r]; buf[n].t = (int32_t)(r / K); buf[n].r = (int32_t)r; ++n; }
    expert_counts[e] = (int32_t)n;
    qsort(buf, (size_t)n, sizeof(route_key), cmp_prob_desc_token_asc);
    int64_t kept = n < cap ? n : cap;
    kept_counts[e] = (int32_t)kept;
    qsort(buf, (size_t)kept, sizeof(route_key), cmp_token_asc); /* kept ones in ascending t */
    for (int64_t j = 0; j < kept; ++j) {
      int64_t slot = (int64_t)e * cpad + j;
      sorted_slot_ids[slot] = buf[j].t;
      keep[buf[j].r] = 1;
      token_routes[buf[j].r] = (int32_t)slot;
    }
    block_start[e] = (int32_t)((int64_t)e * cpad / bm);
  }
  const int64_t nblocks = (int64_t)E * cpad / bm;
  for (int64_t b = 0; b < nblocks; ++b) {
    int64_t e = b / (cpad / bm);
    int64_t first = b * bm - e * cpad; /* first slot of the block within expert e */
    expert_ids[b] = (first < kept_counts[e]) ? (int32_t)e : -1;
  }
  *num_tokens_post_padded = (int32_t)((int64_t)E * cpad);
  free(buf);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Gated activations of the expert FFN, act(gate) * up ("Permute-Free       */
/* Grouped GEMM for MoE (bf16, gfx950)", section 3: act(gate)*up; section 8: */
/* silu and gelu). act 0: silu(v) = v * sigma(v) = v / (1 + exp(-v)).        */
/* act 1: gelu(v) = v * Phi(v) = 0.5 v (1 + erf(v / sqrt 2)), the exact form.*/
/* act_grad is the derivative: silu' = sigma(v) (1 + v (1 - sigma(v))),      */
/* gelu' = Phi(v) + v phi(v), phi(v) = exp(-v^2/2) / sqrt(2 pi).             */
/* ------------------------------------------------------------------------ */
static float act_fn(int act, float v) {
  if (act == 1) return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
  return v / (1.0f + expf(-v));
}

static float act_grad(int act, float v) {
  if (act == 1) {
    const float cdf = 0.5f * (1.0f + erff(v * 0.70710678118654752f));
    const float pdf = expf(-0.5f * v * v) * 0.39894228040143268f;
    return cdf + v * pdf;
  }
  const float sg = 1.0f / (1.0f + expf(-v));
  return sg * (1.0f + v * (1.0f - sg));
}

/* ------------------------------------------------------------------------ */
/* Step 5: expert FFN for one route: token row x[t], expert e.               */
/*   g_i = sum_h x_h*Wg[e,h,i], u_i = sum_h x_h*Wu[e,h,i] (ascending h),     */
/*   a_i = act(g_i)*u_i*scale (scale = p' when the routing probability is    */
/*   applied in the activation, else 1),                                     */
/*   o_j = sum_i a_i*Wd[e,i,j] (ascending i).                                */
/* wg/wu point at expert e's [H,I] block, wd at its [I,H] block (bf16 bits). */
/* h_out (optional, [I]) receives a; o_out ([H]) receives o.                 */
/* ------------------------------------------------------------------------ */
static void ffn_one(int H, int I, const uint16_t* xrow, const uint16_t* wg, const uint16_t* wu,
                    const uint16_t* wd, int act, float scale, float* g, float* u, float* h_out,
                    float* o_out) {
  for (int i = 0; i < I; ++i) { g[i] = 0.0f; u[i] = 0.0f; }
  for (int h = 0; h < H; ++h) {
    const float xv = bf16_to_f32(xrow[h]);
    const uint16_t* wgr = wg + (size_t)h * I;
    const uint16_t* wur = wu + (size_t)h * I;
    for (int i = 0; i < I; ++i) {
      g[i] = g[i] + xv * bf16_to_f32(wgr[i]);
      u[i] = u[i] + xv * bf16_to_f32(wur[i]);
    }
  }
  for (int i = 0; i < I; ++i) {
    g[i] = act_fn(act, g[i]) * u[i] * scale; /* g now holds the activation a */
    if (h_out) h_out[i] = g[i];
  }
  for (int j = 0; j < H; ++j) o_out[j] = 0.0f;
  for (int i = 0; i < I; ++i) {
    const float a = g[i];
    const uint16_t* wdr = wd + (size_t)i * H;
    for (int j = 0; j < H; ++j) o_out[j] = o_out[j] + a * bf16_to_f32(wdr[j]);
  }
}

/* FFN for a list of (token, expert) pairs. Expert weights are addressed via
 * per-expert pointer tables so callers can hold only the experts they need.
 * act: gated activation (0 silu, 1 gelu); scales: [n] per-route factor of the
 * activation, or NULL for 1. h_out: [n,I] or NULL; o_out: [n,H]. */
int oracle_ffn_routes(int n, const int32_t* tokens, const int32_t* experts, int H, int I,
                      const uint16_t* x, const uint16_t* const* wg, const uint16_t* const* wu,
                      const uint16_t* const* wd, int act, const float* scales, float* h_out,
                      float* o_out) {
  int bad = 0;
#pragma omp parallel
  {
    float* g = (float*)malloc(sizeof(float) * (size_t)I);
    float* u = (float*)malloc(sizeof(float) * (size_t)I);
    if (!g || !u) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int j = 0; j < n; ++j) {
        const int e = experts[j];
        ffn_one(H, I, x + (size_t)tokens[j] * H, wg[e], wu[e], wd[e], act,
                scales ? scales[j] : 1.0f, g, u, h_out ? h_out + (size_t)j * I : NULL,
                o_out + (size_t)j * H);
      }
    }
    free(g); free(u);
  }
  return bad ? -2 : 0;
}

/* ------------------------------------------------------------------------ */
/* Step 6: gather-combine for tokens t in [t0, t1):                          */
/*   y[t] = sum over k = 0..K-1 with keep[t,k] of p'[t,k] * o_route[t,k],    */
/* fp32, in k order; a token with no kept route gives y = 0. topk_p NULL:    */
/* unit weights (the probability was applied in the activation).             */
/* o_routes: [(t1-t0)*K, H] rows, the FFN output of route (t,k) (rows of     */
/* dropped routes are ignored).                                              */
/* ------------------------------------------------------------------------ */
int oracle_combine(int t0, int t1, int K, int H, const uint8_t* keep, const float* topk_p,
                   const float* o_routes, float* y) {
#pragma omp parallel for schedule(static)
  for (int t = t0; t < t1; ++t) {
    float* yr = y + (size_t)(t - t0) * H;
    for (int j = 0; j < H; ++j) yr[j] = 0.0f;
    for (int k = 0; k < K; ++k) {
      const size_t r = (size_t)t * K + k;
      if (!keep[r]) continue;
      const float w = topk_p ? topk_p[r] : 1.0f;
      const float* orow = o_routes + ((size_t)(t - t0) * K + k) * H;
      for (int j = 0; j < H; ++j) yr[j] = yr[j] + w * orow[j];
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Whole forward for tokens [t0, t1) given the routing of all N tokens:      */
/* FFN of every kept route of those tokens, then the combine.                */
/* ------------------------------------------------------------------------ */
int oracle_forward_tokens(int t0, int t1, int K, int H, int I, const uint16_t* x,
                          const uint16_t* const* wg, const uint16_t* const* wu,
                          const uint16_t* const* wd, const int32_t* topk_ids,
                          const float* topk_p, const uint8_t* keep, int act, int prob_in_act,
                          float* y) {
  const int nt = t1 - t0;
  if (nt <= 0) return 0;
  float* o = (float*)calloc((size_t)nt * K * H, sizeof(float));
  int32_t* tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)nt * K);
  int32_t* ex = (int32_t*)malloc(sizeof(int32_t) * (size_t)nt * K);
  int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)nt * K);
  float* sc = (float*)malloc(sizeof(float) * (size_t)nt * K);
  if (!o || !tok || !ex || !pos || !sc) {
    free(o); free(tok); free(ex); free(pos); free(sc);
    return -2;
  }
  int n = 0;
  for (int t = t0; t < t1; ++t)
    for (int k = 0; k < K; ++k) {
      const size_t r = (size_t)t * K + k;
      if (!keep[r]) continue;
      tok[n] = t; ex[n] = topk_ids[r]; pos[n] = (t - t0) * K + k; sc[n] = topk_p[r]; ++n;
    }
  float* on = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1) * H);
  if (!on) { free(o); free(tok); free(ex); free(pos); free(sc); return -2; }
  int rc = oracle_ffn_routes(n, tok, ex, H, I, x, wg, wu, wd, act, prob_in_act ? sc : NULL, NULL, on);
  for (int j = 0; j < n; ++j) memcpy(o + (size_t)pos[j] * H, on + (size_t)j * H, sizeof(float) * (size_t)H);
  if (rc == 0) rc = oracle_combine(t0, t1, K, H, keep, prob_in_act ? NULL : topk_p, o, y);
  free(on); free(o); free(tok); free(ex); free(pos); free(sc);
  return rc;
}

/* ======================================================================== */
/* Dropless, bucketed variant ("[4/5] feat: capture the FFN experts at      */
/* bucketed padded shapes", What this adds): the rungs are multiples of the */
/* expected rows per expert; an expert's extent is the first rung at or     */
/* above its count, or its count rounded to the block when no rung fits.   */
/* Per expert: rung_j = roundup(ceil(num_j*R / (den*E)), bm) with R = N*K;  */
/* extent_e = the smallest rung >= count_e, else roundup(count_e, bm).      */
/* Nothing is dropped. Expert e's slots start at the exclusive scan of the  */
/* extents; its tokens fill them in ascending t, the rest hold sentinel N.  */
/* Slots past the total up to s_max hold N, their blocks -1.                */
/* ======================================================================== */
int64_t oracle_dropless_extent(int64_t count, int64_t R, int64_t E, int bm, const int32_t* ladder_num,
                               int ladder_len, int ladder_den) {
  for (int j = 0; j < ladder_len; ++j) {
    const int64_t num = (int64_t)ladder_num[j] * R;
    const int64_t den = (int64_t)ladder_den * E;
    int64_t rung = (num + den - 1) / den;
    rung = (rung + bm - 1) / bm * bm;
    if (count <= rung) return rung;
  }
  return (count + bm - 1) / bm * bm;
}

int oracle_dropless_layout(int N, int E, int K, int bm, const int32_t* ladder_num, int ladder_len,
                           int ladder_den, int64_t s_max, const int32_t* topk_ids,
                           int32_t* expert_counts, int32_t* extents, int32_t* block_start,
                           int32_t* sorted_slot_ids, int32_t* expert_ids,
                           int32_t* num_tokens_post_padded, int32_t* token_routes) {
  const int64_t R = (int64_t)N * K;
  for (int e = 0; e < E; ++e) expert_counts[e] = 0;
  for (int64_t r = 0; r < R; ++r) expert_counts[topk_ids[r]] += 1;
  int64_t base = 0;
  for (int e = 0; e < E; ++e) {
    extents[e] = (int32_t)oracle_dropless_extent(expert_counts[e], R, E, bm, ladder_num, ladder_len,
                                                 ladder_den);
    block_start[e] = (int32_t)(base / bm);
    base += extents[e];
  }
  if (base > s_max) return -3;
  *num_tokens_post_padded = (int32_t)base;
  for (int64_t s = 0; s < s_max; ++s) sorted_slot_ids[s] = N;
  for (int64_t b = 0; b < s_max / bm; ++b) expert_ids[b] = -1;
  for (int e = 0; e < E; ++e) {
    const int64_t b0 = (int64_t)block_start[e] * bm;
    int64_t j = 0;
    for (int t = 0; t < N; ++t) /* ascending token order */
      for (int k = 0; k < K; ++k)
        if (topk_ids[(int64_t)t * K + k] == e) {
          sorted_slot_ids[b0 + j] = t;
          token_routes[(int64_t)t * K + k] = (int32_t)(b0 + j);
          ++j;
        }
    for (int64_t b = 0; b < extents[e] / bm; ++b)
      expert_ids[b0 / bm + b] = (b * bm < expert_counts[e]) ? e : -1;
  }
  return 0;
}

/* ======================================================================== */
/* Backward of the expert path for one route (token t, expert e, weight p'): */
/* the vector-Jacobian product of y[t] += p' * o with o = a . Wd[e],        */
/* a = act(g)*u, g = x_t . Wg[e], u = x_t . Wu[e], given dY[t] (the same   */
/* whether p' multiplies in the combine or in the activation):              */
/*   dA0_i = sum_j dY_j * Wd[e,i,j]        (FC2 data gradient, route space) */
/*   dprob = sum_i a_i * dA0_i             (gradient of the routing weight) */
/*   dA = p' * dA0                                                          */
/*   dg_i = dA_i * u_i * act'(g_i)         (act_grad above)                 */
/*   du_i = dA_i * act(g_i)                                                 */
/*   dXr_h = sum_i dg_i*Wg[e,h,i] + du_i*Wu[e,h,i]                          */
/* SwiGLU is recomputed from g and u ("Permute-Free ...", section 6: "swiglu */
/* is just an op", recomputed in the backward). fp32, fixed orders.          */
/* Outputs (any may be NULL): dprob, dxr [H], dg [I], du [I], aw [I] = p'*a. */
/* ======================================================================== */
static void bwd_one(int H, int I, int act, float p, const uint16_t* xrow, const uint16_t* dyrow,
                    const uint16_t* wg, const uint16_t* wu, const uint16_t* wd, float* g, float* u,
                    float* da0, float* dprob, float* dxr, float* dg_out, float* du_out,
                    float* aw_out) {
  for (int i = 0; i < I; ++i) { g[i] = 0.0f; u[i] = 0.0f; }
  for (int h = 0; h < H; ++h) {
    const float xv = bf16_to_f32(xrow[h]);
    for (int i = 0; i < I; ++i) {
      g[i] = g[i] + xv * bf16_to_f32(wg[(size_t)h * I + i]);
      u[i] = u[i] + xv * bf16_to_f32(wu[(size_t)h * I + i]);
    }
  }
  for (int i = 0; i < I; ++i) {
    float acc = 0.0f;
    const uint16_t* wdr = wd + (size_t)i * H;
    for (int j = 0; j < H; ++j) acc = acc + bf16_to_f32(dyrow[j]) * bf16_to_f32(wdr[j]);
    da0[i] = acc;
  }
  float dp = 0.0f;
  for (int i = 0; i < I; ++i) {
    const float ag = act_fn(act, g[i]);
    const float a = ag * u[i];
    dp = dp + a * da0[i];
    const float dA = p * da0[i];
    const float dgi = dA * u[i] * act_grad(act, g[i]);
    const float dui = dA * ag;
    if (aw_out) aw_out[i] = p * a;
    da0[i] = dgi; /* reuse: da0 now holds dg */
    u[i] = dui;   /* reuse: u now holds du */
  }
  if (dprob) *dprob = dp;
  if (dg_out) memcpy(dg_out, da0, sizeof(float) * (size_t)I);
  if (du_out) memcpy(du_out, u, sizeof(float) * (size_t)I);
  if (dxr) {
    for (int h = 0; h < H; ++h) {
      float acc = 0.0f;
      const uint16_t* wgr = wg + (size_t)h * I;
      const uint16_t* wur = wu + (size_t)h * I;
      for (int i = 0; i < I; ++i)
        acc = acc + da0[i] * bf16_to_f32(wgr[i]) + u[i] * bf16_to_f32(wur[i]);
      dxr[h] = acc;
    }
  }
}

/* Backward for a list of n routes (token, expert, p'). Per route outputs as in
 * bwd_one, stored row-wise; NULL skips an output. */
int oracle_bwd_routes(int n, const int32_t* tokens, const int32_t* experts, const float* probs, int H,
                      int I, int act, const uint16_t* x, const uint16_t* dy, const uint16_t* const* wg,
                      const uint16_t* const* wu, const uint16_t* const* wd, float* dprob,
                      float* dxr, float* dg, float* du, float* aw) {
  int bad = 0;
#pragma omp parallel
  {
    float* g = (float*)malloc(sizeof(float) * (size_t)I);
    float* u = (float*)malloc(sizeof(float) * (size_t)I);
    float* d = (float*)malloc(sizeof(float) * (size_t)I);
    if (!g || !u || !d) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int r = 0; r < n; ++r) {
        const int e = experts[r];
        const int t = tokens[r];
        bwd_one(H, I, act, probs[r], x + (size_t)t * H, dy + (size_t)t * H, wg[e], wu[e], wd[e], g, u, d,
                dprob ? dprob + r : NULL, dxr ? dxr + (size_t)r * H : NULL,
                dg ? dg + (size_t)r * I : NULL, du ? du + (size_t)r * I : NULL,
                aw ? aw + (size_t)r * I : NULL);
      }
    }
    free(g); free(u); free(d);
  }
  return bad ? -2 : 0;
}

/* Weight gradients of one expert from its routes in ascending slot order:
 *   dWd[i,j] = sum_s aw_s[i] * dY[t_s, j]     (aw = p' * a)
 *   dWg[h,i] = sum_s x[t_s, h] * dg_s[i],  dWu[h,i] = sum_s x[t_s, h] * du_s[i]
 * n routes; rows of aw/dg/du [n, I]; outputs fp32 (any may be NULL). */
int oracle_wgrad_expert(int n, const int32_t* tokens, int H, int I, const uint16_t* x,
                        const uint16_t* dy, const float* aw, const float* dg, const float* du,
                        float* dwd /*[I,H]*/, float* dwg /*[H,I]*/, float* dwu /*[H,I]*/) {
  if (dwd) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < I; ++i)
      for (int j = 0; j < H; ++j) {
        float acc = 0.0f;
        for (int s = 0; s < n; ++s)
          acc = acc + aw[(size_t)s * I + i] * bf16_to_f32(dy[(size_t)tokens[s] * H + j]);
        dwd[(size_t)i * H + j] = acc;
      }
  }
  if (dwg || dwu) {
#pragma omp parallel for schedule(static)
    for (int h = 0; h < H; ++h)
      for (int i = 0; i < I; ++i) {
        float ag = 0.0f, au = 0.0f;
        for (int s = 0; s < n; ++s) {
          const float xv = bf16_to_f32(x[(size_t)tokens[s] * H + h]);
          ag = ag + xv * dg[(size_t)s * I + i];
          au = au + xv * du[(size_t)s * I + i];
        }
        if (dwg) dwg[(size_t)h * I + i] = ag;
        if (dwu) dwu[(size_t)h * I + i] = au;
      }
  }
  return 0;
}

/* ======================================================================== */
/* Router backward: the gradient of the routing probabilities p' (dprob,    */
/* [N,K], d loss / d p'[t,k]) through top-K renormalisation and the softmax */
/* to the logits, then to W_r, the bias and x. The chosen set is the one of */
/* the forward (top-K selection is piecewise constant). Per token t, with   */
/* p = softmax(l) and the chosen experts e_k:                               */
/*   renorm:  d = sum_k p[e_k],  p'_k = p[e_k]/d,                           */
/*            g[e_k] = (dprob_k - sum_j dprob_j p'_j) / d                   */
/*   no renorm: g[e_k] = dprob_k;   g[e] = 0 for experts not chosen         */
/*   dl[e] = p[e] * (g[e] - sum_j g[e_j] p[e_j])                            */
/* and dWr[h,e] = sum_t x[t,h] dl[t,e], dbias[e] = sum_t dl[t,e],           */
/* dx[t,h] = sum_e dl[t,e] Wr[h,e]. probs [N,E] from oracle_router.         */
/* Outputs may be NULL except dlogits.                                      */
/* ======================================================================== */
int oracle_router_backward(int N, int H, int E, int K, int renorm, const uint16_t* x,
                           const float* wr, const float* probs, const int32_t* topk_ids,
                           const float* dprob, float* dlogits, float* dwr, float* dbias,
                           float* dx) {
  if (N < 0 || H <= 0 || E <= 0 || K <= 0 || K > E || K > 16 || !dlogits) return -1;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < N; ++t) {
    const float* p = probs + (size_t)t * E;
    const int32_t* ids = topk_ids + (size_t)t * K;
    const float* dp = dprob + (size_t)t * K;
    float* dl = dlogits + (size_t)t * E;
    float gk[16];
    if (renorm) {
      float d = 0.0f;
      for (int k = 0; k < K; ++k) d = d + p[ids[k]];
      float c = 0.0f;
      for (int k = 0; k < K; ++k) c = c + dp[k] * (p[ids[k]] / d);
      for (int k = 0; k < K; ++k) gk[k] = (dp[k] - c) / d;
    } else {
      for (int k = 0; k < K; ++k) gk[k] = dp[k];
    }
    float s = 0.0f;
    for (int k = 0; k < K; ++k) s = s + gk[k] * p[ids[k]];
    for (int e = 0; e < E; ++e) dl[e] = -p[e] * s;
    for (int k = 0; k < K; ++k) dl[ids[k]] = p[ids[k]] * (gk[k] - s);
  }
  if (dwr) {
#pragma omp parallel for schedule(static)
    for (int h = 0; h < H; ++h)
      for (int e = 0; e < E; ++e) {
        float acc = 0.0f;
        for (int t = 0; t < N; ++t)
          acc = acc + bf16_to_f32(x[(size_t)t * H + h]) * dlogits[(size_t)t * E + e];
        dwr[(size_t)h * E + e] = acc;
      }
  }
  if (dbias) {
    for (int e = 0; e < E; ++e) {
      float acc = 0.0f;
      for (int t = 0; t < N; ++t) acc = acc + dlogits[(size_t)t * E + e];
      dbias[e] = acc;
    }
  }
  if (dx) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < N; ++t)
      for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int e = 0; e < E; ++e) acc = acc + dlogits[(size_t)t * E + e] * wr[(size_t)h * E + e];
        dx[(size_t)t * H + h] = acc;
      }
  }
  return 0;
}

/* ======================================================================== */
/* FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no      */
/* infinities; exponent 15 with mantissa 7 is NaN; max finite 448).          */
/* Normal code (e >= 1): (1 + m/8) * 2^(e-7); subnormal (e = 0): m/8 * 2^-6. */
/* ======================================================================== */
float oracle_e4m3_decode(uint8_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
  return (c & 0x80) ? -v : v;
}

/* Nearest finite E4M3 value, ties to the even code (even mantissa), values at
 * or beyond 448 in magnitude saturate to +-448; NaN gives 0x7F. The 127 finite
 * non-negative codes ascend in value with the code, so the nearest one is the
 * smallest code whose value is >= |v| (found by bisection) or the code below
 * it. */
uint8_t oracle_e4m3_encode(float v) {
  if (v != v) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0;
  const float a = fabsf(v);
  if (a >= 448.0f) return sign | 0x7E;
  int lo = 0, hi = 0x7E;  /* decode(0x7E) = 448 > a */
  while (lo < hi) {
    const int mid = (lo + hi) / 2;
    if (oracle_e4m3_decode((uint8_t)mid) >= a) hi = mid;
    else lo = mid + 1;
  }
  if (lo == 0) return sign;  /* a == 0 */
  const float dc = oracle_e4m3_decode((uint8_t)lo) - a;      /* above, >= 0 */
  const float db = a - oracle_e4m3_decode((uint8_t)(lo - 1)); /* below, > 0 */
  const int best = (dc < db || (dc == db && (lo & 1) == 0)) ? lo : lo - 1;
  return sign | (uint8_t)best;
}

/* Row-wise FP8 quantisation of an [rows, cols] bf16 matrix: per row,
 * scale = max|v| / 448 (1 for an all-zero row), q = E4M3(v / scale) with the
 * division in fp32. */
int oracle_quantize_rows_fp8(int rows, int cols, const uint16_t* m, uint8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    const uint16_t* row = m + (size_t)r * cols;
    float amax = 0.0f;
    for (int c = 0; c < cols; ++c) amax = fmaxf(amax, fabsf(bf16_to_f32(row[c])));
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    scale[r] = s;
    for (int c = 0; c < cols; ++c) q[(size_t)r * cols + c] = oracle_e4m3_encode(bf16_to_f32(row[c]) / s);
  }
  return 0;
}

/* FC1 in FP8 for a list of (token, expert) routes: with x quantised per token
 * (xq [N,H], xs [N]) and the packed gate/up rows quantised per row
 * (wq [E,2I,H], ws [E,2I]; rows [0,I) gate, [I,2I) up),
 *   g_i = sum_h (E4M3(xq[t,h]) xs[t]) (E4M3(wq[e,i,h]) ws[e,i]),  u likewise,
 *   h_i = act(g_i) u_i (times scales[j] when given),
 * fp32, ascending h. h_out [n, I]. */
int oracle_fc1_fp8_routes(int n, const int32_t* tokens, const int32_t* experts, int H, int I,
                          const uint8_t* xq, const float* xs, const uint8_t* wq, const float* ws,
                          int act, const float* scales, float* h_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int j = 0; j < n; ++j) {
    const int t = tokens[j], e = experts[j];
    const uint8_t* xr = xq + (size_t)t * H;
    for (int i = 0; i < I; ++i) {
      const size_t rg = (size_t)e * 2 * I + i, ru = rg + I;
      const uint8_t* wg = wq + rg * H;
      const uint8_t* wu = wq + ru * H;
      float g = 0.0f, u = 0.0f;
      for (int h = 0; h < H; ++h) {
        const float xv = oracle_e4m3_decode(xr[h]) * xs[t];
        g = g + xv * (oracle_e4m3_decode(wg[h]) * ws[rg]);
        u = u + xv * (oracle_e4m3_decode(wu[h]) * ws[ru]);
      }
      h_out[(size_t)j * I + i] = act_fn(act, g) * u * (scales ? scales[j] : 1.0f);
    }
  }
  return 0;
}

/* FC2 in FP8 for n routes: with each route's h row quantised (hq [n,I],
 * hs [n]) and each w2 row quantised (wq [E,H,I], ws [E,H]; row c of expert e
 * is the c-th column of W_down[e]),
 *   o_c = sum_i (E4M3(hq[j,i]) hs[j]) (E4M3(wq[e,c,i]) ws[e,c]),
 * fp32, ascending i. o_out [n, H]. */
int oracle_fc2_fp8_routes(int n, const int32_t* experts, int H, int I, const uint8_t* hq,
                          const float* hs, const uint8_t* wq, const float* ws, float* o_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int j = 0; j < n; ++j) {
    const int e = experts[j];
    const uint8_t* hr = hq + (size_t)j * I;
    for (int c = 0; c < H; ++c) {
      const size_t r = (size_t)e * H + c;
      const uint8_t* wr = wq + r * I;
      float o = 0.0f;
      for (int i = 0; i < I; ++i)
        o = o + (oracle_e4m3_decode(hr[i]) * hs[j]) * (oracle_e4m3_decode(wr[i]) * ws[r]);
      o_out[(size_t)j * H + c] = o;
    }
  }
  return 0;
}

/* ======================================================================== */
/* MX block-scaled FP8 (MXFP8 E4M3). No page defines a block-scaled format; */
/* the definition is the OCP Microscaling Formats (MX) v1.0 specification,  */
/* the format tcgen05's kind::mxf8f6f4 consumes: a block of 32 consecutive  */
/* values along the contraction shares one scale X = 2^s, stored as an E8M0 */
/* byte (code c encodes 2^(c-127); 255 is NaN), and each value is an E4M3   */
/* code P_i, the value being P_i * X.                                       */
/* Quantisation of one block (the specification's conversion):             */
/*   s = floor(log2(max_i |v_i|)) - 8, 8 being the exponent of the largest  */
/*       power of two E4M3 holds (256 <= 448 < 512); s clamped to           */
/*       [-127, 127]; an all-zero block takes s = -127 (code 0);            */
/*   P_i = E4M3(v_i / 2^s), round to nearest even, saturating at +-448 (a   */
/*       block maximum in [448, 512) * 2^s saturates).                      */
/* The division by 2^s is exact (a power of two).                           */
/* ======================================================================== */
float oracle_e8m0_decode(uint8_t c) {
  if (c == 255) return NAN;
  return ldexpf(1.0f, (int)c - 127);
}

static int mx_block_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  int e;
  frexpf(amax, &e);  /* amax = f * 2^e with f in [0.5, 1): floor(log2 amax) = e - 1 */
  int s = (e - 1) - 8;
  if (s < -127) s = -127;
  if (s > 127) s = 127;
  return s;
}

/* MX quantisation of an [rows, cols] bf16 matrix along its rows (cols a
 * multiple of 32): codes q [rows, cols], scale codes sc [rows, cols / 32]. */
int oracle_quantize_mx_fp8(int rows, int cols, const uint16_t* m, uint8_t* q, uint8_t* sc) {
  if (cols % 32 != 0) return -1;
  const int nb = cols / 32;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < nb; ++b) {
      const uint16_t* blk = m + (size_t)r * cols + (size_t)b * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(bf16_to_f32(blk[i])));
      const int s = mx_block_exponent(amax);
      sc[(size_t)r * nb + b] = (uint8_t)(s + 127);
      for (int i = 0; i < 32; ++i)
        q[(size_t)r * cols + (size_t)b * 32 + i] = oracle_e4m3_encode(ldexpf(bf16_to_f32(blk[i]), -s));
    }
  }
  return 0;
}

/* FC1 on MX operands for a list of (token, expert) routes: x quantised along
 * H per token (xq [N,H], xs [N,H/32]), the packed gate/up rows along H
 * (wq [E,2I,H], ws [E*2I, H/32]; rows [0,I) gate, [I,2I) up):
 *   g_i = sum_h (E4M3(xq[t,h]) X(xs[t,h/32])) (E4M3(wq[e,i,h]) X(ws[e,i,h/32])),
 *   u likewise, h_i = act(g_i) u_i (times scales[j] when given),
 * fp32, ascending h. h_out [n, I]. */
int oracle_fc1_mx_routes(int n, const int32_t* tokens, const int32_t* experts, int H, int I,
                         const uint8_t* xq, const uint8_t* xs, const uint8_t* wq, const uint8_t* ws,
                         int act, const float* scales, float* h_out) {
  if (H % 32 != 0) return -1;
  const int nb = H / 32;
#pragma omp parallel for schedule(dynamic, 1)
  for (int j = 0; j < n; ++j) {
    const int t = tokens[j], e = experts[j];
    const uint8_t* xr = xq + (size_t)t * H;
    const uint8_t* xsr = xs + (size_t)t * nb;
    for (int i = 0; i < I; ++i) {
      const size_t rg = (size_t)e * 2 * I + i, ru = rg + I;
      const uint8_t* wg = wq + rg * H;
      const uint8_t* wu = wq + ru * H;
      float g = 0.0f, u = 0.0f;
      for (int h = 0; h < H; ++h) {
        const int b = h / 32;
        const float xv = oracle_e4m3_decode(xr[h]) * oracle_e8m0_decode(xsr[b]);
        g = g + xv * (oracle_e4m3_decode(wg[h]) * oracle_e8m0_decode(ws[rg * nb + b]));
        u = u + xv * (oracle_e4m3_decode(wu[h]) * oracle_e8m0_decode(ws[ru * nb + b]));
      }
      h_out[(size_t)j * I + i] = act_fn(act, g) * u * (scales ? scales[j] : 1.0f);
    }
  }
  return 0;
}

/* FC2 on MX operands for n routes: each route's h row quantised along I
 * (hq [n,I], hs [n,I/32]) and each w2 row along I (wq [E,H,I],
 * ws [E*H, I/32]):
 *   o_c = sum_i (E4M3(hq[j,i]) X(hs[j,i/32])) (E4M3(wq[e,c,i]) X(ws[e,c,i/32])),
 * fp32, ascending i. o_out [n, H]. */
int oracle_fc2_mx_routes(int n, const int32_t* experts, int H, int I, const uint8_t* hq,
                         const uint8_t* hs, const uint8_t* wq, const uint8_t* ws, float* o_out) {
  if (I % 32 != 0) return -1;
  const int nb = I / 32;
#pragma omp parallel for schedule(dynamic, 1)
  for (int j = 0; j < n; ++j) {
    const int e = experts[j];
    const uint8_t* hr = hq + (size_t)j * I;
    const uint8_t* hsr = hs + (size_t)j * nb;
    for (int c = 0; c < H; ++c) {
      const size_t r = (size_t)e * H + c;
      const uint8_t* wr = wq + r * I;
      float o = 0.0f;
      for (int i = 0; i < I; ++i) {
        const int b = i / 32;
        o = o + (oracle_e4m3_decode(hr[i]) * oracle_e8m0_decode(hsr[b])) *
                    (oracle_e4m3_decode(wr[i]) * oracle_e8m0_decode(ws[r * nb + b]));
      }
      o_out[(size_t)j * H + c] = o;
    }
  }
  return 0;
}
