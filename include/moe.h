/*
 * moe.h: C ABI of the capacity-bounded Mixture-of-Experts layer forward on a
 * single NVIDIA GB300 (sm_103a).
 *
 * Data flow, one stream, no host synchronisation, no allocation:
 *
 *   moe_route_align : x . W_r (+ b) -> softmax -> top-K -> renormalise
 *                     -> per-expert counts -> drop-and-pad selection
 *                     -> expert-sorted, block-padded route list
 *   moe_ffn_forward : FC1 gather-GEMM (rows of x gathered by sorted_slot_ids
 *                     inside the tile load) with the gated activation
 *                     (SwiGLU or GeGLU) in its epilogue, then
 *                     FC2 grouped GEMM over the same slots
 *   moe_combine     : each token sums its kept routes, weighted by the
 *                     renormalised routing probability
 *
 * Sources ("the pages"):
 *  [FC]  "feat(cuda-graphs): capture fixed-capacity MoE execution", NVIDIA-NeMo
 *        Automodel #2932: Design notes (capacity, drop-and-pad, constant
 *        per-expert row counts), What does this PR do (captured boundary).
 *  [PF]  "Permute-Free Grouped GEMM for MoE (bf16, gfx950)", ROCm
 *        TransformerEngine #694: section 2 Core idea (gather-in-GEMM,
 *        contention-free gather-combine), section 3 End-to-end flow, section 4
 *        Data structures (sorted_slot_ids, expert_ids, block_start,
 *        num_tokens_post_padded, token_routes), section 5 Kernels.
 *  [BK]  "[4/5] feat: capture the FFN experts at bucketed padded shapes",
 *        vllm-project/afd-plugin #335: What this adds (a grouped GEMM takes
 *        its grouping from a device-side count vector).
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers owned by the caller, allocated
 *    to the static sizes given below. The library never allocates, frees,
 *    synchronises, or reads device data on the host, so every call may be
 *    captured in a CUDA graph ([PF] section 6 "CUDA-graph capturable").
 *  - Row-major layouts; bf16 tensors are passed as `const void*` holding IEEE
 *    bfloat16 values. Pointers to bf16 tensors must be 16-byte aligned.
 *  - Return 0 on success, a negative MOE_ERR_* code otherwise. Invalid
 *    arguments are rejected before any launch; unsupported shapes fail closed
 *    (never a silent fallback), as [FC] Changelog / Known limitations does.
 *  - `stream` is the CUDA stream all work is queued on (0 = legacy default).
 *  - The forward-path kernels are launched with programmatic stream
 *    serialization: each may start its on-chip setup while the previous
 *    kernel in the stream drains, and waits for that kernel to complete
 *    before its first global-memory access, so stream order semantics hold.
 *    Stream capture records these as programmatic edges.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)       /* null pointer, misaligned pointer, bad field */
#define MOE_ERR_UNSUPPORTED_SHAPE (-2) /* shape outside what the kernels implement */
#define MOE_ERR_WORKSPACE (-3)         /* workspace missing or smaller than required */
#define MOE_ERR_CUDA (-4)              /* a CUDA launch or driver call failed */
#define MOE_ERR_DEVICE (-5)            /* a kernel recorded an error (moe_device_error) */

/* Layer shape and routing policy.
 *  n_tokens  N   tokens in the batch (0 allowed: every call is a no-op)
 *  hidden    H   model width; multiple of 128
 *  n_experts E   1..256
 *  top_k     K   1..min(E,16) experts per token
 *  inter     I   gated-activation width per expert; multiple of 128
 *  cap_num/cap_den  capacity factor F = cap_num/cap_den; the source
 *                capacity is cap = ceil(N*K*F/E) ([FC] Design notes).
 *                cap_num = 0 selects the dropless, bucketed layout: no route
 *                is dropped and expert e's slot region has the extent of the
 *                smallest ladder rung that holds its route count ([BK] What
 *                this adds), or its count rounded up to bm if none does
 *  block_m   bm  padding granularity of the route list: 16, 32, 64 or 128
 *  renorm    1 = renormalise the K chosen probabilities to sum to 1, 0 = keep
 *                the softmax probabilities
 *  ladder_len, ladder_den, ladder_num (dropless only; ladder_len 0..16)
 *                rung j = roundup(ceil(ladder_num[j]*N*K / (ladder_den*E)), bm):
 *                multiples ladder_num[j]/ladder_den of the expected rows per
 *                expert; ladder_num is a host array, ascending, positive
 *  activation    the experts' gated activation act(gate)*up ([PF] section 3;
 *                section 8 tests silu and gelu): MOE_ACT_SWIGLU (silu) or
 *                MOE_ACT_GEGLU (gelu, the exact form v*Phi(v))
 *  prob_in_act   1 = the routing probability p' multiplies the activation in
 *                FC1's epilogue (act(gate)*up*p', [PF] section 3) and the
 *                combine sums the routes with unit weights; 0 = p' weights the
 *                combine. The same function either way.
 *  n_valid       NULL, or a DEVICE pointer to an int32 holding the live token
 *                count n <= n_tokens, read by the kernels when they run: the
 *                batch is x[0..n), n_tokens is only the static bound that sizes
 *                the buffers and grids. Capacity, the ladder and every routing
 *                result follow n ([PF] section 2: real extents carried as device
 *                scalars); rows n <= t < n_tokens get topk_ids -1, topk_p 0,
 *                keep 0, token_routes -1 and y = 0; the sentinel in sorted_slot_ids
 *                stays n_tokens. This lets one captured CUDA graph serve every
 *                batch up to its bound (moe_ladder_*). Forward calls only: the
 *                backward calls reject it (MOE_ERR_UNSUPPORTED_SHAPE). */
typedef struct moe_config {
  int32_t n_tokens;
  int32_t hidden;
  int32_t n_experts;
  int32_t top_k;
  int32_t inter;
  int32_t cap_num;
  int32_t cap_den;
  int32_t block_m;
  int32_t renorm;
  int32_t ladder_len;
  int32_t ladder_den;
  const int32_t* ladder_num;
  int32_t activation;
  int32_t prob_in_act;
  const int32_t* n_valid;
} moe_config_t;

#define MOE_ACT_SWIGLU 0
#define MOE_ACT_GEGLU 1

/* Routing metadata written by moe_route_align ([PF] section 4). All device
 * pointers, caller-allocated. With Cpad = roundup(cap, bm) and
 * S = E*Cpad = moe_max_slots():
 *  topk_ids        [N,K] i32  chosen experts, in descending probability
 *  topk_p          [N,K] f32  renormalised routing probabilities p'
 *  keep            [N,K] u8   1 if the route holds a slot, 0 if dropped
 *  expert_counts   [E]   i32  routes per expert before capacity
 *  kept_counts     [E]   i32  min(expert_counts, cap): the device-side count
 *                             vector the GEMMs take their grouping from ([BK])
 *  sorted_slot_ids [S]   i32  slot -> token row; expert e owns slots
 *                             [e*Cpad, (e+1)*Cpad), kept tokens first in
 *                             ascending token order, the rest hold the
 *                             sentinel N (a gather of row N reads zeros)
 *  expert_ids      [S/bm] i32 expert owning each bm-slot block, -1 for a block
 *                             holding no kept route
 *  block_start     [E]   i32  first block of expert e (slots start at
 *                             block_start[e]*bm)
 *  num_tokens_post_padded [1] i32  padded extent S, as a device scalar
 *  token_routes    [N,K] i32  inverse map: slot of route (t,k), -1 if dropped
 *  slot_prob       [S]   f32  p' of the route each slot holds, 0 for padding
 *  gemm_sched      [4]   i32  work counters of the expert GEMMs' tile scheduler;
 *                             zeroed by moe_route_align and left zeroed by every
 *                             GEMM call (a routes object serves one stream at a
 *                             time: GEMM calls sharing it must not overlap) */
typedef struct moe_routes {
  int32_t* topk_ids;
  float* topk_p;
  uint8_t* keep;
  int32_t* expert_counts;
  int32_t* kept_counts;
  int32_t* sorted_slot_ids;
  int32_t* expert_ids;
  int32_t* block_start;
  int32_t* num_tokens_post_padded;
  int32_t* token_routes;
  int32_t* gemm_sched;
  float* slot_prob;
} moe_routes_t;

/* Host-side size queries (no GPU work). Negative on an invalid config. */
int64_t moe_capacity(const moe_config_t* cfg);    /* cap = ceil(N*K*F/E); N when dropless */
/* S = E*roundup(cap,bm); dropless: N*K + E*(top rung + bm), the static bound of
 * the padded extent (the real extent is num_tokens_post_padded) */
int64_t moe_max_slots(const moe_config_t* cfg);
int64_t moe_max_blocks(const moe_config_t* cfg);  /* S / bm */
/* Bytes of scratch moe_route_align needs (0 when N == 0). */
int64_t moe_route_workspace_bytes(const moe_config_t* cfg);

/* Router, per-expert scan, drop-and-pad selection and route-list layout.
 *  x        [N,H] bf16 token activations
 *  w_router [H,E] f32 router weight; logits l[t,e] = sum_h x[t,h]*W_r[h,e]
 *           accumulated in ascending h with one fp32 fma per term, then + b[e]
 *  bias     [E]   f32 per-expert logit bias, or NULL for none
 *  out      routing metadata (every field required)
 *  workspace/ws_bytes  device scratch of at least moe_route_workspace_bytes
 * Softmax uses the library's own fp32 exp (Cody-Waite reduction, degree-7
 * Taylor polynomial); top-K ties go to the lower expert id; capacity keeps,
 * per expert, the routes with the highest p', ties to the lower token index
 * ([FC] Design notes: "selected by routing probability"). Results are
 * bit-identical from run to run. */
int moe_route_align(const moe_config_t* cfg, const void* x, const float* w_router,
                    const float* bias, const moe_routes_t* out, void* workspace,
                    size_t ws_bytes, cudaStream_t stream);

/* FC1 gather-GEMM + gated activation ([PF] section 2 and 3).
 *  x    [N,H] bf16; row sorted_slot_ids[s] of x feeds slot s
 *  w13  [E,2I,H] bf16 packed expert weights (moe_pack_w13): rows [0,I) of
 *       expert e are W_gate[e]^T, rows [I,2I) are W_up[e]^T
 *  h    [S,I] bf16 output, h[s,:] = act(x_s W_gate[e]) * (x_s W_up[e]) (times the
 *       slot's p' when cfg->prob_in_act) for
 *       s in expert e's slots; fp32 accumulation. Rows of slots at or past
 *       roundup(kept_counts[e],16) within an expert are not written; rows of
 *       padding slots below that bound are written as 0. */
int moe_fc1_forward(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                    const void* w13, void* h, cudaStream_t stream);

/* FC2 grouped GEMM ([PF] section 3: FC2 reads its rows by route position).
 *  h    [S,I] bf16 from moe_fc1_forward
 *  w2   [E,H,I] bf16 packed (moe_pack_w2): row j of expert e is W_down[e][:,j]
 *  o    [S,H] bf16 output, o[s,:] = h[s,:] W_down[e]; same written-row rule as h */
int moe_fc2_forward(const moe_config_t* cfg, const moe_routes_t* routes, const void* h,
                    const void* w2, void* o, cudaStream_t stream);

/* moe_fc1_forward followed by moe_fc2_forward on the same stream. */
int moe_ffn_forward(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                    const void* w13, const void* w2, void* h, void* o, cudaStream_t stream);

/* Training forward: moe_ffn_forward that also saves FC1's pre-activations for
 * moe_ffn_backward ("Permute-Free Grouped GEMM for MoE (bf16, gfx950)",
 * section 5: the FC1 kernel optionally writes the 2F pre-activation).
 *  preact [S,2I] bf16 output: columns [0,I) hold g = x_s W_gate[e], columns
 *         [I,2I) hold u = x_s W_up[e] (fp32 accumulation rounded to bf16); same
 *         written-row rule as h. Required (non-NULL) when N > 0.
 * Other arguments and outputs as moe_ffn_forward. */
int moe_ffn_forward_train(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                          const void* w13, const void* w2, void* h, void* o, void* preact,
                          cudaStream_t stream);

/* Contention-free gather-combine ([PF] section 2 and 5 "route_gather_combine").
 *  o  [S,H] bf16 expert outputs;  y [N,H] bf16 output:
 *  y[t,:] = sum over k with token_routes[t,k] >= 0 of topk_p[t,k]*o[token_routes[t,k],:]
 *  in fp32, in k order (unit weights instead of topk_p when cfg->prob_in_act).
 *  Dropped routes contribute nothing; a token with every route dropped gets
 *  y = 0. Each output row is written by one CTA; no atomics. */
int moe_combine(const moe_config_t* cfg, const moe_routes_t* routes, const void* o, void* y,
                cudaStream_t stream);

/* One-time weight packing into the K-major layouts the GEMMs read.
 *  w_gate, w_up [E,H,I] bf16 (x . W_gate[e] is [N,I]);  w13 [E,2I,H] bf16
 *  w_down       [E,I,H] bf16;                          w2  [E,H,I] bf16 */
int moe_pack_w13(const moe_config_t* cfg, const void* w_gate, const void* w_up, void* w13,
                 cudaStream_t stream);
int moe_pack_w2(const moe_config_t* cfg, const void* w_down, void* w2, cudaStream_t stream);

/* ---- FP8 (E4M3) expert GEMMs ------------------------------------------------
 * The pages run their experts in bf16 and reject FP8 ([FC] Changelog / Known
 * limitations: BF16 experts only); this is an extension beyond them, not a
 * mode they define. Operands are E4M3 codes (1 sign, 4 exponent bits with bias
 * 7, 3 mantissa bits, largest finite 448, no infinities) with one fp32 scale
 * per row: value = decode(code) * scale. The GEMMs accumulate the code products
 * in fp32 on the tensor cores and apply the weight-row scale times the
 * activation-row scale in the epilogue. */

/* Row-wise quantisation of a bf16 matrix.
 *  m         [rows, cols] bf16, rows <= INT32_MAX, cols a multiple of 8
 *  rows_dev  device int32 or NULL: when given, only rows below *rows_dev (read
 *            on the device when the kernel runs, e.g. num_tokens_post_padded
 *            for the slot rows of h) are quantised; the others are left as
 *            they are
 *  q         [rows, cols] u8 output codes, 16-byte aligned
 *  scale     [rows] f32 output: amax(|row|)/448 (fp32, correctly rounded), 1
 *            for an all-zero row
 * q = E4M3(m / scale): correctly rounded fp32 divide, then round to nearest
 * even with saturation to +-448. Weights are quantised once (w13 rows as
 * [E*2I, H], w2 rows as [E*H, I]); activations on each call. */
int moe_quantize_rows_fp8(const void* m, int64_t rows, const int32_t* rows_dev, int cols, void* q,
                          float* scale, cudaStream_t stream);

/* FC1 on FP8 operands, otherwise as moe_fc1_forward.
 *  xq  [N,H] u8, x_scale [N] f32    quantised token rows
 *  w13q [E,2I,H] u8, w13_scale [E*2I] f32   quantised packed gate/up rows
 *  h   [S,I] bf16 output, h[s,i] = act(g) u (times p' when cfg->prob_in_act),
 *      g = x_scale[t] w13_scale[e*2I+i] sum_k xq[t,k] w13q[e,i,k] (decoded codes),
 *      u likewise from row e*2I+I+i; fp32 accumulation; written-row rule as h
 *      in moe_fc1_forward. H must be a multiple of 128. */
int moe_fc1_forward_fp8(const moe_config_t* cfg, const moe_routes_t* routes, const void* xq,
                        const float* x_scale, const void* w13q, const float* w13_scale, void* h,
                        cudaStream_t stream);

/* FC2 on FP8 operands, otherwise as moe_fc2_forward.
 *  hq  [S,I] u8, h_scale [S] f32    quantised slot rows of h
 *  w2q [E,H,I] u8, w2_scale [E*H] f32   quantised packed w2 rows
 *  o   [S,H] bf16 output, o[s,c] = h_scale[s] w2_scale[e*H+c] sum_i hq[s,i] w2q[e,c,i]
 *      for the kept slots s of expert e; o = 0 in padding slots below
 *      roundup(kept_counts[e],16). I must be a multiple of 128. */
int moe_fc2_forward_fp8(const moe_config_t* cfg, const moe_routes_t* routes, const void* hq,
                        const float* h_scale, const void* w2q, const float* w2_scale, void* o,
                        cudaStream_t stream);

/* FP8 expert path for bf16 input: quantise x into xq/x_scale, FC1 on FP8
 * into h (bf16), quantise the slot rows of h that lie below
 * num_tokens_post_padded into hq/h_scale, FC2 on FP8 into o. Four launches on
 * one stream; the caller owns every buffer:
 *  x [N,H] bf16;  xq [N,H] u8;  x_scale [N] f32;  h [S,I] bf16;  hq [S,I] u8;
 *  h_scale [S] f32;  o [S,H] bf16;  weights as above. */
int moe_ffn_forward_fp8(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                        const void* w13q, const float* w13_scale, const void* w2q,
                        const float* w2_scale, void* xq, float* x_scale, void* h, void* hq,
                        float* h_scale, void* o, cudaStream_t stream);

/* ---- MX block-scaled FP8 (MXFP8 E4M3) expert GEMMs --------------------------
 * An extension beyond the pages as well (they run bf16 experts and reject FP8:
 * [FC] Changelog / Known limitations); the format is the OCP Microscaling
 * Formats (MX) v1.0 MXFP8: each block of 32 consecutive values along the
 * contraction shares one scale 2^s stored as an E8M0 byte (s + 127), each
 * value an E4M3 code; value = decode(code) * 2^s. Quantisation of a block:
 * s = floor(log2(max |v|)) - 8 clamped to [-127, 127] (-127 for an all-zero
 * block), code = E4M3(v * 2^-s) rounded to nearest even, saturating at +-448.
 * The tensor cores (tcgen05.mma kind::mxf8f6f4) apply both operands' block
 * scales inside the contraction, fp32 accumulation. */

/* MX quantisation of a bf16 matrix along its rows.
 *  m         [rows, cols] bf16, cols a multiple of 32, 16-byte aligned
 *  rows_dev  device int32 or NULL: only rows below *rows_dev (read on the
 *            device) are quantised; the others are left as they are
 *  q         [rows, cols] u8 output E4M3 codes, 16-byte aligned
 *  scale     [rows, cols/32] u8 output E8M0 codes, row-major
 * Used for the activations (x per token, h per slot) on each call. */
int moe_quantize_mx_fp8(const void* m, int64_t rows, const int32_t* rows_dev, int cols, void* q,
                        void* scale, cudaStream_t stream);

/* MX quantisation of packed weights (w13 rows as [E*2I, H], w2 rows as
 * [E*H, I]); rows and cols multiples of 128. Codes as above; the
 * rows*cols/32 scale bytes go in the layout the MX GEMMs copy to tensor
 * memory: 512-byte atoms, atom (rt, kt) = rows 128rt.., blocks 4kt..4kt+3 at
 * byte (rt * cols/128 + kt) * 512, row r's block b inside it at
 * (r%32)*16 + ((r%128)/32)*4 + b%4. Done once, before any forward. */
int moe_quantize_mx_fp8_weights(const void* m, int64_t rows, int cols, void* q, void* scale_atoms,
                                cudaStream_t stream);

/* FC1 on MX operands, otherwise as moe_fc1_forward.
 *  xq [N,H] u8, x_sf [N,H/32] u8    MX-quantised token rows (moe_quantize_mx_fp8)
 *  w13q [E,2I,H] u8, w13_sf         MX-quantised packed gate/up rows, scale atoms
 *                                   (moe_quantize_mx_fp8_weights)
 *  h [S,I] bf16 output: h = act(g) u (times p' with cfg->prob_in_act),
 *      g[s,i] = sum_k xq[t,k] 2^(x_sf[t,k/32]-127) w13q[e,i,k] 2^(sf(e*2I+i,k/32)-127)
 *      (decoded codes), u from row e*2I+I+i; fp32 accumulation. All scale
 *      buffers 16-byte aligned. */
int moe_fc1_forward_mx(const moe_config_t* cfg, const moe_routes_t* routes, const void* xq,
                       const void* x_sf, const void* w13q, const void* w13_sf, void* h,
                       cudaStream_t stream);

/* FC2 on MX operands, otherwise as moe_fc2_forward.
 *  hq [S,I] u8, h_sf [S,I/32] u8    MX-quantised slot rows of h
 *  w2q [E,H,I] u8, w2_sf            MX-quantised w2 rows, scale atoms
 *  o [S,H] bf16 output, o = 0 in padding slots below roundup(kept_counts[e],16). */
int moe_fc2_forward_mx(const moe_config_t* cfg, const moe_routes_t* routes, const void* hq,
                       const void* h_sf, const void* w2q, const void* w2_sf, void* o,
                       cudaStream_t stream);

/* MX expert path for bf16 input: quantise x into xq/x_sf, FC1 into h (bf16),
 * quantise the slot rows of h below num_tokens_post_padded into hq/h_sf, FC2
 * into o. Four launches on one stream; the caller owns every buffer:
 *  x [N,H] bf16; xq [N,H] u8; x_sf [N,H/32] u8; h [S,I] bf16; hq [S,I] u8;
 *  h_sf [S,I/32] u8; o [S,H] bf16; weights as above. */
int moe_ffn_forward_mx(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                       const void* w13q, const void* w13_sf, const void* w2q, const void* w2_sf,
                       void* xq, void* x_sf, void* h, void* hq, void* h_sf, void* o,
                       cudaStream_t stream);

/* Bytes of scratch moe_ffn_backward needs: about S*(2 + 6I + 2H) bytes plus
 * S*I/8 for the dprob partials (S = moe_max_slots). */
int64_t moe_backward_workspace_bytes(const moe_config_t* cfg);

/* Backward of the expert path y = sum_k p'_k FFN_e(x) for a given dY
 * ("Permute-Free Grouped GEMM for MoE (bf16, gfx950)", section 3 End-to-end
 * flow, backward, and section 5 Kernels: FC2 dgrad with the SwiGLU backward
 * in its epilogue, FC1 dgrad, FC1's input gradient reduced by the
 * gather-combine, weight gradients contracted over the token slots). Works in
 * both layouts; dropped routes contribute nothing.
 *  x, w13, w2  as in the forward;  preact [S,2I] bf16 from moe_ffn_forward_train
 *  dy     [N,H] bf16 gradient of y
 *  dx     [N,H] bf16 output: the gradient of y with respect to x through the
 *         experts, dX[t] = sum over kept k of (dg W_gate[e]^T + du W_up[e]^T)
 *         (the router's path is not included)
 *  dw13   [E,2I,H] f32 output, the gradient of the packed w13 (rows [0,I):
 *         dW_gate[e]^T, rows [I,2I): dW_up[e]^T); zero for an expert with no
 *         kept route
 *  dw2    [E,H,I] f32 output, the gradient of the packed w2 (dW_down[e]^T)
 *  dprob  [N,K] f32 output: dL/dp'[t,k] = <act(g) u, dY[t] W_down[e]^T> for a
 *         kept route, 0 for a dropped one
 *  workspace/ws_bytes  device scratch of at least moe_backward_workspace_bytes
 * fp32 accumulation everywhere; dPre = [dg | du], p' a and the per-route input
 * gradients are bf16 intermediates in the workspace. Outputs are overwritten. */
int moe_ffn_backward(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                     const void* w13, const void* w2, const void* preact, const void* dy,
                     void* dx, float* dw13, float* dw2, float* dprob, void* workspace,
                     size_t ws_bytes, cudaStream_t stream);

/* Bytes of scratch moe_router_backward needs: the logit gradient (N*E*4), its
 * bf16 split copy (N*C*2) and W_r's (H*C*2), C = 2*E rounded up to 128, and
 * the per-split partial sums of dW_r (one wave of CTA tiles). */
int64_t moe_router_backward_workspace_bytes(const moe_config_t* cfg);

/* Router backward: the gradient of the routing probabilities p' (dprob, e.g.
 * from moe_ffn_backward) through top-K renormalisation and the softmax to the
 * logits, then to the router weight, the bias and x. The chosen experts are
 * those in routes->topk_ids (moe_route_align of the same x, W_r, bias): top-K
 * selection is piecewise constant, so it passes no gradient. The pages'
 * routing probabilities carry a gradient to the router ("Permute-Free Grouped
 * GEMM for MoE (bf16, gfx950)", section 6: the SwiGLU backward optionally
 * computes the route-prob grad); this call continues that gradient. Per token,
 * with p = softmax(l) recomputed exactly as moe_route_align computes it:
 *   renorm: d = sum_k p[e_k], c = sum_k dprob_k p'_k, g_k = (dprob_k - c)/d
 *   else:   g_k = dprob_k;   s = sum_k g_k p[e_k]
 *   dl[e] = p[e] (g[e] - s)   (g = 0 for the experts not chosen)
 *  x, w_router, bias   the forward's inputs (bias may be NULL)
 *  logits     [N,E] f32: the logits moe_route_align left in its workspace
 *             (moe_route_workspace_logits), valid while that workspace is
 *             untouched; or NULL to recompute them (bit-identical either way)
 *  dprob      [N,K] f32 d loss / d p'
 *  dx         [N,H] bf16, in/out, 16-byte aligned: dx += dl . W_r^T, summed in
 *             fp32 and rounded to bf16 once (add the router's path to the
 *             experts' dX)
 *  dw_router  [H,E] f32 output: sum_t x[t,:]^T dl[t,:]
 *  dbias      [E] f32 output sum_t dl[t,:], or NULL
 * Outputs other than dx are overwritten. dl is computed in fp32; the two
 * contractions run on the tensor cores with dl and W_r each carried as a pair
 * of bf16 values (hi = bf16(v), lo = bf16(v - hi), 16 significant bits) and
 * fp32 accumulation, so they match fp32 sums up to accumulation order
 * (dx: hi.hi + lo.hi + hi.lo; dW_r: x.hi + x.lo, x being bf16); dbias is an
 * fp32 sum. Deterministic. x and dx misaligned: MOE_ERR_INVALID_ARG. */
int moe_router_backward(const moe_config_t* cfg, const moe_routes_t* routes, const void* x,
                        const float* w_router, const float* bias, const float* logits,
                        const float* dprob, void* dx, float* dw_router, float* dbias,
                        void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Where moe_route_align leaves the router logits l [N,E] f32 (before the
 * softmax, bias included) inside its workspace; NULL for an invalid config or
 * workspace. Host-side pointer arithmetic only. */
const float* moe_route_workspace_logits(const moe_config_t* cfg, const void* workspace);

/* ---------------------------------------------------------------- graph ladder
 * Captured CUDA graphs of the forward at a ladder of token-count buckets, for
 * batches whose size changes from call to call ("[4/5] feat: capture the FFN
 * experts at bucketed padded shapes", What this adds). A batch of n tokens
 * replays the first bucket >= n, or runs eagerly when n is above the top
 * bucket or that bucket exceeds max_pad_ratio * n; graphs are captured from
 * the top bucket down after one warm-up call at the top size. A bucket's
 * graph is moe_route_align + moe_ffn_forward +
 * moe_combine captured at n_tokens = the bucket with n_valid set, so its
 * replay on n <= bucket tokens computes what those calls compute on exactly n
 * tokens (y bit-identical; the sentinel in sorted_slot_ids is the bucket). */

/* Buffers of one layer instance, every one sized for the top bucket. */
typedef struct moe_layer_buffers {
  const void* x;           /* [Ntop,H] bf16; a forward of n tokens reads x[0..n) */
  const float* w_router;   /* [H,E] f32 */
  const float* bias;       /* [E] f32 or NULL */
  const void* w13;         /* packed, as moe_ffn_forward */
  const void* w2;
  moe_routes_t routes;     /* allocated for the top bucket */
  void* route_workspace;   /* moe_route_workspace_bytes(top) bytes */
  size_t route_workspace_bytes;
  void* h;                 /* [S_top,I] bf16 */
  void* o;                 /* [S_top,H] bf16 */
  void* y;                 /* [Ntop,H] bf16; a forward of n tokens writes y[0..n) */
  int32_t* n_valid;        /* one device int32 the ladder writes the live count to */
} moe_layer_buffers_t;

typedef struct moe_ladder moe_ladder_t; /* opaque */

/* Host-side bucket choice: the index of the smallest bucket >= n, or -1 when
 * n exceeds every bucket or the bucket is more than max_pad_ratio * n
 * (max_pad_ratio <= 0: no limit). buckets ascending. */
int moe_ladder_pick(const int32_t* buckets, int n_buckets, int32_t n, float max_pad_ratio);

/* Captures one graph per bucket (from the top bucket down, after one warm-up
 * forward at the top size on a private stream; synchronises that stream). top: the layer
 * config with n_tokens = buckets[n_buckets-1] and n_valid NULL. The buffers'
 * device memory must stay allocated, and the weights' contents in place, for
 * the ladder's lifetime (the graphs hold their addresses). *out is NULL on
 * failure. */
int moe_ladder_create(const moe_config_t* top, const int32_t* buckets, int n_buckets,
                      float max_pad_ratio, const moe_layer_buffers_t* bufs, moe_ladder_t** out);

/* One forward of n <= Ntop tokens on `stream`: writes n to n_valid and
 * replays the chosen bucket's graph, or runs the three calls eagerly with
 * n_tokens = n. *bucket (optional) receives the bucket index, -1 for eager.
 * One ladder serves one stream at a time. */
int moe_ladder_forward(moe_ladder_t* ladder, int32_t n, cudaStream_t stream, int* bucket);

/* Frees the graphs (not the caller's buffers). */
int moe_ladder_destroy(moe_ladder_t* ladder);

/* Size of the library's built-in route scratch used by moe_route_align_noalloc. */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/* moe_route_align for callers that cannot allocate device memory. No page
 * describes this call; it exists for users of this library. Some callers run
 * where cudaMalloc is unavailable or forbidden: a custom op or plugin inside
 * another runtime that owns every device allocation and hands the plugin no
 * allocator; a latency-bound serving loop that bans allocator calls, because
 * cudaMalloc may synchronise the device and stall every stream; a deployment
 * that fixes its memory budget before the first request. They cannot provide
 * the workspace moe_route_align asks for, so this variant uses an 8 MiB
 * scratch array built into the library instead (every GPU that loads the
 * library holds it until the process exits). Arguments and results are those
 * of moe_route_align, without workspace/ws_bytes.
 *  - Returns MOE_ERR_WORKSPACE, without launching anything, when
 *    moe_route_workspace_bytes(cfg) exceeds MOE_NOALLOC_SCRATCH_BYTES (for
 *    example N*E*4 bytes of logits alone above 8 MiB).
 *  - The first call on each device looks up the scratch array's device
 *    address (with that device current); make that first call before any
 *    stream capture on the device.
 *  - All calls on a device share the one scratch array and it keeps the last
 *    call's contents; nothing in it needs to start at zero, because every
 *    word the kernels read is written earlier in the same call. Calls whose
 *    work overlaps on the GPU (different streams, or different threads without
 *    ordering) race on that array: order them on one stream.
 *  - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call. */
int moe_route_align_noalloc(const moe_config_t* cfg, const void* x, const float* w_router,
                            const float* bias, const moe_routes_t* out, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int status);

/* Number of kernels this library has launched in this process so far. */
uint64_t moe_launch_count(void);

/* Reads and clears the device error word of the current device. Kernels set
 * it (instead of trapping) when a bounded wait runs out. Synchronises the
 * device: call outside of timed regions and outside stream capture.
 * *out receives the word (0 = no error). Returns MOE_OK or MOE_ERR_CUDA. */
int moe_device_error(uint32_t* out);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
