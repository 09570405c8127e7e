"""The pins catch plausible mistakes: each case plants one mistake in a
temporary copy of the oracle's C source, builds it, and requires that a pin
fails against it. (Mistakes are planted in the oracle, on the CPU.)"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import test_oracle_backward_pins as bp
import test_oracle_pins as fp
import test_oracle_fp8_pins as fx
import test_oracle_mx_pins as mx
import test_oracle_router_backward_pins as rb

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTATIONS = [
    ("top-K ties to the higher expert", "p[e] > p[best]) best = e;", "p[e] >= p[best]) best = e;",
     lambda: fp.test_router_hand_worked_cases()),
    ("capacity rounded down", "return (num + den - 1) / den;", "return num / den;",
     lambda: fp.test_capacity_worked_values()),
    ("selection ignores the probability", "if (x->p > y->p) return -1;\n  if (x->p < y->p) return 1;",
     "", lambda: [fp.test_selection_matches_brute_force_rank(s) for s in range(6)]),
    ("kept tokens laid out in probability order",
     "    qsort(buf, (size_t)kept, sizeof(route_key), cmp_token_asc); /* kept ones in ascending t */\n",
     "", lambda: fp.test_layout_hand_worked("layout_prob_k2.txt")),
    ("silu without its gate factor", "return v / (1.0f + expf(-v));",
     "return 1.0f / (1.0f + expf(-v));",
     lambda: fp.test_single_expert_top1_is_plain_swiglu_mlp()),
    ("renormalisation skipped", "topk_p[(size_t)t * K + k] = topk_p[(size_t)t * K + k] / d;",
     "topk_p[(size_t)t * K + k] = topk_p[(size_t)t * K + k];",
     lambda: fp.test_router_matches_fp64_library_routines(37, 64, 8, 2, False)),
    ("SwiGLU backward loses the derivative term", "(1.0f + v * (1.0f - sg))", "(1.0f)",
     lambda: bp.test_backward_matches_central_differences(0)),
    ("dprob taken from the weighted gradient", "dp = dp + a * da0[i];", "dp = dp + a * p * da0[i];",
     lambda: bp.test_backward_matches_central_differences(1)),
    ("dW_down without the routing weight", "if (aw_out) aw_out[i] = p * a;",
     "if (aw_out) aw_out[i] = a;", lambda: bp.test_weight_gradients_match_fp64_closed_form()),
    ("dropless extent ignores the ladder", "    if (count <= rung) return rung;", "",
     lambda: bp.test_dropless_layout_hand_worked()),
    ("GELU backward without the density term", "return cdf + v * pdf;", "return cdf;",
     lambda: bp.test_backward_matches_central_differences_gelu(0)),
    ("GELU with the erf argument unscaled", "erff(v * 0.70710678118654752f));\n  return v",
     "erff(v));\n  return v", lambda: fp.test_gelu_closed_form_values()),
    ("E4M3 ties rounded away from the even code", "(dc == db && (lo & 1) == 0)", "(dc == db)",
     lambda: [fx.test_e4m3_encode_rounding(v, c) for v, c in ((1.0625, 0x38), (1.1875, 0x3A))]),
    ("E4M3 subnormals with the normal exponent bias", "ldexpf((float)m, -9)", "ldexpf((float)m, -10)",
     lambda: fx.test_e4m3_decode_table(0x01, 2.0 ** -9)),
    ("FP8 FC2 scales the weight row by the expert's first row", "(oracle_e4m3_decode(wr[i]) * ws[r]);",
     "(oracle_e4m3_decode(wr[i]) * ws[(size_t)e * H]);",
     lambda: fx.test_fc2_fp8_matches_fp64_dequantised_reference()),
    ("FP8 FC1 scales the up row by the gate row's scale", "u = u + xv * (oracle_e4m3_decode(wu[h]) * ws[ru]);",
     "u = u + xv * (oracle_e4m3_decode(wu[h]) * ws[rg]);",
     lambda: fx.test_fc1_fp8_matches_fp64_dequantised_reference(0)),
    ("router backward skips the renormalisation term", "gk[k] = (dp[k] - c) / d;",
     "gk[k] = dp[k] / d;", lambda: rb.test_router_backward_matches_central_differences(0, True)),
    ("router backward skips the softmax normaliser", "dl[ids[k]] = p[ids[k]] * (gk[k] - s);",
     "dl[ids[k]] = p[ids[k]] * gk[k];", lambda: rb.test_router_backward_matches_central_differences(1, False)),
    ("MX block exponent with the wrong element emax", "int s = (e - 1) - 8;", "int s = (e - 1) - 7;",
     lambda: mx.test_block_scale_exponent_worked_values(1.0, 119)),
    ("E8M0 decoded with bias 128", "return ldexpf(1.0f, (int)c - 127);", "return ldexpf(1.0f, (int)c - 128);",
     lambda: mx.test_e8m0_decode(127, 1.0)),
    ("MX FC1 gate weight scaled by its first block", "oracle_e8m0_decode(ws[rg * nb + b])",
     "oracle_e8m0_decode(ws[rg * nb])", lambda: mx.test_fc1_mx_matches_fp64_dequantised_reference(0)),
    ("MX FC2 h scaled by its first block", "oracle_e8m0_decode(hsr[b])", "oracle_e8m0_decode(hsr[0])",
     lambda: mx.test_fc2_mx_matches_fp64_dequantised_reference()),
    ("exp's sixth-order coefficient off", "p = fmaf(p, r, (float)(1.0 / 720.0));",
     "p = fmaf(p, r, (float)(1.0 / 700.0));", lambda: fp.test_exp_is_the_stated_method_step_by_step()),
    ("exp reduction without the low part of ln 2", "  r = fmaf(-n, ln2_lo, r);\n", "",
     lambda: fp.test_exp_is_the_stated_method_step_by_step()),
    ("softmax without the max subtraction", "p[e] = oracle_exp(l[e] - m);", "p[e] = oracle_exp(l[e]);",
     lambda: fp.test_router_is_the_exact_fp32_chain()),
    ("router logits with a rounded product before each add",
     "acc = fmaf(bf16_to_f32(x[(size_t)t * H + h]), wr[(size_t)h * E + e], acc);",
     "acc = acc + bf16_to_f32(x[(size_t)t * H + h]) * wr[(size_t)h * E + e];",
     lambda: fp.test_router_is_the_exact_fp32_chain()),
    ("router logits summed over descending h",
     "for (int h = 0; h < H; ++h) acc = fmaf(bf16_to_f32(x",
     "for (int h = H - 1; h >= 0; --h) acc = fmaf(bf16_to_f32(x",
     lambda: fp.test_router_is_the_exact_fp32_chain()),
    ("router bias added before the chain", "      float acc = 0.0f;\n      for (int h = 0; h < H; ++h) acc = fmaf(",
     "      float acc = bias ? bias[e] : 0.0f;\n      for (int h = 0; h < H; ++h) acc = fmaf(",
     lambda: fp.test_router_is_the_exact_fp32_chain()),
    ("router dx with the weight transposed", "acc = acc + dlogits[(size_t)t * E + e] * wr[(size_t)h * E + e];",
     "acc = acc + dlogits[(size_t)t * E + e] * wr[(size_t)e * H + h];",
     lambda: rb.test_router_backward_matches_central_differences(2, True)),
]


@pytest.mark.parametrize("name,old,new,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_fails_on_planted_mistake(name, old, new, pin, monkeypatch):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site must be unique: " + name
    tmp = tempfile.mkdtemp(prefix="oracle_mut_")
    try:
        c = os.path.join(tmp, "moe_oracle.c")
        so = os.path.join(tmp, "liboracle.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fopenmp",
                        "-fPIC", "-shared", c, "-o", so, "-lm"], check=True)
        monkeypatch.setattr(oracle, "_SRC", c)
        monkeypatch.setattr(oracle, "_LIB", so)
        monkeypatch.setattr(oracle, "_lib", None)
        with pytest.raises(AssertionError):
            pin()
    finally:
        oracle._lib = None
        shutil.rmtree(tmp, ignore_errors=True)
