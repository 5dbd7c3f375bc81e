"""Plant plausible mistakes in copies of the oracle and check that the pins catch each one.

Every mutant is a textual patch of oracle/moe_oracle.c compiled into a temporary library; the
real oracle is never modified. A mutant that no pin rejects would mean the pins are too weak.
"""

import os

import pytest

import oracle
import oracle_bwd_pins
import oracle_mx_pins
import oracle_nvfp4_pins
import oracle_pins

MUTANTS = {
    "gate_up_swapped": [
        ("wg = job->w13 + ((size_t)e * 2 + 0)", "wg = job->w13 + ((size_t)e * 2 + 1)"),
        ("wu = job->w13 + ((size_t)e * 2 + 1)", "wu = job->w13 + ((size_t)e * 2 + 0)"),
    ],
    "score_dropped": [("acc[j] += s * y;", "acc[j] += y;")],
    "silu_sign": [("expf(-g)", "expf(g)")],
    "silu_wrong_slope": [("1.0f + expf(-g)", "1.0f + expf(-2.0f * g)")],
    "w2_transposed": [("w2e[(size_t)j * F + f]", "w2e[(size_t)f * D + j]")],
    "gate_transposed": [("wg[(size_t)f * D + d]", "wg[(size_t)d * F + f]")],
    "last_k_dropped": [("for (int32_t k = 0; k < K; ++k)", "for (int32_t k = 0; k + 1 < K; ++k)")],
    "wrong_token_row": [("job->x[t * D + d]", "job->x[((t + 1) % job->t_end) * D + d]")],
    "up_not_multiplied": [("h[f] = silu * u;", "h[f] = silu;")],
    "offsets_not_prefix": [("offsets[e + 1] = offsets[e] + counts[e];", "offsets[e + 1] = counts[e];")],
    "unstable_order": [
        ("    for (int64_t i = 0; i < R; ++i) {\n        int32_t e = ids[i];\n        int32_t key",
         "    for (int64_t i = R - 1; i >= 0; --i) {\n        int32_t e = ids[i];\n        int32_t key"),
    ],
    "invalid_ids_kept": [("int32_t key = (e >= 0 && e < E) ? e : E;", "int32_t key = (e >= 0 && e < E) ? e : 0;")],
    "inv_identity": [("inv[i] = (int32_t)r;", "inv[i] = (int32_t)i;")],
    "round_h_truncates": [("u += 0x7fffu + ((u >> 16) & 1u);", "u += 0u;")],
    # route-wise RMSNorm post-processing
    "rms_sum_not_mean": [("const float rstd = 1.0f / sqrtf(ss / (float)D + job->rms_eps);",
                          "const float rstd = 1.0f / sqrtf(ss + job->rms_eps);")],
    "rms_score_dropped": [("for (int32_t j = 0; j < D; ++j) acc[j] += s * (xt_y[j] * rstd);",
                           "for (int32_t j = 0; j < D; ++j) acc[j] += (xt_y[j] * rstd);")],
    # backward
    "bwd_silu_grad_sign": [("return sig * (1.0f + g * (1.0f - sig));", "return sig * (1.0f - g * (1.0f - sig));")],
    "bwd_dh_without_score": [("const float dh = s * w2t[f];", "const float dh = w2t[f];")],
    "bwd_dw2_without_score": [("const float dy = s * dout_t[j];", "const float dy = dout_t[j];")],
    "bwd_dx_without_up_term": [(" + bf16_to_f32(wu[(size_t)f * D + d]) * du[f];", ";")],
    "bwd_dscore_scaled": [("ds += w2t[f] * h[f];", "ds += w2t[f] * h[f] * s;")],
    "bwd_du_from_gate": [("du[f] = dh * a[f];", "du[f] = dh * g[f];")],
    "bwd_dwu_from_dg": [("dwu[(size_t)f * D + d] += du[f] * xt[d];", "dwu[(size_t)f * D + d] += dg[f] * xt[d];")],
    # MXFP8: the MX format and the block-scaled forward
    "mx_scale_off_by_one": [("int e = (ex - 1) - 8;", "int e = ex - 8;")],
    "mx_emax_of_e5m2": [("int e = (ex - 1) - 8;", "int e = (ex - 1) - 15;")],
    "mx_no_saturation": [("if (r > 448.0) r = 448.0;", "")],
    "mx_ties_away_from_zero": [("nearbyint(ldexp(a, 3 - k))", "round(ldexp(a, 3 - k))")],
    "mx_amax_over_half_block": [("for (int i = 0; i < 32; ++i)\n        if (fabs((double)v[i]) > amax)",
                                 "for (int i = 0; i < 16; ++i)\n        if (fabs((double)v[i]) > amax)")],
    "mx_zero_loses_sign": [("if (r == 0) return sign;", "if (r == 0) return 0;")],
    "mx_no_subnormals": [("const int k = (a > 0 && ex - 1 > -6) ? ex - 1 : -6;",
                          "const int k = (a > 0) ? ex - 1 : -6;")],
    "mx_e4m3_bias": [("ldexp((double)(8 + man), ex - 10)", "ldexp((double)(8 + man), ex - 11)")],
    "mx_scale_sign": [("ldexp(value[codes[b * 32 + i]], e)", "ldexp(value[codes[b * 32 + i]], -e)")],
    "mx_h_not_quantized": [("mx_dequantize_row(value, q, qs, F, hd);", "memcpy(hd, h, sizeof(float) * (size_t)F);")],
    "mx_x_not_quantized": [("g += wg[d] * xd[d];\n                    u += wu[d] * xd[d];",
                            "g += wg[d] * xt[d];\n                    u += wu[d] * xt[d];")],
    "mx_gate_uses_up_scales": [("job->w13s + grow * (size_t)(D / 32)", "job->w13s + urow * (size_t)(D / 32)")],
    # NVFP4: the two-level format and the block-scaled forward
    "nv_scale_over_4": [("const float t = 6.0f * G;", "const float t = 4.0f * G;")],
    "nv_ties_away_from_zero": [("double r = nearbyint(a / step) * step;", "double r = round(a / step) * step;")],
    "nv_no_saturation": [("if (r > 6.0) r = 6.0;", "")],
    "nv_zero_scale_unguarded": [("    if (S == 0.0f) {\n        for (int i = 0; i < 16; ++i) codes[i] = 0;\n        return;\n    }\n", "")],
    "nv_tensor_scale_not_applied": [("out[b * 16 + i] = (float)(e2m1_value(codes[b * 16 + i]) * S) * G;",
                                     "out[b * 16 + i] = (float)(e2m1_value(codes[b * 16 + i]) * S);")],
    "nv_weight_scale_448": [("return amax > 0.0f ? amax / 2688.0f : 1.0f;", "return amax > 0.0f ? amax / 448.0f : 1.0f;")],
    "nv_h_not_quantized": [("nvfp4_dequantize_row(q, qs, nj->gh, F, hd);", "memcpy(hd, h, sizeof(float) * (size_t)F);")],
    "nv_x_scale_dropped": [("nvfp4_dequantize_row(q, qs, nj->gx, D, xd);", "nvfp4_dequantize_row(q, qs, 1.0f, D, xd);")],
    "nv_scales_per_32": [("const float S = (float)e4m3_value(scales[b]);", "const float S = (float)e4m3_value(scales[b / 2]);")],
    "nv_sign_lost": [("const uint8_t sign = signbit(v) ? 8 : 0;", "const uint8_t sign = 0;")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    with open(oracle.SOURCE) as fh:
        src = fh.read()
    for old, new in MUTANTS[name]:
        assert src.count(old) >= 1, f"patch anchor not found: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    lib_path = str(tmp_path / "libmutant.so")
    oracle.compile_oracle(str(path), lib_path)
    lib = oracle.load_library(lib_path)
    failed = []
    for check in oracle_pins.ALL_PINS + oracle_bwd_pins.BWD_PINS + oracle_mx_pins.MX_PINS + oracle_nvfp4_pins.NV_PINS:
        try:
            check(lib=lib)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin rejects mutant {name}"
