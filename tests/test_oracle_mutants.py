"""Planted mistakes in the oracle, on the CPU.

Each entry below is a plausible error in the oracle -- a wrong rounding rule,
an index or layout mix-up, a dropped term, a wrong sign -- written into a copy
of its source (``oracle/fp8fg_oracle.c`` or ``oracle/mx.py``).  The copy is
built and the oracle's own pins (the ``tests/test_oracle_*.py`` files and the
other CPU tests that fix the oracle to something other than itself) are run
against it in a child process: at least one pin must fail.  This checks the
pins, not the oracle; the committed oracle passes every pin in the rest of the
CPU suite.  Nothing here touches the GPU path.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C_SRC = os.path.join(ROOT, "oracle", "fp8fg_oracle.c")
MX_SRC = os.path.join(ROOT, "oracle", "mx.py")

FORMATS = "tests/test_oracle_formats.py"
QUANT = "tests/test_oracle_quant.py"
GEMM = "tests/test_oracle_gemm.py"
GLUE = "tests/test_oracle_delayed_moe_glue.py"
ADAM = "tests/test_oracle_adam.py"
MX = "tests/test_oracle_mx.py"
MXRULE = "tests/test_mx_exponent_rule.py"
MONITOR = "tests/test_monitor_rules.py"
ALL_PINS = [QUANT, GEMM, GLUE, ADAM, MX, MXRULE, MONITOR, FORMATS]

# name -> (source, [(text, replacement), ...], pin files to try first)
# Every text must occur in the source; all its occurrences are replaced.
MUTANTS = {
    # FP8 encoding (R1) and decoding
    "encode_ties_away_from_zero": ("c", [("n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;   /* tie: even */",
                                          "n = fl + 1.0;   /* tie: even */")], [FORMATS]),
    "encode_overflow_to_nan": ("c", [("if (a >= f.fmax) return sign | f.maxcode;",
                                      "if (a >= f.fmax) return sign | 0x7F;")], [FORMATS]),
    "encode_subnormal_binade_shifted": ("c", [("if (E < f.emin) E = f.emin;              /* subnormal binade */",
                                               "if (E < f.emin - 1) E = f.emin - 1;")], [FORMATS]),
    "decode_exponent_bias_off_by_one": ("c", [("e - f.bias);\n    return sign ? -v : v;",
                                               "e - f.bias + 1);\n    return sign ? -v : v;")], [FORMATS]),
    "decode_e4m3_nan_code_misplaced": ("c", [("if (fmt == ORC_E4M3 && e == 15 && m == 7) return NAN;",
                                              "if (fmt == ORC_E4M3 && e == 15 && m == 6) return NAN;")], [FORMATS]),
    "bf16_rounding_ties_toward_zero": ("c", [("else n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;\n    val = n * quantum;\n    if (val >= ldexp(1.0, 128))",
                                              "else n = fl;\n    val = n * quantum;\n    if (val >= ldexp(1.0, 128))")],
                                       [FORMATS]),
    "decode_subnormal_spacing_halved": ("c", [("v = ldexp((double)m, f.emin - f.mbits);",
                                               "v = ldexp((double)m, f.emin - f.mbits - 1);")], [FORMATS]),
    "bf16_subnormals_flushed": ("c", [("memcpy(&f, &u, sizeof f);\n    return f;",
                                       "memcpy(&f, &u, sizeof f);\n    return (b & 0x7F80) == 0 ? 0.0f : f;")],
                                [FORMATS]),
    "nonfinite_inputs_not_reported": ("c", [("if (!isfinite(v)) bad = 1;", "if (0) bad = 1;")], [QUANT, GLUE]),
    # scale and quotient (R2, R3: s = fp32(amax / fmax), q = enc(fp32(x / s)))
    "scale_by_reciprocal_of_fmax": ("c", [("return amax / fm;", "return amax * (1.0f / fm);")], [QUANT]),
    "scale_of_zero_group_is_zero": ("c", [("if (amax == 0.0f) return 1.0f;", "if (amax == 0.0f) return 0.0f;")],
                                    [QUANT]),
    "quotient_by_reciprocal": ("c", [("float quotient = x / s;\n    return orc_fp8_encode",
                                      "float quotient = x * (1.0f / s);\n    return orc_fp8_encode")], [QUANT]),
    # tile layouts
    "1x128_scales_row_major": ("c", [("s[cb * rows + r] = sc;", "s[r * (cols / 128) + cb] = sc;")], [QUANT]),
    "128x1_scales_column_major": ("c", [("sT[mb * cols + c] = sc;", "sT[c * (rows / 128) + mb] = sc;")], [QUANT]),
    "128x128_amax_of_first_row_only": ("c", [("        for (i = 0; i < 128; ++i)\n            for (j = 0; j < 128; ++j) {\n"
                                              "                float v = orc_bf16_to_f32(w[",
                                              "        for (i = 0; i < 1; ++i)\n            for (j = 0; j < 128; ++j) {\n"
                                              "                float v = orc_bf16_to_f32(w[")], [QUANT]),
    "128x1_codes_not_transposed": ("c", [("qT[c * rows + mb * 128 + i] =", "qT[(mb * 128 + i) * cols + c] =")],
                                   [QUANT]),
    "128x1_amax_of_a_row_block": ("c", [("float v = orc_bf16_to_f32(x[(mb * 128 + i) * ldx + c]);\n                if",
                                         "float v = orc_bf16_to_f32(x[(mb * 128 + (i & 1)) * ldx + c]);\n                if")],
                                  [QUANT]),
    "pertensor_current_scale_of_zero_is_zero": ("c", [("    sc = scale_of(amax, fmt);\n#pragma omp parallel for schedule(static)\n"
                                                       "    for (r = 0; r < rows; ++r) {\n        int64_t c;\n"
                                                       "        for (c = 0; c < cols; ++c) q[r * cols + c]",
                                                       "    sc = amax / (float)fmt_of(fmt).fmax;\n#pragma omp parallel for schedule(static)\n"
                                                       "    for (r = 0; r < rows; ++r) {\n        int64_t c;\n"
                                                       "        for (c = 0; c < cols; ++c) q[r * cols + c]")], [QUANT]),
    # monitors (R6)
    "distinct_counts_signed_zeros_twice": ("c", [("static uint32_t key_bf16(uint16_t b) { return (b & 0x7FFF) == 0 ? 0u : (uint32_t)b; }",
                                                  "static uint32_t key_bf16(uint16_t b) { return (uint32_t)b; }")],
                                           [QUANT, MONITOR, GLUE]),
    "underflow_misses_negative_zero_codes": ("c", [("if ((qc & 0x7F) == 0) uf++;", "if (qc == 0) uf++;")],
                                             [QUANT, MONITOR, GLUE]),
    "saturation_counts_exact_fmax": ("c", [("if (fabsf(quotient) > fm) sat++;", "if (fabsf(quotient) >= fm) sat++;")],
                                     [QUANT, MONITOR, GLUE]),
    "pertensor_monitor_counts_signed_zeros_twice": ("c", [("px[key_bf16(xb)] = 1;", "px[xb] = 1;")],
                                                    [GLUE, QUANT, MONITOR]),
    "128x1_monitor_scale_grid_transposed": ("c", [("case ORC_GRAN_128x1: sc = s[grow * cols + gcol]; break;",
                                                   "case ORC_GRAN_128x1: sc = s[gcol * (rows / 128) + grow]; break;")],
                                            [QUANT, MONITOR]),
    "128x1_monitor_reads_codes_untransposed": ("c", [("uint8_t qc = (gran == ORC_GRAN_128x1) ? q[c * rows + r] : q[r * cols + c];",
                                                      "uint8_t qc = q[r * cols + c];")], [QUANT, MONITOR]),
    # delayed scaling (R5)
    "history_slot_one_ahead": ("c", [("hist[*step % hist_len] = amax;", "hist[(*step + 1) % hist_len] = amax;")],
                               [GLUE]),
    "margin_with_wrong_sign": ("c", [("*scale = ldexpf(m, margin)", "*scale = ldexpf(m, -margin)")], [GLUE]),
    "most_recent_ignored": ("c", [("if (algo == ORC_ALGO_MOST_RECENT) {", "if (algo == -1) {")], [GLUE]),
    "nonfinite_step_still_updates_history": ("c", [("    if (bad) return ORC_NONFINITE;\n    /* 2. record",
                                                    "    /* 2. record")], [GLUE]),
    "scale_updated_from_an_empty_history": ("c", [("if (m > 0.0f) *scale = ldexpf(m, margin)",
                                                   "*scale = ldexpf(m, margin)")], [GLUE]),
    # GEMM (R7)
    "gemm_drops_b_scale": ("c", [("d += (double)scale_at(sA, granA, ldsA, m, kb) * (double)scale_at(sB, granB, ldsB, n, kb) * p;",
                                  "d += (double)scale_at(sA, granA, ldsA, m, kb) * p;")], [GEMM]),
    "gemm_128x128_scale_grid_transposed": ("c", [("case ORC_GRAN_128x128: return sv[(row / 128) * ld + kb];",
                                                  "case ORC_GRAN_128x128: return sv[kb * ld + row / 128];")], [GEMM]),
    "gemm_scales_of_the_next_chunk": ("c", [("d += (double)scale_at(sA, granA, ldsA, m, kb)",
                                             "d += (double)scale_at(sA, granA, ldsA, m, (kb + 1) % (K / 128))")], [GEMM]),
    "pertensor_gemm_drops_b_scale": ("c", [("return (double)sA[0] * (double)sB[0] * p;", "return (double)sA[0] * p;")],
                                     [GEMM]),
    "grouped_gemm_weights_of_expert_zero": ("c", [("B + ((int64_t)g * N + n) * K", "B + ((int64_t)n) * K")],
                                            [GEMM]),
    "grouped_gemm_expert_bound_inclusive": ("c", [("if (m >= off[e] && m < off[e + 1]) { g = e; break; }",
                                                   "if (m >= off[e] && m <= off[e + 1]) { g = e; break; }")], [GEMM]),
    "grouped_wgrad_scales_from_chunk_zero": ("c", [("sA + (r0 / 128) * N", "sA")], [GEMM]),
    "recompute_error_signed_max": ("c", [("if (fabs(d) > mdd) mdd = fabs(d);", "if (d > mdd) mdd = d;")], [GEMM]),
    "recompute_error_reference_norm_unsquared": ("c", [("srr += r * r;", "srr += fabs(r);")], [GEMM]),
    # AdamW with FP8 moments (R12)
    "adam_without_bias_correction": ("c", [("mh = m / bc1;", "mh = m;")], [ADAM]),
    "adam_eps_inside_sqrt": ("c", [("den = sqrtf(vh) + eps;", "den = sqrtf(vh + eps);")], [ADAM]),
    "adam_weight_decay_on_gradient": ("c", [("t = wd * p[k];", "t = wd * gi;")], [ADAM]),
    "adam_second_moment_of_g_not_g_squared": ("c", [("v = b2 * v + omb2 * gg;", "v = b2 * v + omb2 * gi;")], [ADAM]),
    "adam_v_scaled_with_e4m3_max": ("c", [("s_v = av == 0.0f ? 1.0f : av / 57344.0f;",
                                           "s_v = av == 0.0f ? 1.0f : av / 448.0f;")], [ADAM]),
    "adam_v_encoded_as_e4m3": ("c", [("qv[blk * 128 + i] = orc_fp8_encode(vn[i] / s_v, ORC_E5M2);",
                                      "qv[blk * 128 + i] = orc_fp8_encode(vn[i] / s_v, ORC_E4M3);")], [ADAM]),
    "adam_momentum_without_one_minus_beta": ("c", [("m = b1 * m + omb1 * gi;", "m = b1 * m + gi;")], [ADAM]),
    "adam_update_with_wrong_sign": ("c", [("p[k] = p[k] - t;", "p[k] = p[k] + t;")], [ADAM]),
    "adam_m_scaled_with_e5m2_max": ("c", [("s_m = am == 0.0f ? 1.0f : am / 448.0f;",
                                           "s_m = am == 0.0f ? 1.0f : am / 57344.0f;")], [ADAM]),
    # routing, gather, SwiGLU (R8, R9)
    "route_ties_to_higher_index": ("c", [("if (best < 0 || z[e] > z[best]) best = e;",
                                          "if (best < 0 || z[e] >= z[best]) best = e;")], [GLUE]),
    "route_pads_aligned_experts_too": ("c", [("padded[e] = (int32_t)(((c + align - 1) / align) * align);",
                                              "padded[e] = (int32_t)((c / align + 1) * align);")], [GLUE]),
    "route_probabilities_unnormalised": ("c", [("prob[t * E + e] /= sum;", "prob[t * E + e] /= 1.0;")], [GLUE]),
    "gather_scales_by_row_not_token": ("c", [("sg[kb * cap + r] = s[kb * T + row_token[r]];",
                                              "sg[kb * cap + r] = s[kb * T + r];")], [GLUE]),
    "swiglu_sigmoid_sign_flipped": ("c", [("double sig = 1.0 / (1.0 + exp(-g));\n            h[r * F + j]",
                                           "double sig = 1.0 / (1.0 + exp(g));\n            h[r * F + j]")], [GLUE]),
    "swiglu_grad_drops_sigmoid_derivative": ("c", [("d * u * sig * (1.0 + g * (1.0 - sig))", "d * u * sig")], [GLUE]),
    "route_topk_prob_of_slot_not_expert": ("c", [("topk_prob[t * topk + k] = prob[t * E + best];",
                                                  "topk_prob[t * topk + k] = prob[t * E + k];")], [GLUE]),
    "route_padding_rows_keep_a_probability": ("c", [("row_prob[r] = routed[t * E + e] ? prob[t * E + e] : 0.0;",
                                                     "row_prob[r] = prob[t * E + e];")], [GLUE]),
    "swiglu_forward_drops_gate": ("c", [("h[r * F + j] = orc_f64_to_bf16(g * sig * u);",
                                         "h[r * F + j] = orc_f64_to_bf16(sig * u);")], [GLUE]),
    "swiglu_up_grad_drops_gate": ("c", [("orc_f64_to_bf16(d * g * sig);", "orc_f64_to_bf16(d * sig);")], [GLUE]),
    "route_pads_with_the_last_free_tokens": ("c", [("for (t = 0; t < T && need > 0; ++t)",
                                                    "for (t = T - 1; t >= 0 && need > 0; --t)")], [GLUE]),
    "route_offsets_from_unpadded_counts": ("c", [("offsets[e + 1] = offsets[e] + padded[e];",
                                                  "offsets[e + 1] = offsets[e] + counts[e];")], [GLUE]),
    "swiglu_grad_sigmoid_sign_flipped": ("c", [("double sig = 1.0 / (1.0 + exp(-g));\n            dgu[",
                                                "double sig = 1.0 / (1.0 + exp(g));\n            dgu[")], [GLUE]),
    # MXFP8 (R13-R16)
    "mx_untile_order_swapped": ("mx", [("t.transpose(1, 3, 2, 0, 4)", "t.transpose(1, 2, 3, 0, 4)")], [MX]),
    "mx_quotient_multiplies_by_the_scale": ("mx", [("quot = xb / np.ldexp(1.0, e)[..., None]",
                                                    "quot = xb * np.ldexp(1.0, e)[..., None]")], [MX, MXRULE]),
    "mx_floor_exponent_rule": ("mx", [("e = np.ceil(np.log2(", "e = np.floor(np.log2("),
                                      ("    e = e + (np.ldexp(fm, e) < a)\n", "")], [MXRULE, MX]),
    "mx_scale_code_bias_off_by_one": ("mx", [("(e + E8_BIAS).astype(np.uint8), OK",
                                              "(e + E8_BIAS + 1).astype(np.uint8), OK")], [MX, MXRULE]),
    "mx_zero_block_smallest_scale": ("mx", [("e = np.where(pos, e, 0)", "e = np.where(pos, e, -E8_BIAS)")],
                                     [MX, MXRULE]),
    "mx_exponent_clamped_one_short": ("mx", [("return np.clip(e, -E8_BIAS, E8_BIAS)", "return np.clip(e, -E8_BIAS, E8_BIAS - 1)")],
                                      [MXRULE, MX]),
    "mx_blocks_strided_not_contiguous": ("mx", [("xb = x.reshape(R, C // MX_BLOCK, MX_BLOCK)",
                                                 "xb = x.reshape(R, MX_BLOCK, C // MX_BLOCK).transpose(0, 2, 1)")],
                                         [MX, MXRULE]),
    "mx_gemm_drops_b_scale": ("mx", [("np.ldexp(part, eA[m] + eB[n] - 2 * E8_BIAS)", "np.ldexp(part, eA[m] - E8_BIAS)")],
                              [MX]),
    "mx_dequant_exponent_negated": ("mx", [("np.ldexp(1.0, e8.astype(np.int64) - E8_BIAS)",
                                            "np.ldexp(1.0, E8_BIAS - e8.astype(np.int64))")], [MX]),
    "mx_tile_rows_order_swapped": ("mx", [("t.transpose(3, 0, 2, 1, 4)", "t.transpose(3, 0, 1, 2, 4)")], [MX]),
}

# Runs the pins with the oracle routed through a planted copy.
_DRIVER = r"""
import importlib.util, sys
root, so, mxsrc, *files = sys.argv[1:]
sys.path.insert(0, root)
import oracle
if so:
    oracle.use_library(so)
if mxsrc:
    spec = importlib.util.spec_from_file_location("oracle.mx", mxsrc)
    mod = importlib.util.module_from_spec(spec)
    sys.modules["oracle.mx"] = mod
    spec.loader.exec_module(mod)
    oracle.mx = mod
import pytest
sys.exit(pytest.main(["-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider", *files]))
"""


def _plant(src_path: str, edits) -> str:
    text = open(src_path).read()
    for old, new in edits:
        assert old in text, f"planted edit no longer matches the oracle source: {old[:60]!r}"
        text = text.replace(old, new)
    return text


def _run_one(name: str, workdir: str):
    kind, edits, first = MUTANTS[name]
    so = mxsrc = ""
    if kind == "c":
        src = os.path.join(workdir, f"{name}.c")
        with open(src, "w") as f:
            f.write(_plant(C_SRC, edits))
        so = os.path.join(workdir, f"lib{name}.so")
        subprocess.run(["gcc", "-std=c11", "-O1", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                        "-shared", "-w", "-o", so, src, "-lm"], check=True)
    else:
        mxsrc = os.path.join(workdir, f"{name}_mx.py")
        with open(mxsrc, "w") as f:
            f.write(_plant(MX_SRC, edits))
    files = first + [p for p in ALL_PINS if p not in first]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run([sys.executable, "-c", _DRIVER, ROOT, so, mxsrc, *files], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    return p.returncode, p.stdout[-2000:] + p.stderr[-2000:]


@pytest.fixture(scope="module")
def planted_results(tmp_path_factory):
    work = str(tmp_path_factory.mktemp("planted"))
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {n: ex.submit(_run_one, n, work) for n in MUTANTS}
        return {n: f.result() for n, f in futs.items()}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, planted_results):
    rc, tail = planted_results[name]
    # pytest exit code 1: tests ran and at least one failed (not a crash or a
    # collection error, which would say nothing about the pins)
    assert rc == 1 and " failed" in tail, f"{name}: no pin caught it (exit {rc})\n{tail}"
