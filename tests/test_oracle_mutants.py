"""Planted mistakes in the oracle, on the CPU: the pins must notice each of them.

Every mutant is a copy of the C oracle with one plausible error (a tie sent the
wrong way, a sign rule, a wrong divisor or exponent bias, a dropped floor,
factor or term, a wrong or transposed index, a reversed packing order),
compiled on the side and loaded in place of the real oracle; the pins of
tests/test_oracle_pins.py that guard that step must fail on it. A control run
of the unmodified copy through the same machinery passes them all, so the
failures come from the planted mistakes.

Each mutation keeps every memory access of the oracle within its buffers. The
mutants run in one spawned child process, so that the real oracle loaded by the
other tests is never replaced in this process.

Mutations that cannot change any result are left out on purpose: reading the
two FP4 nibbles of a byte in the other order inside the GEMM references alone
permutes k identically for both operands within one scale block, which leaves
every GEMM result unchanged; the quantizers' leading dimension is always the
column count (the wrapper passes contiguous arrays); an INT4 clamp of -7
instead of -8 never binds, since |w / s| <= 7 (1 + 2^-8) with s = bf16(amax / 7);
and in the K-per-channel zero-point function, the amax of the centred residual
is reached at both ends of the channel's range, so leaving one extreme out of
that amax changes nothing beyond a rounding of the midpoint.
"""
import multiprocessing as mp
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_W4A16_TAIL = "        }\n        y[p] = acc;\n        bound[p] = mag;\n    }\n}\n\n/* FP8 block"

# name: (text in qz_oracle.c, replacement, pins expected to notice it)
MUTANTS = {
    "e4m3_ties_to_odd": ("(d == bestd && (c & 1) == 0 && (best & 1) == 1)",
                         "(d == bestd && (c & 1) == 1 && (best & 1) == 0)",
                         ["test_e4m3_encode_matches_torch_cast"]),
    "e4m3_subnormal_exponent": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)",
                                ["test_e4m3_format_facts", "test_e4m3_encode_matches_torch_cast"]),
    "e2m1_ties_up": ("if (d < bestd) { bestd = d; best = i; }", "if (d <= bestd) { bestd = d; best = i; }",
                     ["test_e2m1_ties_go_to_smaller_magnitude", "test_e2m1_matches_torch_argmin_pipeline"]),
    "e2m1_sign_from_signbit": ("if (y < 0.0f) best |= 8;", "if (signbit(y)) best |= 8;",
                               ["test_e2m1_sign_of_zero"]),
    "e2m1_grid_value": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0}",
                        ["test_e2m1_format_facts", "test_e2m1_matches_torch_argmin_pipeline"]),
    "bf16_ties_down": ("if (dlo < dhi) return lo;", "if (dlo <= dhi) return lo;",
                       ["test_bf16_matches_torch_cast"]),
    "fp8_scale_divisor": ("(amax > or_amax_min() ? amax : or_amax_min()) / OR_FP8_MAX;",
                          "(amax > or_amax_min() ? amax : or_amax_min()) / 447.0f;",
                          ["test_fp8_invariants", "test_fp8_unit_scale_reduces_to_plain_cast"]),
    "fp8_no_clamp_floor": ("float scale = (amax > or_amax_min() ? amax : or_amax_min()) / OR_FP8_MAX;",
                           "float scale = amax / OR_FP8_MAX;",
                           ["test_fp8_all_zero_tensor_uses_clamp_floor"]),
    "fp8_block_rows_always_128": ("case OR_BLOCK128: ur = rows < 128 ? rows : 128;", "case OR_BLOCK128: ur = 128;",
                                  ["test_fp8_block_extent_is_min_128_rows", "test_fp8_block_over_one_row_equals_group"]),
    "mx_exponent_off_by_one": ("int E = or_floor_log2(amax) - 2;", "int E = or_floor_log2(amax) - 1;",
                               ["test_mxfp4_invariants", "test_mxfp4_exponent_is_exact_below_power_of_two"]),
    "mx_e8m0_bias": ("(uint8_t)(E + 127)", "(uint8_t)(E + 128)",
                     ["test_mxfp4_invariants", "test_mxfp4_exponent_is_exact_below_power_of_two"]),
    "mx_block_amax_over_16": ("for (int64_t c = b * 32; c < b * 32 + 32; c++) {\n                float a",
                              "for (int64_t c = b * 32; c < b * 32 + 16; c++) {\n                float a",
                              ["test_mxfp4_invariants"]),
    "nv_global_divisor": ("/ (OR_FP8_MAX * OR_FP4_MAX);", "/ OR_FP8_MAX;", ["test_nvfp4_invariants"]),
    "nv_block_scale_no_floor": ("float s = (bv > or_amax_min() ? bv : or_amax_min()) * g;", "float s = bv * g;",
                                ["test_nvfp4_block_scale_rounding_to_zero_keeps_codes_of_page"]),
    "nv_block_amax_over_4": ("float t = bamax / OR_FP4_MAX / g;", "float t = bamax / 4.0f / g;",
                             ["test_nvfp4_invariants"]),
    "nv_tensor_amax_skips_last_row": (
        "    float amax = 0.0f;\n    for (int64_t r = 0; r < rows; r++)\n        for (int64_t c = 0; c < cols; c++) {",
        "    float amax = 0.0f;\n    for (int64_t r = 0; r < rows - 1; r++)\n        for (int64_t c = 0; c < cols; c++) {",
        ["test_nvfp4_invariants", "test_nvfp4_block_scale_rounding_to_zero_keeps_codes_of_page"]),
    "int4_divisor_8": ("/ 7.0f;", "/ 8.0f;", ["test_int4_g128_invariants"]),
    "int_round_half_away": ("float r = rintf(y);", "float r = roundf(y);",
                            ["test_int_quant_round_half_even_and_clip"]),
    "int4_pack_reversed": ("<< (4 * (k % 8));", "<< (4 * (7 - k % 8));",
                           ["test_int4_g128_invariants", "test_gemm_scale_indexing_matches_quantizer_dequant"]),
    "int4_scale_not_bf16": ("float s = or_bf16_to_f32(sbits);", "float s = sf;",
                            ["test_int4_g128_invariants"]),
    "kv_v_uses_k": ("or_quant_fp8(v, 1, 1, n, n, OR_TENSOR,", "or_quant_fp8(k, 1, 1, n, n, OR_TENSOR,",
                    ["test_kv_write_is_per_tensor_on_k_and_v"]),
    "w4a16_gemm_scale_transposed": ("scale[(k / 128) * N + j]", "scale[j * (K / 128) + k / 128]",
                                    ["test_gemm_scale_indexing_matches_quantizer_dequant"]),
    "w4a16_gemm_drops_last_k": ("for (int64_t k = 0; k < K; k++) {\n            uint32_t word",
                                "for (int64_t k = 0; k < K - 1; k++) {\n            uint32_t word",
                                ["test_gemm_w4a16_integer_case_is_exact_matmul"]),
    "w4a16_gemm_unsigned_codes": ("if (q >= 8) q -= 16;", "",
                                  ["test_gemm_w4a16_integer_case_is_exact_matmul"]),
    "w4a16_gemm_A_transposed": ("or_bf16_to_f32(A[i * K + k])", "or_bf16_to_f32(A[k * M + i])",
                                ["test_gemm_w4a16_integer_case_is_exact_matmul"]),
    "w4a16_gemm_bound_signed": ("            mag += fabs(a * b);\n" + _W4A16_TAIL,
                                "            mag += a * b;\n" + _W4A16_TAIL,
                                ["test_gemm_w4a16_integer_case_is_exact_matmul"]),
    "fp8_gemm_sB_transposed": ("sB[(j / 128) * kb + k / 128]", "sB[(k / 128) * (N / 128) + j / 128]",
                               ["test_gemm_scale_indexing_matches_quantizer_dequant"]),
    "fp8_gemm_sA_per_row": ("(double)sA[i * kb + k / 128]", "(double)sA[i * kb]",
                            ["test_gemm_scale_indexing_matches_quantizer_dequant"]),
    "fp8_gemm_B_transposed": ("or_e4m3_decode(qB[j * K + k])", "or_e4m3_decode(qB[k * N + j])",
                              ["test_gemm_fp8_block_integer_case_is_exact_matmul"]),
    "nv_gemm_drops_gB": ("* or_e4m3_decode(sB[j * (K / 16) + k / 16]) * (double)gB;",
                         "* or_e4m3_decode(sB[j * (K / 16) + k / 16]);",
                         ["test_gemm_scale_indexing_matches_quantizer_dequant"]),
    "nv_gemm_sA_index": ("or_e4m3_decode(sA[i * (K / 16) + k / 16])", "or_e4m3_decode(sA[i * (K / 16) + k / 32])",
                         ["test_gemm_scale_indexing_matches_quantizer_dequant"]),
    "mx_gemm_bias": ("(int)eB[j * (K / 32) + k / 32] - 127", "(int)eB[j * (K / 32) + k / 32] - 126",
                     ["test_gemm_fp4_integer_case_is_exact_matmul"]),
    "e4m3_max_code_416": ("for (int c = 0; c <= 0x7E; c++) {", "for (int c = 0; c <= 0x7D; c++) {",
                          ["test_e4m3_decode_encode_identity_all_codes", "test_e4m3_saturates_like_clamp"]),
    "e4m3_bias_8": ("else v = ldexp(1.0 + (double)m / 8.0, e - 7);", "else v = ldexp(1.0 + (double)m / 8.0, e - 8);",
                    ["test_e4m3_format_facts", "test_e4m3_encode_matches_torch_cast"]),
    "e2m1_no_abs": ("uint8_t or_e2m1_encode(float y)\n{\n    double a = fabs((double)y);",
                    "uint8_t or_e2m1_encode(float y)\n{\n    double a = (double)y;",
                    ["test_e2m1_matches_torch_argmin_pipeline"]),
    "mx_no_clamp_floor": ("            if (amax < or_amax_min()) amax = or_amax_min();\n            int E",
                          "            int E", ["test_fp4_all_zero_blocks_use_clamp_floor"]),
    "nv_block_uses_tensor_amax": ("float t = bamax / OR_FP4_MAX / g;", "float t = amax_t / OR_FP4_MAX / g;",
                                  ["test_nvfp4_invariants"]),
    "int4_amax_signed": ("                float a = fabsf(or_elem(w, is_bf16, k * ldw + n));",
                         "                float a = or_elem(w, is_bf16, k * ldw + n);",
                         ["test_int4_g128_invariants"]),
    "kvh_v_uses_k": ("or_quant_fp8(v + h * TD, 1, 1, TD, TD,", "or_quant_fp8(k + h * TD, 1, 1, TD, TD,",
                     ["test_kv_per_head_reduces_to_per_tensor_per_head"]),
    "kvh_head_stride_halved": ("or_quant_fp8(k + h * TD, 1, 1, TD, TD,", "or_quant_fp8(k + h * (TD / 2), 1, 1, TD, TD,",
                               ["test_kv_per_head_reduces_to_per_tensor_per_head"]),
    "kvh_given_scale_of_head_0": ("scale[h], codes + h * TD", "scale[0], codes + h * TD",
                                  ["test_kv_per_head_given_matches_per_tensor_given"]),
    "kzp_zero_is_min": ("            float z = 0.5f * (mx + mn);", "            float z = mn;",
                        ["test_k_channel_zero_point_extremes_map_to_full_range"]),
    "kzp_zero_half_missing": ("            float z = 0.5f * (mx + mn);", "            float z = (mx + mn);",
                              ["test_k_channel_zero_point_extremes_map_to_full_range",
                               "test_k_channel_zero_point_is_translation_invariant"]),
    "kzp_deq_drops_zero": ("if (deq) deq[h * T * D + t * D + d] = dq + z;", "if (deq) deq[h * T * D + t * D + d] = dq;",
                           ["test_k_channel_zero_point_error_tracks_the_variation"]),
    "kzp_scale_divisor_447": ("/ OR_FP8_MAX;\n            scale[h * D + d] = s;", "/ 447.0f;\n            scale[h * D + d] = s;",
                              ["test_k_channel_zero_point_unit_scale_reduces_to_plain_cast"]),
    "i4zp_no_zero_inclusion": ("            float lo = 0.0f, hi = 0.0f;", "            float lo = 1e30f, hi = -1e30f;",
                               ["test_int4_zp_invariants"]),
    "i4zp_divisor_16": ("/ 15.0f;", "/ 16.0f;", ["test_int4_zp_worked_example"]),
    "i4zp_zero_sign": ("float zr = rintf(-lo / sq);", "float zr = rintf(lo / sq);",
                       ["test_int4_zp_worked_example", "test_int4_zp_invariants"]),
    "i4zp_zero_added_twice": ("float r = rintf(y) + (float)z;", "float r = rintf(y) + (float)(2 * z);",
                              ["test_int4_zp_worked_example", "test_int4_zp_invariants"]),
    "i4zp_gemm_ignores_zero": ("double b = (double)(q - z) *", "double b = (double)q *",
                               ["test_gemm_w4a16_zp_integer_case_is_exact_matmul"]),
    "i4zp_gemm_zero_per_row": ("int z = zero[(k / 128) * N + j];", "int z = zero[(j % (K / 128)) * N + j];",
                               ["test_gemm_w4a16_zp_integer_case_is_exact_matmul"]),
    "w4nv_drops_gB": ("or_e4m3_decode(srow[k / 16]) * (double)gB;", "or_e4m3_decode(srow[k / 16]);",
                      ["test_gemm_w4a16_fp4_equals_matmul_of_decoded_weights"]),
    "w4mx_bias": ("(int)erow[k / 32] - 127", "(int)erow[k / 32] - 126",
                  ["test_gemm_w4a16_fp4_equals_matmul_of_decoded_weights"]),
    "col_amax_signed": ("float a = fabsf(or_elem(x, is_bf16, r * cols + c));\n            if (a > out[c]) out[c] = a;",
                        "float a = or_elem(x, is_bf16, r * cols + c);\n            if (a > out[c]) out[c] = a;",
                        ["test_col_amax_matches_numpy"]),
    "smooth_alpha_swapped": ("s[j] = sqrtf(ax) / sqrtf(aw);", "s[j] = sqrtf(aw) / sqrtf(ax);",
                             ["test_smooth_factors_closed_forms", "test_smoothquant_int8_pipeline_preserves_the_product"]),
    "smooth_no_floor": ("float ax = xmax[j] > or_amax_min() ? xmax[j] : or_amax_min();", "float ax = xmax[j];",
                        ["test_smooth_factors_closed_forms"]),
    "int8_divisor_128": ("/ 127.0f;", "/ 128.0f;", ["test_int8_rows_worked_example", "test_int8_rows_invariants_and_smoothing"]),
    "int8_smooth_ops_swapped": ("            if (smooth == 1) v = v / f[c];\n            else if (smooth == 2) v = v * f[c];\n            if (fabsf(v) > amax)",
                                "            if (smooth == 1) v = v * f[c];\n            else if (smooth == 2) v = v / f[c];\n            if (fabsf(v) > amax)",
                                ["test_int8_rows_invariants_and_smoothing"]),
    "int8_gemm_B_transposed": ("(int64_t)qB[j * K + k]", "(int64_t)qB[k * N + j]", ["test_gemm_int8_is_scaled_integer_matmul"]),
    "int8_gemm_drops_sB": ("double sc = (double)sA[i] * (double)sB[j];", "double sc = (double)sA[i];",
                           ["test_gemm_int8_is_scaled_integer_matmul"]),
    "kv_k_scale_into_v": ("or_quant_fp8(k, 1, 1, n, n, OR_TENSOR, k_codes, k_scale, k_deq);",
                          "or_quant_fp8(k, 1, 1, n, n, OR_TENSOR, k_codes, v_scale, k_deq);",
                          ["test_kv_write_is_per_tensor_on_k_and_v"]),
}


def _run_pins(pins_mod, names):
    """Names of the pins (of `names`) that fail on the oracle currently loaded."""
    failed = []
    for name in names:
        fn = getattr(pins_mod, name)
        params = [(g,) for g in (0, 1, 2, 3)] if name == "test_fp8_invariants" else [()]
        for args in params:
            try:
                fn(*args)
            except Exception:
                failed.append(name)
                break
    return failed


def _child(workdir, q):
    """Spawned: build the control copy and every mutant, run their pins, report."""
    for p in (ROOT, os.path.join(ROOT, "tests")):
        if p not in sys.path:
            sys.path.insert(0, p)
    import oracle
    import test_oracle_pins as pins

    src = open(oracle._SRC, encoding="utf-8").read()
    real_build = oracle.build
    report = {"bad_text": [], "control": None, "caught": {}}

    def load(name, text):
        c = os.path.join(workdir, name + ".c")
        with open(c, "w", encoding="utf-8") as f:
            f.write(text)
        so = real_build(force=True, src=c, out=os.path.join(workdir, "lib" + name + ".so"))
        oracle._lib = None
        oracle.build = lambda force=False, so=so: so

    all_pins = sorted({p for _, _, ps in MUTANTS.values() for p in ps})
    load("control", src)
    report["control"] = _run_pins(pins, all_pins)
    for name, (old, new, names) in MUTANTS.items():
        if src.count(old) != 1:
            report["bad_text"].append(name)
            continue
        load(name, src.replace(old, new))
        report["caught"][name] = _run_pins(pins, names)
    q.put(report)


def test_pins_notice_every_planted_mistake(tmp_path):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    proc = ctx.Process(target=_child, args=(str(tmp_path), q))
    proc.start()
    report = q.get(timeout=600)
    proc.join(60)
    assert proc.exitcode == 0
    assert report["bad_text"] == [], f"mutation text not found exactly once: {report['bad_text']}"
    assert report["control"] == [], f"the unmodified copy fails {report['control']}"
    missed = [name for name, failed in report["caught"].items() if not failed]
    assert missed == [], f"no pin noticed: {missed}"
    assert len(report["caught"]) == len(MUTANTS)
