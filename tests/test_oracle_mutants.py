"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each one.

Every mutant is a one-expression change to oracle/moe_oracle.c (a wrong index,
an off-by-one, a dropped term, a wrong constant, truncation instead of
rounding). It is compiled on the CPU, swapped in for the real oracle, and the
pin tests of test_oracle_pins.py are run against it until one fails.
"""
import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

# (name, original text, planted mistake); each original must occur exactly once
MUTANTS = [
    ("region transposed", "int64_t region = (int64_t)e * R + src;", "int64_t region = (int64_t)src * E + e;"),
    ("slot position off by one", "int pos = counts[region]++;", "int pos = ++counts[region];"),
    ("flag without the +1", "flags[r] = (uint64_t)counts[r] + 1;", "flags[r] = (uint64_t)counts[r];"),
    ("duplicate check skipped", "if (row[jj] == e) return ORC_EINVAL;", "if (row[jj] == e + E) return ORC_EINVAL;"),
    ("header token and choice swapped", "meta[out * 4 + 3] = j;", "meta[out * 4 + 3] = t;"),
    ("scale block index wrong", "scales[i * nsc + h / 128]", "scales[i * nsc + h % nsc]"),
    ("expert factor wrong", "double c = 1.0 + (double)e / 256.0;", "double c = 1.0 + (double)e / 128.0;"),
    ("weight of the wrong choice", "double w = (double)weights[tok * k + j];",
     "double w = (double)weights[tok * k + (k - 1 - j)];"),
    ("one expert dropped", "acc[h] = (j == 0) ? term : acc[h] + term;", "acc[h] = (j == 0) ? 0.0 : acc[h] + term;"),
    ("sum starts from +0", "acc[h] = (j == 0) ? term : acc[h] + term;", "acc[h] = (j == 0) ? 0.0 + term : acc[h] + term;"),
    ("truncation instead of rounding", "double r = rint(a / quantum) * quantum;\n  if (r >= 0x1p128)",
     "double r = floor(a / quantum) * quantum;\n  if (r >= 0x1p128)"),
    ("bf16 subnormal spacing", "if (e < -126) e = -126;", "if (e < -140) e = -140;"),
    ("e4m3 exponent bias", "v = ldexp((double)(8 + m), ex - 10);", "v = ldexp((double)(8 + m), ex - 9);"),
    ("e4m3 subnormal scale", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("header bytes dropped", "out[2] = slots * 16;", "out[2] = slots * 4;"),
    ("T > max_m accepted", "if (T > max_m) return ORC_EINVAL;", "if (T > 2 * max_m) return ORC_EINVAL;"),
    ("e4m3 encoder truncates", "double r = rint(a / quantum) * quantum;\n  if (r < 0x1p-6)",
     "double r = floor(a / quantum) * quantum;\n  if (r < 0x1p-6)"),
    ("e4m3 subnormal boundary", "if (e < -6) e = -6;", "if (e < -7) e = -7;"),
    ("e4m3 no saturation", "if (a >= 448.0) return (uint8_t)(sign | 0x7E);", "if (a >= 480.0) return (uint8_t)(sign | 0x7E);"),
    ("packed offsets skip a region", "    region_offsets[r] = (int32_t)acc;\n    acc += counts[r];",
     "    acc += counts[r];\n    region_offsets[r] = (int32_t)acc;"),
    ("packed position ignored", "int64_t p = (int64_t)region_offsets[region] + slot_id[i] % max_m;",
     "int64_t p = (int64_t)region_offsets[region];"),
    ("silu on the up projection", "h[i] = orc_bf16_from_double(g / (1.0 + exp(-g)) * u);",
     "h[i] = orc_bf16_from_double(u / (1.0 + exp(-u)) * g);"),
    ("silu sign", "h[i] = orc_bf16_from_double(g / (1.0 + exp(-g)) * u);",
     "h[i] = orc_bf16_from_double(g / (1.0 + exp(g)) * u);"),
    ("fp8 silu sign", "hv[i] = g / (1.0 + exp(-g)) * u;", "hv[i] = g / (1.0 + exp(g)) * u;"),
    ("gate weight transposed", "g += xv * orc_bf16_value(w_gate[(int64_t)i * H + k]);",
     "g += xv * orc_bf16_value(w_gate[(int64_t)k * I + i]);"),
    ("down weight transposed", "acc += orc_bf16_value(h[i]) * orc_bf16_value(w_down[(int64_t)j * I + i]);",
     "acc += orc_bf16_value(h[i]) * orc_bf16_value(w_down[(int64_t)i * H + j]);"),
    ("linear weight transposed", "acc += orc_bf16_value(x[k]) * orc_bf16_value(w[(int64_t)n * K + k]);",
     "acc += orc_bf16_value(x[k]) * orc_bf16_value(w[(int64_t)k * N + n]);"),
    ("fp8 weight block scale transposed",
     "double wv = orc_e4m3_value(wq[(int64_t)n * K + k]) * (double)ws[(int64_t)(n / 128) * (K / 128) + k / 128];",
     "double wv = orc_e4m3_value(wq[(int64_t)n * K + k]) * (double)ws[(int64_t)(k / 128) * (K / 128) + n / 128];"),
    ("fp8 row scale dropped", "double xv = orc_e4m3_value(xq[k]) * (double)xs[k / 128];\n      double wv",
     "double xv = orc_e4m3_value(xq[k]);\n      double wv"),
    ("fp8 gate block scale index", "int64_t sb = (int64_t)(i / 128) * (H / 128) + k / 128;",
     "int64_t sb = (int64_t)(i % 128) % (H / 128) + k / 128;"),
    ("fp8 h scale off", "float sc = amax > 0.0f ? amax / 448.0f : 1.0f;\n    hs[b] = sc;",
     "float sc = amax > 0.0f ? amax / 440.0f : 1.0f;\n    hs[b] = sc;"),
    ("masked choice rejected", "if (e == -1) { /* a masked choice names no expert",
     "if (e == -2) { /* a masked choice names no expert"),
    ("masked term wipes the sum", "for (int h = 0; h < H; ++h) acc[h] = (j == 0) ? 0.0 : acc[h] + 0.0;",
     "for (int h = 0; h < H; ++h) acc[h] = 0.0;"),
    ("masked earlier choice read as rank 0", "if (row[jj] == -1) continue;", "if (row[jj] == -2) continue;"),
    ("quantiser scale off", "float s = amax > 0.0f ? amax / 448.0f : 1.0f;", "float s = amax > 0.0f ? amax / 447.0f : 1.0f;"),
]

# the pins, cheapest first; each takes the (unused) oracle_lib fixture value
PINS = [
    lambda: pins.test_validate(None),
    lambda: pins.test_bf16_ties_go_to_even(None),
    lambda: pins.test_e4m3_decode_matches_torch(None),
    lambda: pins.test_bf16_rounding_matches_torch_on_float32_inputs(None),
    lambda: pins.test_buffer_sizes_reproduce_the_printed_estimates(None),
    lambda: pins.test_layout_rejects_bad_routing(None),
    lambda: pins.test_layout_overflow_errors_out(None),
    lambda: pins.test_layout_matches_brute_force(None, 3, 7, 6, 3, 9, 1),
    lambda: pins.test_dispatch_slots_hold_source_rows(None, "tiny"),
    lambda: pins.test_dispatch_fp8_carries_scales(None),
    lambda: pins.test_expert_stub_is_the_nearest_bf16(None),
    lambda: pins.test_combine_identity_experts_return_the_input(None),
    lambda: pins.test_combine_scaling_experts_closed_form(None),
    lambda: pins.test_combine_is_linear_in_the_weights(None),
    lambda: pins.test_e4m3_encoder_saturates_and_round_trips(None),
    lambda: pins.test_e4m3_encoder_matches_torch(None),
    lambda: pins.test_quantize_row_properties(None),
    lambda: pins.test_compaction_groups_each_expert_by_source_then_token(None),
    lambda: pins.test_expert_mlp_row_is_zero_for_zero_gate(None),
    lambda: pins.test_expert_mlp_row_matches_a_library_matmul(None),
    lambda: pins.test_linear_row_matches_a_library_matmul_and_an_identity(None),
    lambda: pins.test_linear_row_fp8_unit_scales_identity(None),
    lambda: pins.test_linear_row_fp8_matches_a_library_matmul(None),
    lambda: pins.test_gate_up_row_fp8_matches_library_ops(None),
    lambda: pins.test_layout_with_masked_choices_matches_brute_force(None, 2, 16, 8, 2, 16, 5),
    lambda: pins.test_combine_with_masked_choices_sums_only_the_others(None),
    lambda: pins.test_route_stats_skip_masked_choices(None),
]


def test_every_mutant_site_exists_once():
    src = oracle.source()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, name


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    oracle._load()
    real = oracle._lib
    lib_path = str(tmp_path / "liboracle_mutant.so")
    oracle.compile_variant(oracle.source().replace(old, new), lib_path)
    oracle._lib = oracle._bind(lib_path)
    caught = None
    try:
        for i, pin in enumerate(PINS):
            try:
                with np.errstate(all="ignore"):
                    pin()
            except (AssertionError, oracle.OracleError, pytest.fail.Exception, ValueError, IndexError, KeyError) as e:
                caught = (i, type(e).__name__)
                break
    finally:
        oracle._lib = real
    assert caught is not None, f"no pin caught the mutant '{name}'"


def test_real_oracle_passes_the_same_pins():
    oracle._load()
    for pin in PINS:
        pin()
