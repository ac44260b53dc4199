"""Plants plausible mistakes in copies of the CPU oracle and checks that the
pins in test_oracle_pins.py catch every one of them.  Runs on the CPU only;
the mutants are compiled into a temporary directory."""
import importlib.util
import os
import subprocess

import pytest

import test_oracle_pins as PINS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qvg_oracle.cpp")
PY = os.path.join(ROOT, "oracle", "oracle.py")

MUTATIONS = {
    "residual sign": ("r[e] = r[e] - deq;", "r[e] = r[e] + deq;"),
    "packing stride": ("codes[(e * b) / 32] |= (uint32_t)q << ((e * b) % 32);",
                       "codes[(e * b) / 32] |= (uint32_t)q << ((e * b) % 16);"),
    "scale divisor": ("float s32 = range / (float)L;", "float s32 = range / (float)(L + 1);"),
    "clamp at 3 for every width": ("int q = qf > 0.0f ? (qf > (float)L ? L : (int)qf) : 0;",
                                   "int q = qf > 0.0f ? (qf > 3.0f ? 3 : (int)qf) : 0;"),
    "quantiser multiplies by the reciprocal": ("float t = (s != 0.0f) ? (r[e] - z) / s : 0.0f;",
                                               "float t = (s != 0.0f) ? (r[e] - z) * (1.0f / s) : 0.0f;"),
    "4-bit field mask": ("& ((1u << b) - 1u);", "& 3u;"),
    "zero from max": ("uint16_t sh = to_f16(s32), zh = to_f16(mn);",
                      "uint16_t sh = to_f16(s32), zh = to_f16(mx);"),
    "rounding floor": ("float qf = std::nearbyint(t);", "float qf = std::floor(t);"),
    "meta halves swapped": ("meta[g] = (uint32_t)sh | ((uint32_t)zh << 16);",
                            "meta[g] = (uint32_t)zh | ((uint32_t)sh << 16);"),
    "argmin ties to highest": ("if (d < best) { best = d; arg = j; }",
                               "if (d <= best) { best = d; arg = j; }"),
    "distance sign": ("double diff = bf16_value(x[i]) - bf16_value(c[i]);",
                      "double diff = bf16_value(x[i]) + bf16_value(c[i]);"),
    "init index rounding": ("int64_t n = ((int64_t)j * N) / C;",
                            "int64_t n = ((int64_t)j * N + C - 1) / C;"),
    "mean divisor": ("to_bf16(sum[(size_t)j * D + i] / (double)cnt[j]);",
                     "to_bf16(sum[(size_t)j * D + i] / (double)(cnt[j] + 1));"),
    "empty cluster reset": ("if (cnt[j] == 0) continue;",
                            "if (cnt[j] == 0) { for (int i = 0; i < D; ++i) cent[(size_t)j * D + i] = 0; continue; }"),
    "decode drops centroid": ("float acc = cent ? bf16_float(cent[(int64_t)ids[n] * D + i]) : 0.0f;",
                              "float acc = 0.0f;"),
    "decode drops last stage": ("for (int s = 0; s < S; ++s)\n                acc = acc + stage_value(codes + ((int64_t)s * N + n)",
                                "for (int s = 0; s + 1 < S; ++s)\n                acc = acc + stage_value(codes + ((int64_t)s * N + n)"),
    "coral drops low rank": ("pred[n * HD + h * D + o] = blk + low;", "pred[n * HD + h * D + o] = blk;"),
    "coral block transposed": ("blk = blk + bf16_value(B[((int64_t)h * D + o) * D + i])",
                               "blk = blk + bf16_value(B[((int64_t)h * D + i) * D + o])"),
    "coral residual sign": ("r[i] = bf16_float(x_next[e]) - pv;", "r[i] = bf16_float(x_next[e]) + pv;"),
    "stream ignores warm start": ("const uint16_t* warm = nv ? versions + (size_t)(nv - 1) * C * D : nullptr;",
                                  "const uint16_t* warm = nullptr;"),
    "ridge sign": ("for (int i = 0; i < D; ++i) Gm[(size_t)i * D + i] = Gm[(size_t)i * D + i] + lambda;",
                   "for (int i = 0; i < D; ++i) Gm[(size_t)i * D + i] = Gm[(size_t)i * D + i] - lambda;"),
    "fit low-rank sign": ("res[o] = bf16_value(y[n * HD + h * D + o]) - low;",
                          "res[o] = bf16_value(y[n * HD + h * D + o]) + low;"),
    "fit output transposed": ("Bh[(size_t)o * D + i] = to_bf16(z);", "Bh[(size_t)i * D + o] = to_bf16(z);"),
    "size meta term": ("double bits = (double)S * b + 32.0 * S / G;", "double bits = (double)S * b + 16.0 * S / G;"),
    "bf16 rounding truncates": ("double r = std::nearbyint(n); // default rounding mode: ties to even",
                                "double r = std::trunc(n);"),
}

PIN_CALLS = [
    (PINS.test_bf16_rounding_is_exact_nearest_even, {}),
    (PINS.test_f16_rounding_matches_ieee, {}),
    (PINS.test_single_stage_no_smoothing_is_rtn, {"D": 128, "G": 64, "b": 2}),
    (PINS.test_single_stage_no_smoothing_is_rtn, {"D": 128, "G": 16, "b": 4}),
    (PINS.test_exact_midpoints_round_to_even_level, {"b": 2}),
    (PINS.test_exact_midpoints_round_to_even_level, {"b": 4}),
    (PINS.test_pack_example_golden, {}),
    (PINS.test_pack_example_4bit_golden, {}),
    (PINS.test_on_grid_values_round_trip, {"b": 2}),
    (PINS.test_on_grid_values_round_trip, {"b": 4}),
    (PINS.test_constant_group, {"b": 2}),
    (PINS.test_constant_group, {"b": 4}),
    (PINS.test_stage_error_bound_and_monotonicity, {"b": 2}),
    (PINS.test_stage_error_bound_and_monotonicity, {"b": 4}),
    (PINS.test_decode_inverts_encode_within_last_stage_bound, {}),
    (PINS.test_decode_stage_sum_order, {}),
    (PINS.test_init_indices_golden, {}),
    (PINS.test_assign_brute_force_exact, {}),
    (PINS.test_update_is_exact_mean_rounded, {}),
    (PINS.test_lloyd_sse_non_increasing_and_zero_mean_residuals, {}),
    (PINS.test_separable_mixture_recovers_partition, {}),
    (PINS.test_stream_protocol, {}),
    (PINS.test_bits_per_element_closed_form, {}),
    (PINS.test_coral_block_part_is_block_diagonal_matmul, {}),
    (PINS.test_coral_low_rank_part, {}),
    (PINS.test_coral_identity_predictor_gives_exact_reconstruction, {}),
    (PINS.test_coral_zero_predictor_is_plain_prq, {}),
    (PINS.test_coral_decode_matches_encoder_reconstruction, {}),
    (PINS.test_coral_fit_block_matches_library_solve, {}),
    (PINS.test_coral_fit_block_recovers_an_exact_block, {}),
    (PINS.test_coral_fit_block_zero_input, {}),
]


def _load_mutant(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not unique/absent: {name}"
    src = tmp_path / "mut.cpp"
    src.write_text(text.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(src)])
    spec = importlib.util.spec_from_file_location("oracle_mutant_" + str(abs(hash(name))), PY)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC, mod._LIB, mod._lib = str(src), str(so), None
    mod.lib()
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    mod = _load_mutant(tmp_path, name, old, new)
    caught = []
    for fn, kw in PIN_CALLS:
        try:
            fn(mod, **kw)
        except Exception:          # an assertion (or a crash of the check) = caught
            caught.append(fn.__name__)
    assert caught, f"no pin caught the planted mistake '{name}'"


# Mistakes planted in the oracle's Python side (the Coral + SAS hybrid
# composition and its bf16 rounding), run against the same compiled oracle.
PY_MUTATIONS = {
    "hybrid residual sign": ("r = f32_to_bf16_bits(bf16_bits_to_f32(x_next) - pred)",
                             "r = f32_to_bf16_bits(bf16_bits_to_f32(x_next) + pred)"),
    "hybrid reconstruction drops the prediction": ("x_hat = f32_to_bf16_bits(pred + bf16_bits_to_f32(rhat))",
                                                   "x_hat = rhat.copy()"),
    "hybrid bf16 rounding truncates": ("return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)",
                                       "return (u >> 16).astype(np.uint16)"),
    "hybrid head slice": ("rh = np.ascontiguousarray(r[:, h * D:(h + 1) * D])",
                          "rh = np.ascontiguousarray(r[:, 0:D])"),
    "attention drops the scale": ("s = float(scale) * (Qf @ Kf.T)", "s = Qf @ Kf.T"),
    "attention weighs the keys": ("return (p @ Vf) / p.sum(axis=1, keepdims=True)",
                                  "return (p @ Kf) / p.sum(axis=1, keepdims=True)"),
    "attention max over queries": ("p = np.exp(s - s.max(axis=1, keepdims=True))",
                                   "p = np.exp(s - s.max(axis=0, keepdims=True))"),
    "attention unnormalised": ("return (p @ Vf) / p.sum(axis=1, keepdims=True)", "return p @ Vf"),
}

PY_PIN_CALLS = [
    (PINS.test_f32_to_bf16_rounding_matches_exact_rationals, {}),
    (PINS.test_coral_sas_zero_prediction_is_plain_qvg, {}),
    (PINS.test_coral_sas_perfect_prediction_reconstructs_exactly, {}),
    (PINS.test_coral_sas_residual_and_reconstruction_arithmetic, {}),
    (PINS.test_attention_matches_torch_sdpa_in_fp64, {}),
    (PINS.test_attention_closed_forms, {}),
    (PINS.test_attention_invariances, {}),
]


@pytest.mark.parametrize("name", sorted(PY_MUTATIONS))
def test_pins_catch_planted_python_mistake(tmp_path, name):
    old, new = PY_MUTATIONS[name]
    text = open(PY).read()
    assert text.count(old) == 1, f"mutation anchor not unique/absent: {name}"
    path = tmp_path / "oracle_mut.py"
    path.write_text(text.replace(old, new))
    spec = importlib.util.spec_from_file_location("oracle_py_mutant_" + str(abs(hash(name))), str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC, mod._LIB, mod._lib = SRC, os.path.join(ROOT, "oracle", "liboracle.so"), None
    mod.lib()
    caught = []
    for fn, kw in PY_PIN_CALLS:
        try:
            fn(mod, **kw)
        except Exception:
            caught.append(fn.__name__)
    assert caught, f"no pin caught the planted mistake '{name}'"
