"""The oracle's pins are sharp: each plausible mistake below (a dropped term,
a wrong sign, index or comparison, a transposed operand), planted in a
temporary copy of oracle.cpp on the CPU, makes at least one pin fail."""
import ctypes as C
import os
import shutil
import tempfile

import pytest

import oracle  # noqa: F401
from oracle import build as ob
import test_oracle_pins as pins

MUTANTS = {
    "ef_term_dropped": ("acc[i] = e ? g[i] + e[i] : g[i];\n  std::vector<uint32_t> key(n);\n  for (int64_t i = 0; i < n; ++i) key[i] = magnitude_key(acc[i]);\n  std::vector<int64_t> S = select_k<LargerFirst>",
                        "acc[i] = g[i];\n  std::vector<uint32_t> key(n);\n  for (int64_t i = 0; i < n; ++i) key[i] = magnitude_key(acc[i]);\n  std::vector<int64_t> S = select_k<LargerFirst>",
                        ["test_ef_topk_equations_and_invariant"]),
    "tie_to_higher_index": ("if (key[a] != key[b]) return key[a] > key[b];\n    return a < b;",
                            "if (key[a] != key[b]) return key[a] > key[b];\n    return a > b;",
                            ["test_select_matches_full_sort_and_lexsort"]),
    "int8_sign_flipped": ("return (int8_t)(std::signbit(x) ? -v : v);", "return (int8_t)(std::signbit(x) ? v : -v);",
                          ["test_topk_int8_codes_are_unbiased"]),
    "sr_compare_le": ("bool up = (double)r < (double)frac * 4294967296.0;",
                      "bool up = (double)r <= (double)frac * 4294967296.0;",
                      ["test_stochastic_round_toy_example"]),
    "momentum_operands_swapped": ("float bu = beta * u[i];\n    u[i] = bu + g[i];", "float bu = beta * g[i];\n    u[i] = bu + u[i];",
                                  ["test_momentum_closed_form_sequences"]),
    "sign_scale_wrong_count": ("float mu = (float)(sum / (double)n);", "float mu = (float)(sum / (double)(n + 1));",
                               ["test_sign_bits_scale_and_residual"]),
    "qsgd_levels_dropped": ("float x = (std::fabs(acc[i]) * (float)s_levels) / sc;", "float x = std::fabs(acc[i]) / sc;",
                            ["test_qsgd_single_nonzero_and_norm"]),
    "philox_key_not_bumped": ("    k0 += W0;\n    k1 += W1;", "    k1 += W1;", ["test_philox_matches_triton_interpreter"]),
    "decompress_tensor_offset_lost": ("out[off[t] + i] = out[off[t] + i] + v;", "out[i] = out[i] + v;",
                                      ["test_sparse_accumulate_matches_numpy_add_at"]),
    "clip_ratio_inverted": ("const float c = max_norm / N;", "const float c = N / max_norm;",
                            ["test_clipping_scales_to_max_norm_and_leaves_small_tensors"]),
    "powersgd_gs_sign": ("for (int64_t i = 0; i < m; ++i) p[i * r + k] = p[i * r + k] - d * p[i * r + j];",
                         "for (int64_t i = 0; i < m; ++i) p[i * r + k] = p[i * r + k] + d * p[i * r + j];",
                         ["test_powersgd_one_step_matches_numpy_and_keeps_the_residual"]),
    "powersgd_q_transposed": ("q[jcol * r + k] = (float)dot_rows(m, &M[jcol], n, p + k, r);",
                              "q[jcol * r + k] = (float)dot_rows(m, &M[jcol], 1, p + k, r);",
                              ["test_powersgd_one_step_matches_numpy_and_keeps_the_residual"]),
    "int8_decode_scale_dropped": ("      d = (float)codes[i] * sc;", "      d = (float)codes[i];",
                                  ["test_int8_decode_exact_on_a_representable_grid_and_restores_acc"]),
    "momentum_int8_residual_zeroed": ("      v[i] = v[i] - d;", "      v[i] = 0.0f;",
                                      ["test_momentum_int8_reduces_to_ef_topk_int8_and_keeps_quantization_error"]),
    "kept_qsgd_norm_by_position": ("for (int64_t i : S) ss += (double)x[i] * (double)x[i];",
                                   "for (size_t i = 0; i < S.size(); ++i) ss += (double)x[i] * (double)x[i];",
                                   ["test_kept_qsgd_norm_is_over_the_kept_set_and_one_kept_value_is_sent_exactly"]),
    "kept_qsgd_draw_purpose": ("const float y = (std::fabs(x[i]) * (float)s_levels) / sc;\n        double m = stochastic_round(y, draw_u32(seed, iter, base + (uint64_t)i, PURPOSE_QSGD));",
                               "const float y = (std::fabs(x[i]) * (float)s_levels) / sc;\n        double m = stochastic_round(y, draw_u32(seed, iter, base + (uint64_t)i, PURPOSE_INT8));",
                               ["test_kept_quantizers_with_every_element_kept_are_the_dense_quantizers"]),
    "kept_sign_bit_inverted": ("      if (!neg) bits[j / 32] |= 1u << (j % 32);", "      if (neg) bits[j / 32] |= 1u << (j % 32);",
                               ["test_kept_sign_bits_mean_and_residual"]),
    "kept_residual_dropped": ("    if (res) res[i] = x[i] - d;", "    if (res) res[i] = 0.0f;",
                              ["test_kept_sign_bits_mean_and_residual"]),
    "receiver_sign_words_not_offset": ("      word0 += (koff[t + 1] - koff[t] + 31) / 32;", "      word0 += 0;",
                                       ["test_quantized_sparse_receiver_restores_the_senders_decoded_values"]),
    "receiver_qsgd_levels_not_divided": ("          const float mag = ((float)level * sc) / (float)s_levels;\n          v = c < 0 ? -mag : mag;",
                                         "          const float mag = ((float)level * sc);\n          v = c < 0 ? -mag : mag;",
                                         ["test_quantized_sparse_receiver_restores_the_senders_decoded_values"]),
    "randk_largest_keys": ("if (key[a] != key[b]) return key[a] < key[b];", "if (key[a] != key[b]) return key[a] > key[b];",
                           ["test_randk_selection_is_k_smallest_keys"]),
}


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, workdir):
    old, new, tests = MUTANTS[name]
    src = open(ob.SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = os.path.join(workdir, name + ".cpp")
    with open(path, "w") as fh:
        fh.write(src.replace(old, new, 1))
    lib = C.CDLL(ob.compile_oracle(path, os.path.join(workdir, name + ".so")))
    oracle._declare(lib)
    saved = oracle._lib
    oracle._lib = lib
    try:
        caught = 0
        for t in tests:
            try:
                getattr(pins, t)()
            except AssertionError:
                caught += 1
            except pytest.skip.Exception:
                pytest.skip("pin unavailable here")
        assert caught >= 1, f"mutant {name} survived {tests}"
    finally:
        oracle._lib = saved
