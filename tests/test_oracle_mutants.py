"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a wrong
order of the momentum updates, the tie rule reversed, a missing mask, > for
>=, a wrong neighbour on the ring, a swapped Philox key word, ...), rebuilds
the copy and runs the oracle's pin tests against it: at least one pin must
fail.  Nothing here touches the CUDA path; the mistakes live only in a
temporary copy of the oracle.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC_PATH = os.path.join(ROOT, "oracle", "gcsgd_oracle.c")
PIN_FILES = ["test_oracle_dgc.py", "test_oracle_adacomp.py", "test_oracle_average_dcd.py", "test_oracle_wire.py"]

# name -> (text in the oracle, planted replacement)
MUTANTS = {
    # DGC (momentum correction, selection, masking, clipping, k)
    "v_before_u": ("            } else {\n                vk[i] = vk[i] + uk[i];\n            }",
                   "            } else {\n                vk[i] = vk[i] + (uk[i] - g) / momentum;\n            }"),
    "no_momentum": ("float mu = momentum * uk[i];", "float mu = 0.0f * uk[i];"),
    "ties_to_higher_index": ("return x->idx < y->idx ? -1 : 1;", "return x->idx > y->idx ? -1 : 1;"),
    "u_not_masked": ("uk[off + i] = 0.0f;\n            }", "}"),
    "v_not_masked": ("vk[off + i] = 0.0f;\n                uk", "uk"),
    "clip_norm_of_first_tensor": ("for (int64_t i = 0; i < N; ++i) csum_add(&acc, (double)G[i] * (double)G[i]);",
                                  "for (int64_t i = 0; i < seg_off[1]; ++i) csum_add(&acc, (double)G[i] * (double)G[i]);"),
    "topk_key_keeps_sign": ("return bits_of(f) & 0x7fffffffu;", "return bits_of(f);"),
    "clip_not_applied": ("float g = clipped ? G[i] * c : G[i];", "float g = G[i];"),
    "clip_ignores_nodes": ("/ sqrt((double)clip_nodes)", "/ 1.0"),
    "clip_scale_inverted": ("if (norm > thr_k) { c = (float)(thr_k / norm)", "if (norm > thr_k) { c = (float)(norm / thr_k)"),
    "k_floor": ("double kd = ceil(density * (double)n);", "double kd = floor(density * (double)n);"),
    # DGC with Nesterov momentum (the reading)
    "nesterov_step_without_momentum": ("float step = momentum * uk[i];", "float step = uk[i];"),
    "nesterov_ignored": ("            if (nesterov) {", "            if (0) {"),
    # DGC with the sampled threshold
    "sampled_strict_gt": ("c += order[i].key >= tau;", "c += order[i].key > tau;"),
    "sampled_rank_floor": ("int64_t a = (ks * m + n / 2) / n;", "int64_t a = (ks * m) / n;"),
    # the sampled threshold limited by the earlier plan's sizes, which the page does not give
    "sampled_only_above_16384": ("if (m > 0) {", "if (m > 0 && n > 16384) {"),
    "sampled_only_at_low_density": ("if (m > 0) {", "if (m > 0 && 5 * ks <= n) {"),
    "sampled_capped_at_16384": ("return m - m % ORACLE_SAMPLE_BLOCK;",
                                "m -= m % ORACLE_SAMPLE_BLOCK;\n    return m > 16384 ? 16384 : m;"),
    "sampled_at_least_one_block": ("return m - m % ORACLE_SAMPLE_BLOCK;",
                                   "m -= m % ORACLE_SAMPLE_BLOCK;\n    return m < ORACLE_SAMPLE_BLOCK ? ORACLE_SAMPLE_BLOCK : m;"),
    "sampled_stride": ("const int64_t nblk = m / ORACLE_SAMPLE_BLOCK, stride = n / nblk;",
                       "const int64_t nblk = m / ORACLE_SAMPLE_BLOCK, stride = n / (nblk + 1);"),
    # AdaComp
    "ada_strict_gt": ("(fabsf(h) >= m)", "(fabsf(h) > m)"),
    "ada_h_without_dw": ("const float h = G[off + i] + dWk[off + i];", "const float h = G[off + i];"),
    "ada_sign_from_h": ("Q[off + i] = G[off + i] > 0.0f ? scale : -scale;", "Q[off + i] = h > 0.0f ? scale : -scale;"),
    "ada_residue_not_reduced": ("Rk[i] = G[i] - Q[i];", "Rk[i] = G[i];"),
    "ada_mean_over_nb_minus_1": ("/ (double)nb);", "/ (double)(nb > 1 ? nb - 1 : 1));"),
    "ada_partial_bin_dropped": ("const int64_t nb = (n + L - 1) / L;", "const int64_t nb = n / L > 0 ? n / L : 1;"),
    # sparse average
    "average_reverse_learner_order": ("    for (int k = 0; k < K; ++k) {\n        if (counts[k] < 0 || counts[k] > cap)",
                                      "    for (int k = K - 1; k >= 0; --k) {\n        if (counts[k] < 0 || counts[k] > cap)"),
    "ada_bin_max_of_dw": ("float a = fabsf(G[off + i]);", "float a = fabsf(dWk[off + i]);"),
    "dgc_sends_u": ("out_val[pos] = vk[off + i];", "out_val[pos] = uk[off + i];"),
    "ada_unselected_residue_dw": ("                Rk[i] = G[i];\n            }", "                Rk[i] = G[i] - Rk[i];\n            }"),
    "ada_scale_of_last_bin": ("const float scale = (float)(csum_value(&acc) / (double)nb);",
                              "const float scale = (float)bmax[nb - 1];"),
    "dcd_reads_updated_left_neighbour": ("const float* xl = xhat + (int64_t)l * d;",
                                         "const float* xl = (l < i ? xn : xhat) + (int64_t)l * d;"),
    "average_not_divided": ("out[j] = out[j] / fk;", "out[j] = out[j];"),
    "update_adds_the_step": ("w[j] = w[j] - step;", "w[j] = w[j] + step;"),
    "update_skips_last_list": ("for (int k = 0; k < K; ++k)\n            for (int64_t p = 0; p < counts[k]; ++p) carried",
                               "for (int k = 0; k < K - 1; ++k)\n            for (int64_t p = 0; p < counts[k]; ++p) carried"),
    # wire encodings
    "wire_escape_width": ("            gap -= 65536;", "            gap -= 65535;"),
    "wire_ada_global_index": ("const uint32_t local = (uint32_t)((int64_t)idx[j] - seg_off[s]);",
                              "const uint32_t local = (uint32_t)((int64_t)idx[j]);"),
    "wire_dgc_decode_gap_off_by_one": ("        memcpy(&dense[pos], &b, 4);\n        ++pos;\n",
                                       "        memcpy(&dense[pos], &b, 4);\n"),
    "wire_sign_bit": ("const uint32_t sign = val[j] < 0.0f ? 1u : 0u;", "const uint32_t sign = val[j] > 0.0f ? 1u : 0u;"),
    # Philox and DCD-PSGD
    "philox_key_word_swapped": ("uint32_t n0 = hi1 ^ c1 ^ k0;", "uint32_t n0 = hi1 ^ c1 ^ k1;"),
    "dcd_wrong_neighbour": ("const int l = (i + n - 1) % n, r = (i + 1) % n;\n        const float* xl",
                            "const int l = (i + n - 1) % n, r = (i + 2) % n;\n        const float* xl"),
    "dcd_ring_weights_mirrored": ("float acc = w[0] * xl[e];\n            acc = acc + w[1] * xi[e];\n            acc = acc + w[2] * xr[e];",
                                  "float acc = w[2] * xl[e];\n            acc = acc + w[1] * xi[e];\n            acc = acc + w[0] * xr[e];"),
    "dcd_compresses_the_model": ("            const float z = xh - xi[e];\n            const uint32_t word = dcd_word(",
                                 "            const float z = xh;\n            const uint32_t word = dcd_word("),
    "dcd_gradient_sign": ("const float xh = acc - gamma * gi[e];", "const float xh = acc + gamma * gi[e];"),
    "dcd_no_unbiasing_scale": ("return ((uint64_t)word < thr) ? z * inv_p : 0.0f;",
                               "return ((uint64_t)word < thr) ? z : 0.0f;"),
    "ecd_estimate_from_uncompressed_z": ("xt[q] = c * xt[q] + e2 * cz;", "xt[q] = c * xt[q] + e2 * z;"),
    "ecd_gradient_sign": ("x_prev[(int64_t)i * d + e] = acc - gamma * g[(int64_t)i * d + e];",
                          "x_prev[(int64_t)i * d + e] = acc + gamma * g[(int64_t)i * d + e];"),
    "ecd_extrapolation_swapped": ("const float z = a * x_prev[q] + b * x[q];", "const float z = b * x_prev[q] + a * x[q];"),
    "ecd_estimate_weight": ("const float c = (float)(1.0 - 2.0 / (double)t)", "const float c = (float)(1.0 - 1.0 / (double)t)"),
    "ecd_self_from_estimate": ("acc = acc + w[1] * x[(int64_t)i * d + e];", "acc = acc + w[1] * xt[(int64_t)i * d + e];"),
    "dcd_counter_words_swapped": ("uint32_t ctr[4] = {(uint32_t)(e >> 2), node, t, (uint32_t)(e >> 34)};",
                                  "uint32_t ctr[4] = {(uint32_t)(e >> 2), t, node, (uint32_t)(e >> 34)};"),
}


def _copy_tree(dst):
    os.makedirs(os.path.join(dst, "tests"))
    for f in ["conftest.py", *PIN_FILES]:
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ["__init__.py", "gcsgd_oracle.c"]:
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, "oracle", f))
    pkg = "gradient_compression_sgd_gb300"
    os.makedirs(os.path.join(dst, pkg))
    for f in ["__init__.py", "workloads.py", "build.py"]:
        shutil.copy(os.path.join(ROOT, pkg, f), os.path.join(dst, pkg, f))
    shutil.copy(os.path.join(ROOT, "pytest.ini"), dst)


def test_unmutated_copy_passes(tmp_path):
    _copy_tree(str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        *[os.path.join("tests", f) for f in PIN_FILES]],
                       cwd=tmp_path, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    src = open(SRC_PATH).read()
    a, b = MUTANTS[name]
    assert src.count(a) >= 1, f"mutation site for {name} no longer in the oracle"
    _copy_tree(str(tmp_path))
    with open(tmp_path / "oracle" / "gcsgd_oracle.c", "w") as f:
        f.write(src.replace(a, b, 1))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        *[os.path.join("tests", f) for f in PIN_FILES]],
                       cwd=tmp_path, capture_output=True, text=True, timeout=600)
    last = (r.stdout.strip().splitlines() or [""])[-1]
    assert r.returncode == 1 and "failed" in last, f"{name} not caught: {last}\n{r.stdout[-1500:]}"
