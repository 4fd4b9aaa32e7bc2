"""The pins must catch plausible mistakes.  Each case plants one mistake in a
copy of the oracle's C source (on the CPU, in a temporary directory),
builds it, points the oracle front end at the mutant and runs the pins; at
least one pin has to fail for every mutant."""
import os
import shutil
import subprocess

import pytest

import oracle.build as obuild
import oracle.oracle as ofront

from tests import test_oracle_aggregate as tagg
from tests import test_oracle_diag as tdiag
from tests import test_oracle_logdiff as tlog
from tests import test_oracle_philox as tphilox
from tests import test_oracle_powersgd as tpsgd
from tests import test_oracle_quant as tquant
from tests import test_oracle_randk as trandk
from tests import test_oracle_topk as ttopk

MUTANTS = {
    "tie_order_reversed": ("if (a->index != b->index) return a->index < b->index ? -1 : 1;",
                           "if (a->index != b->index) return a->index > b->index ? -1 : 1;"),
    "half_away_rounding": ("q = rintf(t);", "q = roundf(t);"),
    "dropped_offset": ("if (mode == ORC_MINMAX) return mag + p.offset;",
                       "if (mode == ORC_MINMAX) return mag;"),
    "stride_pairing": ("scratch[j] = scratch[2 * j] + scratch[2 * j + 1];",
                       "scratch[j] = scratch[j] + scratch[j + half];"),
    "no_key_bump": ("k0 += PHILOX_WEYL_A;", "k0 += 0u;"),
    "msb_first_packing": ("buf[bit >> 3] |= (uint8_t)(code << (bit & 7));",
                          "buf[bit >> 3] |= (uint8_t)(code << (8 - bits - (bit & 7)));"),
    "residual_sign": ("err[i] = c[i] - g_hat[i];", "err[i] = g_hat[i] - c[i];"),
    "topk_residual_not_zeroed": ("err[i] = keep[i] ? 0.0f : c[i];", "err[i] = c[i];"),
    "qsgd_levels_off_by_one": ("p.scale = norm / levels;",
                               "p.scale = norm / (levels + 1.0f);"),
    "ef_add_dropped": ("for (int64_t i = 0; i < n; ++i) c[i] = grad[i] + err[i];",
                       "for (int64_t i = 0; i < n; ++i) c[i] = grad[i];"),
    "stochastic_compare_flipped": ("q = fl + (u < frac ? 1.0f : 0.0f);",
                                   "q = fl + (u > frac ? 1.0f : 0.0f);"),
    "sign_plane_missing": ("if (mode == ORC_QSGD && negative) put_bits(sign_plane, i, 1, 1u);",
                           "(void)sign_plane;"),
    "minmax_range_swapped": ("p.scale = (mx - mn) / levels;", "p.scale = (mx + mn) / levels;"),
    "uniform_word_wrong": ("uint32_t word = r[i & 3u];", "uint32_t word = r[0];"),
    "mgs_no_projection": ("for (int64_t i = 0; i < m; ++i) P[i * r + c] -= d * P[i * r + l];",
                          "(void)d;"),
    "mgs_no_normalise": ("for (int64_t i = 0; i < m; ++i) P[i * r + c] /= nrm;",
                         "(void)nrm;"),
    "powersgd_residual_sign": ("err[i * n + j] = (float)(M[i * n + j] - a);",
                               "err[i * n + j] = (float)(a - M[i * n + j]);"),
    "powersgd_q_transposed": ("for (int64_t i = 0; i < m; ++i) s += M[i * n + j] * P[i * r + c];",
                              "for (int64_t i = 0; i < m && i < n; ++i) s += M[j * n + i] * P[i * r + c];"),
    "aggregate_reverse_rank_order": ("  for (int w = 0; w < W; ++w)\n    for (int64_t j = 0; j < k; ++j) {\n      int64_t at",
                                     "  for (int w = W - 1; w >= 0; --w)\n    for (int64_t j = 0; j < k; ++j) {\n      int64_t at"),
    "aggregate_assign_not_add": ("out[idx[at]] = out[idx[at]] + val[at];", "out[idx[at]] = val[at];"),
    "randk_compare_flipped": ("int keep = orc_uniform(seed, step, (uint64_t)i) < p;",
                              "int keep = orc_uniform(seed, step, (uint64_t)i) >= p;"),
    "randk_residual_not_zeroed": ("if (err) err[i] = keep ? 0.0f : c;", "if (err) err[i] = c;"),
    "log_plus_one_dropped": ("t = p.scale == 0.0f ? 0.0f : orc_logf(fabsf(x[i]) + 1.0f) / p.scale;",
                             "t = p.scale == 0.0f ? 0.0f : orc_logf(fabsf(x[i]) + 0.0f) / p.scale;"),
    "log_levels_ignore_sign_bit": ("float levels = (float)((1 << (bits - 1)) - 1);\n      p.scale = orc_logf",
                                   "float levels = (float)((1 << bits) - 1);\n      p.scale = orc_logf"),
    "log_series_term_dropped": ("r = 0x1.555556p-2f + z * r;", "r = 0x1.555556p-2f + 0.0f * r;"),
    "exp_range_reduction_lo_dropped": ("float r = (y - kf * LN2_HI) - kf * LN2_LO;",
                                       "float r = (y - kf * LN2_HI);"),
    "diff_open_loop_history": ("      ref[i] = g_hat;\n", "      ref[i] = c[i];\n"),
    "diff_refresh_ignored": ("    float r = refresh ? 0.0f : ref[i];\n    d[i] = c[i] - r;",
                             "    float r = ref[i];\n    d[i] = c[i] - r;"),
    "diag_energy_of_c_not_residual": ("s_e += (double)r * (double)r;",
                                      "s_e += (double)c * (double)c;"),
    "diag_sent_norm_from_c": ("s_g += (double)g_hat[j] * (double)g_hat[j];",
                              "s_g += (double)c * (double)c;"),
}


def _pins(golden_dir):
    yield lambda: ttopk.test_hand_cases(golden_dir)
    for s in range(6):
        yield lambda s=s: ttopk.test_brute_force_tiny(s)
    yield lambda: ttopk.test_invariants(1000, 10)
    yield lambda: tquant.test_hand_cases(golden_dir)
    for b in (1, 2, 4, 8):
        yield lambda b=b: tquant.test_packing_is_little_endian_bitstream(b)
    yield lambda: tquant.test_qsgd_sign_plane()
    yield lambda: tquant.test_qsgd_norm_within_tree_bound()
    for mode, bits in (("minmax", 8), ("qsgd", 2), ("tern", 2)):
        yield lambda m=mode, b=bits: tquant.test_error_feedback_identity(m, b)
    for mode in ("minmax", "qsgd", "tern"):
        yield lambda m=mode: tquant.test_stochastic_unbiased(m)
    yield lambda: tquant.test_hybrid_composition()
    yield lambda: tphilox.test_known_answer_vectors(golden_dir)
    yield lambda: tphilox.test_uniform_distribution()
    yield lambda: tpsgd.test_exact_low_rank_is_reconstructed()
    yield lambda: tpsgd.test_orthonormal_and_matches_numpy_qr()
    yield lambda: tagg.test_hand_cases(golden_dir)
    yield lambda: tagg.test_quant_hand_case(golden_dir)
    yield lambda: trandk.test_keep_set_is_the_philox_draw_below_p(1000, 0.1, 3, 0)
    yield lambda: trandk.test_limits()
    yield lambda: tlog.test_log_exp_accuracy()
    yield lambda: tlog.test_log_hand_case()
    yield lambda: tlog.test_diff_hand_case()
    yield lambda: tlog.test_refresh_is_plain_quantisation("minmax", 4)
    yield lambda: tlog.test_closed_loop_over_steps("qsgd", 4)
    yield lambda: tdiag.test_hand_case()
    yield lambda: tdiag.test_hybrid_matches_the_stored_residual(8, 64)


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, mutant_dir, golden_dir):
    old, new = MUTANTS[name]
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, "mutation site not unique: " + name
    d = os.path.join(str(mutant_dir), name)
    os.makedirs(d, exist_ok=True)
    msrc = os.path.join(d, "gc_oracle.c")
    open(msrc, "w").write(src.replace(old, new))
    mlib = os.path.join(d, "libgc_oracle.so")
    subprocess.run(["gcc", *obuild.CFLAGS, "-w", "-shared", msrc, "-o", mlib, "-lm"],
                   check=True)
    saved = (ofront._lib, obuild.LIB, obuild.SRC)
    caught = []
    try:
        ofront._lib = None
        obuild.LIB, obuild.SRC = mlib, msrc
        for pin in _pins(golden_dir):
            try:
                pin()
            except (AssertionError, ofront.OracleError):
                caught.append(pin)
                break
    finally:
        ofront._lib, obuild.LIB, obuild.SRC = saved
        shutil.rmtree(d, ignore_errors=True)
    assert caught, "no pin caught the mutant " + name
