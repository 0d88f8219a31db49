"""The oracle's pins must catch plausible mistakes.

Each case copies ``oracle.c``, plants one mistake (a dropped term, a wrong
sign, a wrong index or bound, a transposed operand, a wrong tie-break),
compiles the copy on the CPU and runs the pin battery of
``tests/oracle_checks.py`` against it: at least one pin must fail.  The
oracle itself is never modified.
"""
import os
import tempfile

import pytest

import oracle
from tests import oracle_checks as oc

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "topk_tie_break": ("if (best < 0 || s[e] > s[best]) best = e;",
                       "if (best < 0 || s[e] >= s[best]) best = e;"),
    "softmax_sign": ("v[k] = expf(s[ids[(size_t)t * K + k]] - m);",
                     "v[k] = expf(m - s[ids[(size_t)t * K + k]]);"),
    "sigmoid_sign": ("v[k] = sigmoidf_(s[ids[(size_t)t * K + k]]);",
                     "v[k] = sigmoidf_(-s[ids[(size_t)t * K + k]]);"),
    "bias_dropped": ("s[e] = bias ? v + bias[e] : v;", "s[e] = v;"),
    "scan_inclusive": ("int p = group_offsets[e] + seen[e];",
                       "int p = group_offsets[e + 1] - 1 - seen[e];"),
    "permute_wrong_row": ("memcpy(xs + (size_t)p * D, x + (size_t)t * D,",
                          "memcpy(xs + (size_t)p * D, x + (size_t)(t / K) * D,"),
    "fc1_transposed_wi": ("for (int n = 0; n < N; ++n) a[n] = a[n] + xv * BF(wr[n]);",
                          "for (int n = 0; n < N; ++n) a[n] = a[n] + xv * BF(W[((size_t)n * D + d) % ((size_t)D * N)]);"),
    "swiglu_no_sigmoid": ("h[(size_t)r * F + f] = RN((g * sigmoidf_(g)) * u);",
                          "h[(size_t)r * F + f] = RN(g * u);"),
    "swiglu_gate_up_swapped": ("float g = a[f], u = a[F + f];", "float g = a[F + f], u = a[f];"),
    "expert_search_off_by_one": ("      while (offs[e + 1] <= r) ++e;\n      const uint16_t* W = wo + (size_t)e * F * D;\n      for (int d = 0; d < D; ++d) a[d] = 0.0f;",
                                 "      while (offs[e + 1] < r) ++e;\n      const uint16_t* W = wo + (size_t)e * F * D;\n      for (int d = 0; d < D; ++d) a[d] = 0.0f;"),
    "combine_weight_dropped": ("acc = acc + wk * BF(ys[(size_t)p * D + d]);",
                               "acc = acc + BF(ys[(size_t)p * D + d]);"),
    "combine_bwd_weight_dropped": ("dys[(size_t)p * D + d] = RN(wk * g);",
                                   "dys[(size_t)p * D + d] = RN(g);"),
    "dw_wrong_slot": ("acc = acc + g * BF(ys[(size_t)p * D + d]);",
                      "acc = acc + g * BF(ys[(size_t)pos[(size_t)t * K] * D + d]);"),
    "swiglu_bwd_term_dropped": ("*dgate = ((dh * u) * s) * (1.0f + g * (1.0f - s));",
                                "*dgate = ((dh * u) * s);"),
    "swiglu_bwd_sign": ("*dgate = ((dh * u) * s) * (1.0f + g * (1.0f - s));",
                        "*dgate = ((dh * u) * s) * (1.0f + g * (s - 1.0f));"),
    "fc2_dlhs_transposed_wo": ("acc = acc + BF(dys[(size_t)r * D + d]) * BF(W[(size_t)f * D + d]);",
                               "acc = acc + BF(dys[(size_t)r * D + d]) * BF(W[((size_t)d * F + f) % ((size_t)F * D)]);"),
    "dwo_first_row_dropped": ("for (int r = offs[e]; r < offs[e + 1]; ++r) {\n            float hv",
                              "for (int r = offs[e] + 1; r < offs[e + 1]; ++r) {\n            float hv"),
    "dwi_uses_wrong_operand": ("float xv = BF(xs[(size_t)r * D + d]);\n            for (int n = 0; n < N; ++n) a[n] = a[n] + xv * BF(dz[(size_t)r * N + n]);",
                               "float xv = BF(xs[(size_t)r * D + d]);\n            for (int n = 0; n < N; ++n) a[n] = a[n] + xv * BF(dz[(size_t)r * N + (n % F)]);"),
    "dxs_gate_half_only": ("for (int n = 0; n < N; ++n) acc = acc + BF(dz[(size_t)r * N + n]) * BF(W[(size_t)d * N + n]);",
                           "for (int n = 0; n < F; ++n) acc = acc + BF(dz[(size_t)r * N + n]) * BF(W[(size_t)d * N + n]);"),
    "bf16_round_half_up": ("u += 0x7fffu + lsb;", "u += 0x8000u;"),
    "mx_emax_7": ("const int s = (ex - 1) - 8;", "const int s = (ex - 1) - 7;"),
    "e4m3_ties_away": ("double m = nearbyint(ldexp(a, 3 - E));",
                       "double m = floor(ldexp(a, 3 - E) + 0.5);"),
    "e4m3_subnormal_spacing": ("const double m = nearbyint(a * 512.0);",
                               "const double m = nearbyint(a * 1024.0);"),
    "e4m3_bias_8": ("ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 11)"),
    "mx_dequant_scale_dropped": ("out[i] = ldexp(oracle_e4m3_to_f64(q[i]), (int)sc[i / 32] - 127);",
                                 "out[i] = oracle_e4m3_to_f64(q[i]);"),
    "mx_scale_block_index": ("(int)sc[i / 32] - 127", "(int)sc[i / 64] - 127"),
    "mx_fc1_gate_up_swapped": ("const double g = a[f], u = a[F + f];",
                               "const double g = a[F + f], u = a[f];"),
    "mx_fc2_first_expert_only": ("const size_t wrow = (size_t)e * D + d;",
                                 "const size_t wrow = (size_t)0 * D + d;"),
    "mx_zero_block_scale": ("if (amax == 0.0) return -127;", "if (amax == 0.0) return 0;"),
    "mx_z_gate_up_swapped": ("z[(size_t)r * N + n] = RN((float)a[n]);",
                             "z[(size_t)r * N + n] = RN((float)a[(n + F) % N]);"),
    "mx_tok_short_block_dropped": ("boff[e + 1] = boff[e] + (offs[e + 1] - offs[e] + 31) / 32;",
                                   "boff[e + 1] = boff[e] + (offs[e + 1] - offs[e]) / 32;"),
    "mx_tok_block_origin_global": ("const int r0 = offs[e] + 32 * (gb - boff[e]);",
                                   "const int r0 = 32 * (offs[e] / 32) + 32 * (gb - boff[e]);"),
    "mx_tok_scale_axis": ("sc[(size_t)gb * C + c] = (uint8_t)(s + 127);",
                          "sc[((size_t)c * NB + gb) % ((size_t)NB * C)] = (uint8_t)(s + 127);"),
    "mx_wgrad_block_index": ("(size_t)((r - offs[e]) / 32)", "(size_t)((r - offs[e]) / 64)"),
    "mx_wgrad_first_row_dropped": ("for (int r = offs[e]; r < offs[e + 1]; ++r) {\n          const size_t blk",
                                   "for (int r = offs[e] + 1; r < offs[e + 1]; ++r) {\n          const size_t blk"),
    "mx_wgrad_b_scale_one_column": ("p2[bsc[blk * Cb + j]]", "p2[bsc[blk * Cb]]"),
    "mx_dgrad_gate_up_swapped": ("swiglu_bwd_one((float)acc, BF(z[(size_t)r * 2 * F + f]), BF(z[(size_t)r * 2 * F + F + f]),",
                                 "swiglu_bwd_one((float)acc, BF(z[(size_t)r * 2 * F + F + f]), BF(z[(size_t)r * 2 * F + f]),"),
    "mx_dgrad_wrong_expert": ("const size_t wrow = (size_t)e * F + f;",
                              "const size_t wrow = (size_t)((e + 1) % E) * F + f;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    mutated = src.replace(old, new, 1)
    csrc = tmp_path / "oracle_mut.c"
    csrc.write_text(mutated)
    so = oracle.build(force=True, src=str(csrc), out=str(tmp_path / "liboracle_mut.so"))
    failed = []
    with oracle.using_library(so):
        for check in oc.ALL_CHECKS:
            try:
                check(oracle)
            except AssertionError:
                failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake '{name}'"
