"""Mutation check of the oracle's pins: each plausible mistake, planted in a
copy of oracle.c (never in the real one), must make at least one pin fail."""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, mutated text): dropped terms, wrong signs/indices, transposed operands, off-by-one bounds
MUTANTS = [
    ("dense: no max shift", "double p = exp(xbuf[j - lo] - M);", "double p = exp(xbuf[j - lo]);"),
    ("dense: score sign", "double x = scale * dot;\n    xbuf[j - lo] = x;", "double x = -scale * dot;\n    xbuf[j - lo] = x;"),
    ("dense: q.v instead of q.k", "dot += q[c] * k[j * d + c];", "dot += q[c] * v[j * d + c];"),
    ("dense: no normalisation", "o[c] /= l;\n  *lse = M + log(l);", "\n  *lse = M + log(l);"),
    ("dense: lse without max", "*lse = M + log(l);", "*lse = log(l);"),
    ("split: overlapping chunks", "int64_t hi = ((c + 1) * Skv) / n_split;", "int64_t hi = ((c + 1) * Skv) / n_split + 1 < Skv ? ((c + 1) * Skv) / n_split + 1 : Skv;"),
    ("merge: weights against M", "double w = exp(lse_part[c * rows + r] - L);", "double w = exp(lse_part[c * rows + r] - M);"),
    ("pool: divide by block", "xp[t * d + c] = s / (double)(hi - lo);", "xp[t * d + c] = s / (double)block;"),
    ("route: mean over NKB+1", "m /= (double)NKB;", "m /= (double)(NKB + 1);"),
    ("route: sample variance", "var /= (double)NKB;", "var /= (double)(NKB - 1);"),
    ("route: strict threshold", "(s[j] >= th) || (j == jmax)", "(s[j] > th) || (j == jmax)"),
    ("route: no forced argmax", "(s[j] >= th) || (j == jmax)", "(s[j] >= th)"),
    ("route: beta sign", "m + beta * sd;", "m - beta * sd;"),
    ("taylor: weight sign", "double w = (double)nk[j] * (1.0 + s[j] - m);", "double w = (double)nk[j] * (1.0 - s[j] + m);"),
    ("taylor: block size dropped", "double w = (double)nk[j] * (1.0 + s[j] - m);", "double w = (1.0 + s[j] - m);"),
    ("taylor: expansion point shifted", "double w = (double)nk[j] * (1.0 + s[j] - m);",
     "double w = (double)nk[j] * (1.0 + s[j] - m - 0.05);"),
    ("taylor: pooled K instead of V", "const double* vb = vp + (bh * NKB + j) * d;", "const double* vb = kp + (bh * NKB + j) * d;"),
    ("sparse: factor sign", "double f = exp(mu[t] - M);", "double f = exp(M - mu[t]);"),
    ("sparse: Taylor mass missing in den", "den += f * W[t];", ""),
    ("sparse: Taylor missing in num", "o[c] += f * T[t * d + c];", ";"),
    ("na: window centred half a step late", "int64_t s = p - K / 2;", "int64_t s = p - (K - 1) / 2;"),
    ("na: low border reflected", "if (s < 0) s = 0;", "if (s < 0) s = -s;"),
    ("na: high border not shifted inward", "if (s > L - K) s = L - K;", "if (s > L - K) s = (L - K) / 2;"),
    ("na: one frame short", "for (int64_t tt = t0; tt < t0 + Kt; ++tt)", "for (int64_t tt = t0; tt < t0 + Kt - 1; ++tt)"),
    ("na: y-fastest raster order", "kbuf[n++] = (tt * Y + yy) * X + xx;", "kbuf[n++] = (tt * X + xx) * Y + yy;"),
    ("na: q.v instead of q.k", "dot += qrow[c] * kh[kbuf[j] * d + c];", "dot += qrow[c] * vh[kbuf[j] * d + c];"),
    ("na: lse without max", "lse[r] = M + log(l);", "lse[r] = log(l);"),
    ("e4m3: exponent bias 8", "(1.0 + m / 8.0) * ldexp(1.0, e - 7)", "(1.0 + m / 8.0) * ldexp(1.0, e - 8)"),
    ("e4m3: subnormal step 2^-10", "const double r = nearbyint(a * 512.0);", "const double r = nearbyint(a * 1024.0);"),
    ("e4m3: ties away from zero", "double r = nearbyint((m - 1.0) * 8.0);", "double r = round((m - 1.0) * 8.0);"),
    ("e4m3: truncation", "double r = nearbyint((m - 1.0) * 8.0);", "double r = floor((m - 1.0) * 8.0);"),
    ("e4m3: no saturation", "if (a >= 448.0) return sgn | 0x7e;", "if (a >= 480.0) return sgn | 0x7e;"),
    ("quant: scale over 240", "const float s = (float)(amax / 448.0);", "const float s = (float)(amax / 240.0);"),
    ("quant: quotient over 240", "(double)row[k] * 448.0 / amax", "(double)row[k] * 240.0 / amax"),
    ("quant: code from the float product with the rounded inverse scale", "(double)row[k] * 448.0 / amax",
     "(double)(row[k] * (448.0f / (float)amax))"),
    ("quant: code from the float quotient by the rounded scale", "(double)row[k] * 448.0 / amax",
     "(double)(row[k] / s)"),
    ("quant: subnormal scales kept", "if (!(s >= ldexp(1.0, -126))) {", "if (!(s > 0.0f)) {"),
    ("gemm: weight scale dropped", "const double f = (double)sa[m] * (double)sw[n];", "const double f = (double)sa[m];"),
    ("gemm: weight transposed", "lut[wq[n * K + k]]", "lut[wq[(k % N) * K + (n % K)]]"),
    ("na: no normalisation", "o[c] /= l;\n      lse[r] = M + log(l);", "\n      lse[r] = M + log(l);"),
]

PINS = [
    lambda: pins.test_dense_matches_library_sdpa(1, 2, 33, 57, 64),
    pins.test_dense_two_keys_closed_form,
    pins.test_dense_identical_keys_give_mean_value,
    pins.test_dense_large_scores_are_stable_and_one_hot,
    pins.test_dense_rows_sum_to_one_before_v,
    lambda: pins.test_split_merge_equals_unsplit(257, 3),
    pins.test_merge_closed_form_two_partials,
    lambda: pins.test_pool_matches_numpy_mean(300, 64),
    lambda: pins.test_route_matches_brute_force_enumeration(256, 64, 64, 0.5),
    pins.test_route_constant_keys_zero_sigma_selects_all,
    pins.test_route_density_monotone_in_beta_and_argmax_kept,
    pins.test_sparse_beta_minus_inf_equals_dense_bitwise,
    pins.test_sparse_without_taylor_equals_masked_library_attention,
    pins.test_taylor_hand_derived_closed_form,
    pins.test_taylor_constant_v_and_unit_mass,
    pins.test_taylor_term_converges_quadratically_to_exact_attention,
    lambda: pins.test_na3d_matches_masked_library_attention(*pins.NA_CASES[0]),
    lambda: pins.test_na3d_matches_masked_library_attention(*pins.NA_CASES[1]),
    lambda: pins.test_na3d_window_indicator(*pins.NA_CASES[0]),
    pins.test_na3d_single_token_window_returns_own_value,
    lambda: pins.test_na3d_mirror_symmetry_odd_window(0),
    pins.test_e4m3_decode_matches_library_for_every_code,
    pins.test_e4m3_encode_round_trips_every_finite_code,
    pins.test_e4m3_encode_matches_library_conversion,
    pins.test_e4m3_encode_saturates,
    pins.test_e4m3_encode_is_the_nearest_value_ties_to_even,
    pins.test_quantize_rows_error_bound_and_row_max,
    pins.test_quantize_rows_codes_are_the_exact_quotients_nearest_value,
    pins.test_fp8_gemm_matches_library_matmul_of_decoded_operands,
]


def caught(pin):
    try:
        pin()
    except Exception:
        return True
    return False


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory() as d:
        yield d
    oracle._swap_library(None)


def test_unmutated_copy_passes_every_pin(workdir):
    lib = os.path.join(workdir, "orig.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", SRC, "-o", lib, "-lm"], check=True)
    oracle._swap_library(lib)
    try:
        assert not any(caught(p) for p in PINS)
    finally:
        oracle._swap_library(None)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught_by_a_pin(workdir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {name}"
    path = os.path.join(workdir, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(workdir, f"mutant_{abs(hash(name))}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", path, "-o", lib, "-lm"], check=True)
    oracle._swap_library(lib)
    try:
        assert any(caught(p) for p in PINS), f"no pin catches the mutant '{name}'"
    finally:
        oracle._swap_library(None)
