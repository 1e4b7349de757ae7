"""Plant plausible mistakes in a copy of the oracle, on the CPU, and check
that the pin battery catches every one of them (no GPU).

Each mutant is a one-line textual change to arf_oracle.c compiled into a
temporary library; the real source is untouched.
"""
import os

import pytest

import oracle
import pins

MUTANTS = {
    "mean_over_H_minus_1": ("ss / (double)H", "ss / (double)(H - 1)"),
    "eps_outside_root": ("1.0 / sqrt(ss / (double)H + (double)eps)", "1.0 / (sqrt(ss / (double)H) + (double)eps)"),
    "no_sqrt": ("1.0 / sqrt(ss / (double)H + (double)eps)", "1.0 / (ss / (double)H + (double)eps)"),
    "round_sum_before_residual": (
        "float t = acc + arf_oracle_widen(dtype, R[rb + i]);",
        "float t = arf_oracle_widen(dtype, arf_oracle_narrow_f32(dtype, acc)) + arf_oracle_widen(dtype, R[rb + i]);"),
    "low_precision_running_sum": (
        "acc = acc + partial_at(partials[r], pdtype, dtype, pb + i);",
        "acc = arf_oracle_widen(dtype, arf_oracle_narrow_f32(dtype, acc + partial_at(partials[r], pdtype, dtype, pb + i)));"),
    "reversed_rank_order": ("for (int r = 0; r < W; ++r) acc", "for (int r = W - 1; r >= 0; --r) acc"),
    "dropped_last_rank": ("for (int r = 0; r < W; ++r) acc", "for (int r = 0; r < W - (W > 1); ++r) acc"),
    "residual_sign": ("float t = acc + arf_oracle_widen", "float t = acc - arf_oracle_widen"),
    "gamma_reversed": ("G[i]", "G[H - 1 - i]"),
    "residual_row_stride_ignored": ("const int64_t rb = m * ld_residual", "const int64_t rb = m * H"),
    "partial_row_stride_ignored": ("const int64_t pb = m * ld_partials", "const int64_t pb = m * H"),
    "f32_partials_read_as_16_bit": ("if (pdtype == 2) return ((const float*)p)[i];", ""),
    "gamma_dropped": ("x * inv * g", "x * inv"),
    "x_misread_in_norm": (
        "double x = (double)arf_oracle_widen(dtype, RO[rob + i]);",
        "double x = (double)arf_oracle_widen(dtype, RO[rob + i]) * (1.0 + 1e-3 * (i == 0));"),
    "ties_away_from_zero": ("(rem == 0.5 && fmod(kf, 2.0) != 0.0)", "(rem == 0.5)"),
    "truncating_narrow": ("if (rem > 0.5 || (rem == 0.5 && fmod(kf, 2.0) != 0.0)) kf += 1.0;", ""),
    "overflow_one_binade_early": ("if (E > f->emax) return sign | inf;", "if (E >= f->emax) return sign | inf;"),
    "f16_subnormal_scale": ("v = ldexp((double)man, -24);", "v = ldexp((double)man, -25);"),
    "f16_normal_bias": ("(int)ex - 25", "(int)ex - 24"),
    "double_rounding_out": (
        "O[ob + i] = arf_oracle_narrow_f64(dtype, x * inv * g);",
        "O[ob + i] = arf_oracle_narrow_f32(dtype, (float)(x * inv * g));"),
    "subnormal_quantum_unclamped": ("if (E < f->emin) E = f->emin;", ""),
    "nan_becomes_inf": ("if (isnan(v)) return sign | f->qnan;", ""),
}


@pytest.fixture(scope="module")
def src():
    return open(oracle.SRC).read()


def test_real_oracle_passes_quick_battery():
    pins.run_battery(oracle.default(), quick=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, src, tmp_path):
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found in the oracle source"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_oracle(str(path), str(tmp_path / f"lib_{name}.so"))
    mutant = oracle.Oracle(so)
    with pytest.raises(AssertionError):
        pins.run_battery(mutant, quick=True)
