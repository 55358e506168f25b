"""Plausible mistakes planted in copies of the oracle fail at least one pin.

Each mutant is the oracle's C source with one textual edit (a flipped index,
a dropped term, a wrong sign, a transposed operand, a wrong rounding rule),
compiled on the CPU into a temporary library. The unmodified oracle is never
touched. A mutant that passes every pin would mean the pins cannot see that
class of mistake.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    # gradX uses weight(k) instead of weight(W-1-k)
    "gradx_weight_not_flipped": ("* tab[w[(W - 1 - k) * H + h]];", "* tab[w[k * H + h]];"),
    # gradX drops its last tap
    "gradx_drops_a_tap": ("        for (int64_t r = 0; r < rows; ++r) {\n            int64_t i = r / B, j = r % B;\n            for (int64_t h = 0; h < H; ++h) {\n                double acc = 0.0;\n                for (int64_t k = 0; k < W; ++k)",
                          "        for (int64_t r = 0; r < rows; ++r) {\n            int64_t i = r / B, j = r % B;\n            for (int64_t h = 0; h < H; ++h) {\n                double acc = 0.0;\n                for (int64_t k = 0; k < W - 1; ++k)"),
    # gradWeight pairs x(i) with gradYMasked(i+k) instead of (i+W-1-k)
    "gradw_wrong_shift": ("gym(tab, gy, mask, S, B, H, i + W - 1 - k, j, h)", "gym(tab, gy, mask, S, B, H, i + k, j, h)"),
    # gradWeight subtracts its terms
    "gradw_wrong_sign": ("acc[k * H + h] += t;", "acc[k * H + h] -= t;"),
    # mask indexed [S,B] instead of [B,S]
    "mask_transposed": ("double m = mask ? (mask[j * S + i] ? 1.0 : 0.0) : 1.0;\n    return",
                        "double m = mask ? (mask[i * B + j] ? 1.0 : 0.0) : 1.0;\n    return"),
    # mask ignored
    "mask_ignored": ("double m = mask ? (mask[j * S + i] ? 1.0 : 0.0) : 1.0;\n    return",
                     "double m = 1.0;\n    return"),
    # gradY read as [B,S,H]
    "gy_layout_transposed": ("return m * tab[gy[(i * B + j) * H + h]];", "return m * tab[gy[(j * S + i) * H + h]];"),
    # last row of S treated as padding
    "boundary_off_by_one": ("if (i < 0 || i >= S)\n        return 0.0;", "if (i < 0 || i >= S - 1)\n        return 0.0;"),
    # ties round away from zero
    "ties_away_from_zero": ("if (d > 0.5 || (d == 0.5 && fmod(r, 2.0) != 0.0))", "if (d >= 0.5)"),
    # subnormals decoded one binade low
    "subnormal_decode": ("v = ldexp((double)m, f.emin - f.man_bits);", "v = ldexp((double)m, f.emin - f.man_bits - 1);"),
    # no gradual underflow when rounding
    "flush_subnormal_results": ("    if (E < f.emin)\n        E = f.emin;", "    if (E < f.emin)\n        return sign;"),
    # point-wise gradX with the weight not flipped
    "gradx_at_weight_not_flipped": ("acc += g * mcc1d_oracle_to_double(w[(W - 1 - k) * H + h], dtype);",
                                    "acc += g * mcc1d_oracle_to_double(w[k * H + h], dtype);"),
    # implied forward with the taps reversed (the transposition pins must see it)
    "forward_taps_reversed": ("int64_t s = t - (W - 1) + k;", "int64_t s = t - k;"),
    # sum|terms| of gradWeight summed with signs (no absolute value)
    "gradw_abs_signed": ("mag[k * H + h] += fabs(t);", "mag[k * H + h] += t;"),
    # sum|terms| taken over the unshifted pair gYm(i) * x(i) for every tap
    "gradw_abs_unshifted": ("mag[k * H + h] += fabs(t);",
                            "mag[k * H + h] += fabs(gym(tab, gy, mask, S, B, H, i, j, h) * "
                            "tab[x[(i * B + j) * H + h]]);"),
    # sum|terms| of the unmasked gradY (the mask left out of the scale only)
    "gradw_abs_unmasked": ("mag[k * H + h] += fabs(t);",
                           "mag[k * H + h] += fabs(gym(tab, gy, NULL, S, B, H, i + W - 1 - k, j, h) * "
                           "tab[x[(i * B + j) * H + h]]);"),
    # sum|terms| twice too large
    "gradw_abs_doubled": ("mag[k * H + h] += fabs(t);", "mag[k * H + h] += 2.0 * fabs(t);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as fh:
        src = fh.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.compile_oracle(str(mpath), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
