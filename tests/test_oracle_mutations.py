"""The pins of test_oracle_pins.py catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped or
wrong term, sign, shift, index, rounding mode), compiles it on the host and
runs every pin against it: at least one pin must fail.  Nothing here touches
a GPU."""
import inspect

import pytest

import oracle
import test_oracle_pins as pins
from conftest import page_facts

MUTANTS = {
    "q6k high-bit shift": ("(blk[128 + half * 32 + l] >> (2 * g)) & 3",
                           "(blk[128 + half * 32 + l] >> (2 * (g ^ 1))) & 3"),
    "q6k nibble choice": ("(g < 2) ? (qlb & 0x0f) : (qlb >> 4)", "(g < 2) ? (qlb >> 4) : (qlb & 0x0f)"),
    "q6k ql byte address": ("blk[half * 64 + (g & 1) * 32 + l]", "blk[half * 64 + (g >> 1) * 32 + l]"),
    "q6k offset": ("return (lo | (hi << 4)) - 32;", "return (lo | (hi << 4)) - 31;"),
    "q6k scale index": ("q6k_scale(blk, e >> 4)", "q6k_scale(blk, e >> 5)"),
    "q6k gemv scale index": ("q6k_scale(blk, s) * d8v", "q6k_scale(blk, s ^ 1) * d8v"),
    "q6k gemv activation scale index": ("d8[(size_t)b * 8 + s / 2]", "d8[(size_t)b * 8 + s / 4]"),
    "q6k gemv activation index": ("q8[(size_t)b * QK + e];\n                const double d8v",
                                  "q8[(size_t)b * QK + (e ^ 1)];\n                const double d8v"),
    "q6k f32 activation index": ("(double)x[(size_t)b * QK + e]", "(double)x[(size_t)b * QK + (e ^ 1)]"),
    "q6k f32 scale index": ("const double w = d * (double)q6k_scale(blk, e >> 4)",
                            "const double w = d * (double)q6k_scale(blk, e >> 5)"),
    "q6k f32 dropped block scale": ("const double w = d * ", "const double w = 1.0 * "),
    "q8 rounding mode": ("int q = (int)rintf(p);", "int q = (int)roundf(p);"),
    "q8 scale divisor": ("const float d = am / 127.0f;", "const float d = am / 128.0f;"),
    "q8 dropped clamp+sum": ("        s += q;\n", ""),
    "q4k min sign": ("acc += t1 - t2;", "acc += t1 + t2;"),
    "q4k dequant min sign": ("(double)q4k_q(blk, e) - dmin * (double)m",
                             "(double)q4k_q(blk, e) + dmin * (double)m"),
    "q4k high scale bits": ("*sc = (s[k + 4] & 15) | ((s[k - 4] >> 6) << 4);",
                            "*sc = (s[k + 4] & 15) | ((s[k - 4] >> 6) << 3);"),
    "q4k min bits swapped": ("*m = (s[k + 4] >> 4) | ((s[k] >> 6) << 4);",
                             "*m = (s[k + 4] & 15) | ((s[k] >> 6) << 4);"),
    "q4k nibble order": ("(k & 1) ? (byte >> 4) : (byte & 0x0f)", "(k & 1) ? (byte & 0x0f) : (byte >> 4)"),
    "q4k dropped min term": ("acc += t1 - t2;", "acc += t1;"),
    "q5k fifth-bit index": ("16 * ((blk[16 + l] >> k) & 1)", "16 * ((blk[16 + l] >> (k ^ 1)) & 1)"),
    "q5k fifth-bit weight": ("16 * ((blk[16 + l] >> k) & 1)", "32 * ((blk[16 + l] >> k) & 1)"),
    "q5k qh offset": ("16 * ((blk[16 + l] >> k) & 1)", "16 * ((blk[17 + (l & 15)] >> k) & 1)"),
    "q5k qs offset": ("blk[48 + 32 * (k >> 1) + l]", "blk[16 + 32 * (k >> 1) + l]"),
    "q5k gemv min sign": ("isum += q5k_q(blk, e) * xv;\n                    qsum += xv;",
                          "isum += q5k_q(blk, e) * xv;\n                    qsum -= xv;"),
    "rms eps outside root": ("sqrt(ss / (double)n + (double)eps)", "(sqrt(ss / (double)n) + (double)eps)"),
    "rms sum not mean": ("sqrt(ss / (double)n + (double)eps)", "sqrt(ss + (double)eps)"),
    "swiglu sign": ("exp(-gv)", "exp(gv)"),
    "f16 truncates": ("const float m = rintf(ldexpf(a, 10 - e));", "const float m = floorf(ldexpf(a, 10 - e));"),
    "f16 subnormal scale": ("v = ldexpf((float)man, -24);", "v = ldexpf((float)man, -23);"),
}


def all_pins():
    return [(n, f) for n, f in inspect.getmembers(pins, inspect.isfunction) if n.startswith("test_")]


def run_pin(fn, facts):
    kwargs = {}
    params = inspect.signature(fn).parameters
    if "orc" in params:
        kwargs["orc"] = oracle
    if "facts" in params:
        kwargs["facts"] = facts
    fn(**kwargs)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source()
    assert src.count(old) >= 1, f"mutation site for {name!r} not found"
    facts = page_facts()
    caught = []
    with oracle.variant(src.replace(old, new, 1), str(tmp_path)):
        for pin_name, fn in all_pins():
            try:
                run_pin(fn, facts)
            except (AssertionError, ValueError, OverflowError):
                caught.append(pin_name)
    assert caught, f"no pin caught the planted mistake: {name}"


def test_unmutated_oracle_passes_every_pin(tmp_path):
    facts = page_facts()
    with oracle.variant(oracle.source(), str(tmp_path)):
        for _, fn in all_pins():
            run_pin(fn, facts)
