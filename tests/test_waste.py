"""Pins of the waste accounting against the page's printed simulation and its closed form.

The closed form below is computed by enumerating every length of each
uniform component of the mix, independently of oracle.waste.
"""
import math
from fractions import Fraction

import synth
from golden_io import table
from oracle import waste

MIX = ((Fraction(7, 10), 32, 511), (Fraction(1, 4), 512, 2047), (Fraction(1, 20), 2048, 4095))


def _moments(block):
    """Exact E[len], E[paged slots], Var[len], Var[paged slots] of the mix."""
    e_len = e_pg = e_len2 = e_pg2 = Fraction(0)
    for w, lo, hi in MIX:
        n = hi - lo + 1
        s1 = sum(range(lo, hi + 1))
        s2 = sum(x * x for x in range(lo, hi + 1))
        p1 = sum(-(-x // block) * block for x in range(lo, hi + 1))
        p2 = sum((-(-x // block) * block) ** 2 for x in range(lo, hi + 1))
        e_len += w * Fraction(s1, n)
        e_len2 += w * Fraction(s2, n)
        e_pg += w * Fraction(p1, n)
        e_pg2 += w * Fraction(p2, n)
    return e_len, e_pg, e_len2 - e_len**2, e_pg2 - e_pg**2


def test_closed_form_values():
    e_len, e_pg, _, _ = _moments(16)
    assert e_len == Fraction(1327, 2)  # 663.5
    assert e_pg - e_len == Fraction(15, 2)  # tail waste averages 7.5 slots
    assert abs(float(1 - e_len / 4096) - 0.83801) < 1e-5
    assert abs(float(1 - e_len / e_pg) - 0.011177) < 1e-6
    assert abs(float(4096 / e_pg) - 6.1043) < 1e-4


def test_page_printout_is_a_plausible_draw():
    g, _ = table("waste_simulation.txt")
    n = int(g["N"][0])
    e_len, e_pg, var_len, _ = _moments(int(g["block"][0]))
    sigma_reserved = math.sqrt(float(var_len) / n) / 4096 * 100  # pp
    res = float(1 - e_len / 4096) * 100
    assert abs(float(g["reserved_waste_pct"][0]) - res) < 3 * sigma_reserved + float(g["print_resolution"][0])
    assert abs(float(g["paged_waste_pct"][0]) - float(1 - e_len / e_pg) * 100) < 0.3
    assert abs(float(g["concurrency"][0]) - float(4096 / e_pg)) < 0.35


def test_seeded_simulation_within_sampling_error():
    e_len, e_pg, var_len, var_pg = _moments(16)
    for seed in (1, 2, 3):
        lens = synth.lengths_mix(synth.stream_seed(280000 + seed, 1), 1000)
        r = waste.simulate(lens, 4096, 16)
        sig = math.sqrt(float(var_len) / 1000) / 4096
        assert abs(r["reserved_waste"] - float(1 - e_len / 4096)) < 3 * sig
        assert r["paged_waste"] < 0.04  # the pages: under 4 % with paging
        assert r["reserved_waste"] > 0.6  # the pages: 60-80 % or more reserved waste
        assert 0 <= r["paged"] - r["used"] <= 15 * 1000  # tail-only waste, < bs per request
        assert r["concurrency"] == r["reserved"] / r["paged"]
