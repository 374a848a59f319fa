"""Pins of ``oracle.valid_sets``, the near-tie rule of the routing check.

The parity rule fixes which expert sets count as correct when a token's K-th and
(K+1)-th probabilities nearly tie: experts above p_K + tol*S must be chosen (S = the
mass of the K largest probabilities), and the remaining slots may hold any experts
within tol*S of p_K, both bounds inclusive.  The pins below are hand-built probability
vectors whose values are dyadic rationals, so every comparison at a band edge is
exact, and the expected sets are written out by hand.  Two planted mistakes (the band
without the factor S, and the must-choose set built with >=) must each fail a pin.
"""
from __future__ import annotations

import numpy as np
import pytest

from oracle import Oracle, valid_choices, valid_sets
from synth import Dims

K = 8
TOL = 2.0 ** -13          # a power of two, so that tol * S is exact for dyadic S


def _vec(head, tail_len=8, tail=2.0 ** -12):
    """Descending probabilities: `head` then `tail_len` copies of a small value; expert
    ids are 100 + rank, so a set is readable as ranks."""
    ps = np.array(list(head) + [tail] * tail_len, np.float64)
    assert np.all(np.diff(ps) <= 0)
    order = np.arange(len(ps)) + 100
    return ps, order


def _ranks(sets):
    return [sorted(e - 100 for e in s) for s in sets]


def _own(order):
    return list(order[:K])


def _top6(mass):
    """Six dyadic probabilities, well separated, summing to `mass`."""
    return [mass * v for v in (0.25, 0.1875, 0.1875, 0.125, 0.125, 0.125)]


def check_exact_tie(vs):
    # p8 == p9 exactly; p7 and p10 far away: the own set and the one that swaps ranks 7 and 8
    p8 = 2.0 ** -5
    head = _top6(1.0 - 2.0 ** -4 - p8) + [2.0 ** -4, p8, p8]
    ps, order = _vec(head)
    assert abs(ps[:K].sum() - 1.0) == 0.0
    got = _ranks(vs(ps, order, _own(order), K, TOL))
    assert got == [list(range(8)), [0, 1, 2, 3, 4, 5, 6, 8]], got


def check_three_way_band(vs):
    # ranks 6, 7, 8 all within tol*S of p_K = ps[7]; rank 9 far below: 6 sure experts,
    # 2 slots from a band of 3 -> the 3 pairs
    p8 = 2.0 ** -5
    e = TOL / 2
    head = _top6(1.0 - (p8 + e) - p8) + [p8 + e, p8, p8 - e]
    ps, order = _vec(head)
    S = ps[:K].sum()
    assert S == 1.0
    got = _ranks(vs(ps, order, _own(order), K, TOL))
    assert sorted(got) == sorted([list(range(8)), [0, 1, 2, 3, 4, 5, 6, 8], [0, 1, 2, 3, 4, 5, 7, 8]]), got


def check_band_edges_inclusive(vs):
    # p7 = p8 + tol*S and p9 = p8 - tol*S exactly: both lie in the band (inclusive), so
    # rank 6 is not a must-choose expert and rank 8 may replace either of ranks 6, 7
    p8 = 2.0 ** -5
    head = _top6(1.0 - (p8 + TOL) - p8) + [p8 + TOL, p8, p8 - TOL]
    ps, order = _vec(head)
    assert ps[:K].sum() == 1.0
    got = _ranks(vs(ps, order, _own(order), K, TOL))
    assert sorted(got) == sorted([list(range(8)), [0, 1, 2, 3, 4, 5, 6, 8], [0, 1, 2, 3, 4, 5, 7, 8]]), got


def check_just_outside_band(vs):
    # p9 = p8 - tol*S - 2^-20: outside the band, only the own set is valid
    p8 = 2.0 ** -5
    head = _top6(1.0 - 2.0 ** -4 - p8) + [2.0 ** -4, p8, p8 - TOL - 2.0 ** -20]
    ps, order = _vec(head)
    got = _ranks(vs(ps, order, _own(order), K, TOL))
    assert got == [list(range(8))], got


def check_band_scales_with_mass(vs):
    # S = 1/2 (the top-8 hold half the mass): the band is tol*S = 2^-14; p9 sits 1.5 *
    # 2^-14 below p8, outside it (a band of tol, without S, would take it in)
    p8 = 2.0 ** -6
    d = 1.5 * 2.0 ** -14
    head = _top6(0.5 - 2.0 ** -5 - p8) + [2.0 ** -5, p8, p8 - d]
    ps, order = _vec(head, tail_len=40, tail=(0.5 - (p8 - d)) / 40)
    assert ps[:K].sum() == 0.5
    got = _ranks(vs(ps, order, _own(order), K, TOL))
    assert got == [list(range(8))], got
    # and 0.5 * 2^-14 below p8 it is inside
    head = _top6(0.5 - 2.0 ** -5 - p8) + [2.0 ** -5, p8, p8 - 2.0 ** -15]
    ps, order = _vec(head, tail_len=40, tail=(0.5 - p8) / 40 * 0.5)
    got = _ranks(vs(ps, order, _own(order), K, TOL))
    assert got == [list(range(8)), [0, 1, 2, 3, 4, 5, 6, 8]], got


def check_no_tie_single_set(vs):
    # well-separated probabilities: one valid set, the own one
    head = _top6(1.0 - 2.0 ** -4 - 2.0 ** -5) + [2.0 ** -4, 2.0 ** -5, 2.0 ** -7]
    ps, order = _vec(head)
    assert _ranks(vs(ps, order, _own(order), K, TOL)) == [list(range(8))]


PINS = [check_exact_tie, check_three_way_band, check_band_edges_inclusive, check_just_outside_band,
        check_band_scales_with_mass, check_no_tie_single_set]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_valid_sets_pins(pin):
    pin(valid_sets)


@pytest.mark.parametrize("mutant", [1, 2], ids=["band without S", "must-choose set with >="])
def test_valid_sets_mutants_caught(mutant):
    caught = []
    for pin in PINS:
        try:
            pin(lambda *a, **k: valid_sets(*a, mutant=mutant, **k))
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches valid_sets mutant {mutant}"


def test_valid_choices_from_logits_exact_tie():
    """Through the oracle's own routing of fp32 logits: two experts with equal logits at
    the top-8 boundary are interchangeable, and the oracle's own set (lowest index on the
    tie) comes first."""
    d = Dims(hidden=64, n_experts=16, top_k=8, inter=32, shared_inter=32, group=32)
    logits = np.full(16, -4.0, np.float32)
    logits[[0, 1, 2, 3, 4, 5, 6]] = [3.0, 2.5, 2.0, 1.5, 1.0, 0.5, 0.25]
    logits[[9, 12]] = 0.0                      # tie for the 8th slot
    sets = valid_choices(Oracle(), d, logits)
    assert [sorted(s) for s in sets] == [[0, 1, 2, 3, 4, 5, 6, 9], [0, 1, 2, 3, 4, 5, 6, 12]]
    assert list(sets[0])[-1] == 9
