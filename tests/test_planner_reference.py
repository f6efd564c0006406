"""Pins for the planner reference against the pages' printed grid arithmetic.

Source: "Kimi K3 decode on 2x8 B200: DP16 vs DP2 x DCP8", section "MLA: bytes
conserved, DP16 kernel slowed by wave quantisation" (figures in
tests/golden/pages_wave_arithmetic.json).
"""
import json
import os

import pytest

from oracle import planner as ref

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "pages_wave_arithmetic.json")))


def test_split_rule_reproduces_the_pages():
    n = GOLD["split_is_one_for_B_at_least"]
    for B in range(n, 129):
        assert ref.pages_heuristic_split(B, 5) == 1
    assert ref.pages_heuristic_split(n - 1, 5) > 1
    # small batches get more splits, capped at 32
    assert ref.pages_heuristic_split(1, 5) == 14
    assert ref.pages_heuristic_split(1, 1) == 32


@pytest.mark.parametrize("case", GOLD["grids"], ids=lambda c: c["what"][:24])
def test_grid_and_wave_counts_reproduce_the_pages(case):
    split = ref.pages_heuristic_split(case["B"], case["q_len"])
    assert split == case["split"]
    ctas, waves = ref.pages_waves(case["B"], case["q_len"], split, GOLD["sms"])
    assert ctas == case["ctas"]
    if "excess_over_sms" in case:
        assert ctas - GOLD["sms"] == case["excess_over_sms"]
    if "grid_y" in case:
        assert ref.pages_grid(case["B"], case["q_len"], split)[1] == case["grid_y"]
    if "waves" in case:
        assert round(waves, 2 if case["waves"] < 2 else 1) == case["waves"]


@pytest.mark.parametrize("est", GOLD["wave_rounded_estimates_us"], ids=lambda e: str(e["B"]))
def test_wave_rounded_estimates_scale_by_cta_count(est):
    ctas, _ = ref.pages_waves(est["B"], est["q_len"], 1, GOLD["sms"])
    us = GOLD["single_cta_scan_us"] * ctas / GOLD["sms"]
    assert abs(us - est["us"]) < 1.0


def test_brute_force_plan_fills_whole_waves_for_uniform_batches():
    # 38 cluster slots (152 SMs / 4), 96 heads x q_len 5 = 480 rows = 2 row
    # units of 256: 38 = 2 x 19, so 19 splits give exactly B waves for any B.
    for B in (1, 2, 4, 8, 12, 16, 20, 24):
        for L in (100_000, 400_000):
            S, eff, _ = ref.plan([L] * B, 96, 5, slots=38)
            assert eff >= 0.9, (B, L, S, eff)


def test_makespan_is_list_scheduling():
    assert ref.makespan([3, 3, 3], 2) == 6
    assert ref.makespan([5, 1, 1, 1, 1, 1], 2) == 5
    assert ref.makespan([], 4) == 0
    costs = ref.unit_costs([128], 96, 5, 2, c0=0)
    assert costs == [1] * 4  # 2 pages dealt 1 + 1, two row units each
    assert ref.unit_costs([128], 96, 5, 2, c0=0, rows_per_unit=128) == [1] * 8
