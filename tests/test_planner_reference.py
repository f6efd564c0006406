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


# ------------------------------------------------- work-balanced scheduler
def _opt_makespan(costs, m):
    """Optimal makespan of independent jobs on m identical slots, by
    enumerating every assignment (tiny cases only)."""
    import itertools
    best = float("inf")
    for assign in itertools.product(range(m), repeat=len(costs)):
        load = [0.0] * m
        for c, k in zip(costs, assign):
            load[k] += c
        best = min(best, max(load))
    return best


def test_lpt_order_is_longest_first_then_by_id():
    units = [(0, 3.0), (1, 5.0), (2, 3.0), (3, 1.0), (4, 5.0)]
    assert [i for i, _ in ref.lpt_order(units)] == [1, 4, 0, 2, 3]


def test_lpt_list_schedule_meets_grahams_bound():
    """Graham's bound for longest-processing-time-first list scheduling:
    makespan <= (4/3 - 1/(3m)) x optimum.  Launch order alone misses it on
    the first case (short jobs first, the long one last)."""
    import random
    cases = [([1, 1, 1, 1, 4], 2)]
    rng = random.Random(5)
    for _ in range(60):
        m = rng.choice([2, 3])
        cases.append(([rng.randint(1, 20) for _ in range(rng.randint(2, 8))], m))
    for costs, m in cases:
        units = [(i, float(c)) for i, c in enumerate(costs)]
        lpt = ref.makespan([c for _, c in ref.lpt_order(units)], m)
        opt = _opt_makespan(costs, m)
        assert lpt <= (4 / 3 - 1 / (3 * m)) * opt + 1e-9, (costs, m)
    assert ref.makespan([1, 1, 1, 1, 4], 2) == 6 > (4 / 3 - 1 / 6) * 4


def test_sched_work_list_is_a_longest_first_permutation():
    lens = [1198, 152649, 2686, 60048, 10681, 170646, 4569, 25096, 1586]
    S, bnd, work, eff, ms = ref.plan_sched(lens, 96, 5, 76, rows_per_unit=128)
    U = 4
    assert sorted(work) == list(range(len(lens) * S * U))
    P = [-(-L // 64) for L in lens]
    cost = dict(ref.parts_units(P, U, S, bnd, 32.0))
    seq = [cost[i] for i in work]
    assert all(a >= b for a, b in zip(seq, seq[1:]))
    # the list-scheduling makespan of that order is the reported one
    assert ref.makespan(seq, 76) == ms
    for L, row in zip(lens, bnd):
        assert row[0] == 0 and row[-1] == -(-L // 64)
        assert all(a <= b for a, b in zip(row, row[1:]))


def test_sched_shortens_a_ragged_batch():
    """24 requests of 1k..200k tokens (log-uniform) on 76 two-CTA slots:
    taking the longest units first shortens the modelled makespan well below
    the part-major launch order's, and within 15% of the average load."""
    import numpy as np
    rng = np.random.default_rng(0)
    lens = [int(x) for x in np.exp(rng.uniform(np.log(1_000), np.log(200_000), 24))]
    _, _, _, ms_parts = ref.plan_parts(lens, 96, 5, 76, rows_per_unit=128)
    S, bnd, work, eff, ms = ref.plan_sched(lens, 96, 5, 76, rows_per_unit=128)
    avg = sum(-(-L // 64) for L in lens) * 4 / 76
    assert ms < 0.9 * ms_parts
    assert ms < 1.15 * (avg + 32 * len(work) / 76)


# ------------------------------------ the plan's quality, pinned from outside
def _lower_bound(lens, H, q_len, slots, c0=32.0, lam=1.0, s_max=64, rows_per_unit=256):
    """A closed-form lower bound on the scheduler's objective over every
    per-request split table with up to s_max parts (not only the planner's
    candidate families): with S parts per request, the units cost at least
    U * sum_v (P_v + S c0) in total, spread over `slots` slots, and the part
    holding a request's largest share costs at least ceil(P_v / S) + c0; add
    the objective's split term lam * S * rows / 1024."""
    U = -(-H * q_len // rows_per_unit)
    P = [-(-L // 64) for L in lens]
    rows = len(lens) * q_len * H
    best = float("inf")
    for S in range(1, s_max + 1):
        total = U * sum(p + S * c0 for p in P)
        ms = max(total / slots, max(-(-p // S) + c0 for p in P))
        best = min(best, ms + lam * S * rows / 1024.0)
    return best


# The bound treats work as fluid; with 40 or 48 row-unit jobs of one request
# each on 36 slots (B = 20, 24 at 100k) no split table reaches it (a denser
# search of capped tables, below, gets within 1.5% of the scheduler there).
_LOOSE = {(20, 100_000): 1.11, (24, 100_000): 1.04}


@pytest.mark.parametrize("B", [1, 2, 4, 8, 12, 16, 20, 24])
@pytest.mark.parametrize("L", [100_000, 400_000])
def test_sched_objective_is_near_a_closed_form_lower_bound(B, L):
    """On the uniform sweep points (96 heads x q_len 5, 36 four-CTA cluster
    slots) the scheduler's objective is at least the bound (a check of the
    bound and of the cost arithmetic) and within 3% of it at 14 of the 16
    points: the candidate families leave little on the table at these
    shapes."""
    lens = [L] * B
    S, bnd, work, eff, ms = ref.plan_sched(lens, 96, 5, 36)
    J = ms + 1.0 * S * B * 5 * 96 / 1024.0
    lb = _lower_bound(lens, 96, 5, 36)
    assert J >= lb - 1e-6
    assert J <= _LOOSE.get((B, L), 1.03) * lb, (B, L, S, J, lb)


@pytest.mark.parametrize("B,L", [(4, 400_000), (12, 100_000), (20, 100_000), (24, 100_000)])
def test_denser_cap_search_gains_little(B, L):
    """The capped family tries 32 cap values per part count; trying every
    third page as the cap (same objective, longest-first schedule) improves
    the objective by less than 2%, so the coarse grid is not what separates
    the plan from the lower bound above."""
    lens = [L] * B
    P = [-(-L // 64)] * B
    rows = B * 480
    S0, bnd0, work, eff, ms0 = ref.plan_sched(lens, 96, 5, 36)
    J0 = ms0 + S0 * rows / 1024.0
    best = J0
    p = P[0]
    for S in range(2, 9):
        for b in range(1, p + 1, 3):
            rest = p - b
            row = [0] + [b + (m - 1) * rest // (S - 1) for m in range(1, S + 1)]
            ms, _ = ref.parts_makespan(P, 2, S, [row] * B, 36, 32.0, lpt=True)
            best = min(best, ms + S * rows / 1024.0)
    assert best <= J0 + 1e-9
    assert best >= J0 / 1.02, (B, L, J0, best)


def _all_tables(P, S):
    """Every split of P pages into S consecutive parts (parts may be empty),
    as boundary rows [0, b1, ..., P]."""
    import itertools
    for cuts in itertools.combinations_with_replacement(range(P + 1), S - 1):
        yield [0, *cuts, P]


def _opt_objective(lens, U, slots, c0, lam, s_max, H=1, q_len=1):
    """The objective's optimum over every split table with up to s_max parts
    per request and every assignment of units to slots (exhaustive; tiny
    cases only): the planner's candidate families and its longest-first list
    schedule are both restrictions of this search."""
    import itertools
    P = [-(-L // 64) for L in lens]
    rows = len(lens) * q_len * H
    best = float("inf")
    for S in range(1, s_max + 1):
        for bnd in itertools.product(*[list(_all_tables(p, S)) for p in P]):
            costs = [c for _, c in ref.parts_units(P, U, S, [list(r) for r in bnd], c0)]
            best = min(best, _opt_makespan(costs, slots) + lam * S * rows / 1024.0)
    return best


def test_sched_is_within_grahams_factor_of_the_exhaustive_optimum():
    """Tiny batches (2 requests, up to 6 pages each, 1 row unit, 2 or 3
    slots, up to 3 parts): the scheduler, which searches three families of
    split tables and schedules longest first, never exceeds 4/3 of the
    optimum over all split tables and all schedules, and reaches it exactly
    on (at least 90% of) the 40 seeded cases.  c0 = 1 and lam = 0.5 keep the per-unit and per-split terms in the
    same range as a page."""
    import random
    rng = random.Random(11)
    worst, hits, n = 0.0, 0, 0
    for _ in range(40):
        lens = [64 * rng.randint(1, 6) for _ in range(2)]
        slots = rng.choice([2, 3])
        S, bnd, work, eff, ms = ref.plan_sched(lens, 1, 1, slots, s_max=3,
                                               max_parts=3, c0=1.0, lam=0.5,
                                               rows_per_unit=1)
        J = ms + 0.5 * S * len(lens) / 1024.0
        opt = _opt_objective(lens, 1, slots, 1.0, 0.5, 3)
        assert J >= opt - 1e-9
        worst = max(worst, J / opt)
        hits += abs(J - opt) < 1e-9
        n += 1
    assert worst <= 4 / 3 + 1e-9, worst
    assert hits >= 0.9 * n, (hits, n)
