"""Reference for the split planner (test infrastructure only).

Two things live here, both written plainly so they can be read against their
sources:

1. The pages' own split heuristic and grid arithmetic ("Kimi K3 decode on 2x8
   B200: DP16 vs DP2 x DCP8", section "MLA: bytes conserved, DP16 kernel slowed
   by wave quantisation"): split = min(148 // B // (q_len * 2), 32), with the
   floor of 1 that the same paragraph implies ("split = 1 for B >= 8"), and the
   grid (2, B * q_len, split) on 148 SMs.

2. A brute-force statement of this library's wave-rounding objective, the
   one the C planner must reproduce exactly:
     units       one work unit per (split s, virtual request v, row unit u),
                 launched in that order (u fastest), U = ceil(H*q_len / R),
                 R = rows_per_unit (256: the library's kernel serves 256
                 query rows with one 4-CTA cluster)
     unit cost   pages(v, s) + c0 page-tiles, where request v's P_v =
                 ceil(L_v / 64) pages are dealt to splits as
                 floor((s+1) P_v / S) - floor(s P_v / S)
     makespan    list scheduling of the units, in launch order, onto `slots`
                 unit slots (each unit starts on the slot that frees first)
     objective   J(S) = makespan(S) + lam * S * rows / 1024, rows = V*q_len*H
                 (the partial outputs each extra split writes and re-reads)
     choice      the S in [1, S_max] with the smallest J; ties go to fewer
                 splits.  Wave efficiency = sum(unit costs) / (slots *
                 makespan).
"""
from __future__ import annotations

import heapq
from typing import List, Sequence, Tuple

PAGES_SMS = 148          # B200 SM count used by the pages' heuristic
ROWS_PER_UNIT = 256      # query rows per work unit of the library's kernel


def pages_heuristic_split(B: int, q_len: int, sms: int = PAGES_SMS) -> int:
    """The pages' split rule, with the implied floor of one split."""
    return max(1, min(sms // B // (q_len * 2), 32))


def pages_grid(B: int, q_len: int, split: int) -> Tuple[int, int, int]:
    """The pages' grid (2, B * q_len, split) for the M128 2-CTA path."""
    return (2, B * q_len, split)


def pages_waves(B: int, q_len: int, split: int, sms: int = PAGES_SMS):
    """CTAs of the pages' grid and how many waves they take on `sms` SMs."""
    x, y, z = pages_grid(B, q_len, split)
    ctas = x * y * z
    return ctas, ctas / sms


def split_pages(P: int, S: int, s: int) -> int:
    return (s + 1) * P // S - s * P // S


def makespan(costs: Sequence[float], slots: int) -> float:
    heap = [0.0] * min(slots, max(1, len(costs)))
    heapq.heapify(heap)
    end = 0.0
    for c in costs:
        t = heapq.heappop(heap) + c
        end = max(end, t)
        heapq.heappush(heap, t)
    return end


def unit_costs(seq_lens: Sequence[int], H: int, q_len: int, S: int,
               c0: float, page: int = 64,
               rows_per_unit: int = ROWS_PER_UNIT) -> List[float]:
    """Unit costs in launch order: split s of every request before split
    s + 1, row units innermost."""
    G = -(-H * q_len // rows_per_unit)
    out = []
    for s in range(S):
        for L in seq_lens:
            P = -(-L // page)
            c = split_pages(P, S, s) + c0
            out.extend([c] * G)
    return out


def plan(seq_lens: Sequence[int], H: int, q_len: int, slots: int,
         s_max: int = 64, c0: float = 4.0, lam: float = 1.0,
         rows_per_unit: int = ROWS_PER_UNIT):
    """Brute-force planner: returns (S, wave_efficiency, makespan)."""
    rows = len(seq_lens) * q_len * H
    best = None
    for S in range(1, s_max + 1):
        costs = unit_costs(seq_lens, H, q_len, S, c0,
                           rows_per_unit=rows_per_unit)
        ms = makespan(costs, slots)
        J = ms + lam * S * rows / 1024.0
        if best is None or J < best[0] - 1e-9:
            best = (J, S, sum(costs) / (slots * ms), ms)
    return best[1], best[2], best[3]


# ---------------------------------------------------------------- parts
N_CAPS = 32        # cap candidates b = ceil(Pmax * k / 32), k = 1..32
EMPTY_COST = 1.0   # an empty work unit


def parts_units(P: Sequence[int], U: int, S: int, bnd: List[List[int]],
                c0: float):
    """Every work unit of a per-request split schedule as (id, cost), id =
    (s * V + v) * U + u in increasing order (part s of every request before
    part s + 1, row units innermost); a unit costs its pages + c0, an empty
    one EMPTY_COST."""
    V = len(P)
    units = []
    for s in range(S):
        for v in range(V):
            pages = bnd[v][s + 1] - bnd[v][s]
            c = float(pages) + c0 if pages > 0 else EMPTY_COST
            for u in range(U):
                units.append(((s * V + v) * U + u, c))
    return units


def lpt_order(units):
    """Longest processing time first: by decreasing cost, equal costs by
    increasing id."""
    return sorted(units, key=lambda iu: (-iu[1], iu[0]))


def parts_makespan(P: Sequence[int], U: int, S: int, bnd: List[List[int]],
                   slots: int, c0: float, lpt: bool = False):
    """List-scheduling makespan of a per-request split schedule, its units
    taken in launch order (increasing id) or, with lpt, longest first.
    Returns (makespan, total cost)."""
    units = parts_units(P, U, S, bnd, c0)
    if lpt:
        units = lpt_order(units)
    costs = [c for _, c in units]
    return makespan(costs, slots), sum(costs)


def plan_parts(seq_lens: Sequence[int], H: int, q_len: int, slots: int,
               s_max: int = 64, max_parts: int = 8, c0: float = 32.0,
               lam: float = 1.0, rows_per_unit: int = ROWS_PER_UNIT,
               page: int = 64, lpt: bool = False):
    """Brute force over three candidate families (uniform deals for
    S = 1..s_max; first part capped at b, the rest dealt over S - 1 parts for
    S = 2..max_parts; equal chunks of ceil(Pmax / S) pages for S =
    2..max_parts), scored by makespan + lam * S * rows / 1024, first of equal
    scores kept; the makespan takes the units in launch order, or longest
    first with lpt.  Returns (S, boundaries [V][S+1], wave_eff, makespan)."""
    U = -(-H * q_len // rows_per_unit)
    rows = len(seq_lens) * q_len * H
    P = [-(-max(L, 0) // page) for L in seq_lens]
    pmax = max(P)
    best = None

    def consider(S, bnd):
        nonlocal best
        ms, tot = parts_makespan(P, U, S, bnd, slots, c0, lpt)
        J = ms + lam * S * rows / 1024.0
        if best is None or J < best[0] - 1e-9:
            best = (J, S, bnd, tot / (slots * ms) if ms > 0 else 1.0, ms)

    for S in range(1, s_max + 1):
        consider(S, [[k * p // S for k in range(S + 1)] for p in P])
    for S in range(2, max_parts + 1):
        prev = -1
        for k in range(1, N_CAPS + 1):
            b = (pmax * k + N_CAPS - 1) // N_CAPS
            if b == prev or b < 1:
                continue
            prev = b
            bnd = []
            for p in P:
                first = min(p, b)
                rest = p - first
                bnd.append([0] + [first + (m - 1) * rest // (S - 1)
                                  for m in range(1, S + 1)])
            consider(S, bnd)
    for S in range(2, max_parts + 1):
        u = -(-pmax // S)
        if u < 1:
            continue
        consider(S, [[min(p, m * u) for m in range(S + 1)] for p in P])
    return best[1], best[2], best[3], best[4]


def plan_sched(seq_lens: Sequence[int], H: int, q_len: int, slots: int,
               s_max: int = 64, max_parts: int = 8, c0: float = 32.0,
               lam: float = 1.0, rows_per_unit: int = ROWS_PER_UNIT,
               page: int = 64):
    """The work-balanced scheduler: plan_parts scored with the units taken
    longest first, and that order as the work list.  Returns (S, boundaries
    [V][S+1], work ids in launch order, wave_eff, makespan)."""
    S, bnd, eff, ms = plan_parts(seq_lens, H, q_len, slots, s_max, max_parts,
                                 c0, lam, rows_per_unit, page, lpt=True)
    U = -(-H * q_len // rows_per_unit)
    P = [-(-max(L, 0) // page) for L in seq_lens]
    work = [i for i, _ in lpt_order(parts_units(P, U, S, bnd, c0))]
    return S, bnd, work, eff, ms
