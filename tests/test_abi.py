"""Host-side tests of the C ABI (no GPU needed, no kernel launched).

* the library loads and exports every function include/mla_decode.h declares;
* the pages' split rule and the wave-rounding planner agree with the
  brute-force reference in oracle/planner.py;
* the page-table check accepts the generator's tables and rejects planted
  faults; bad arguments are rejected on the host before any launch.
"""
import ctypes
import os
import random
import re

import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth
from oracle import planner as ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mla.library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mla_decode.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "mla_decode_partial" in names and "mla_lse_combine" in names
    for n in names:
        assert hasattr(lib, n), n


def test_pages_rule_matches_reference(lib):
    for B in range(1, 200):
        for q in range(1, 8):
            assert mla.plan_heuristic(B, q) == ref.pages_heuristic_split(B, q)
    with pytest.raises(mla.MlaError):
        mla.plan_heuristic(0, 5)


def test_planner_matches_brute_force(lib):
    rng = random.Random(7)
    cases = [([100_000] * B, 96, 5, 38) for B in (1, 2, 4, 8, 12, 16, 20, 24)]
    cases += [([12_500] * 1024, 96, 5, 38), ([256], 16, 1, 38)]
    for _ in range(40):
        V = rng.randint(1, 30)
        lens = [int(np.exp(rng.uniform(np.log(5), np.log(200_000)))) for _ in range(V)]
        cases.append((lens, rng.choice([16, 96, 128]), rng.randint(1, 6),
                      rng.choice([1, 7, 37, 38, 76])))
    for lens, H, q, slots in cases:
        c0, lam = rng.choice([(4.0, 1.0), (0.0, 0.0), (2.5, 3.0)])
        rpu = rng.choice([128, 256])
        S, eff, ms = mla.plan_ex(lens, q, H, slots, 64, c0, lam, rows_per_unit=rpu)
        S2, eff2, ms2 = ref.plan(lens, H, q, slots, 64, c0, lam, rows_per_unit=rpu)
        assert (S, ms) == (S2, ms2), (lens[:4], H, q, slots)
        assert eff == pytest.approx(eff2, rel=1e-6)


def test_planner_leaves_no_partial_wave_tail(lib):
    """The pages' rule leaves a partial second wave (B=16: 160 CTAs on 148
    SMs).  The planner's grid either fits in one wave or fills its waves to
    at least 90%.  152 SMs -> 38 cluster slots; 96 heads x q_len 5 -> 2 row
    units of 256 per request."""
    for B in (1, 2, 4, 8, 12, 16, 20, 24):
        for L in (100_000, 400_000):
            S, eff = mla.plan(B, 5, 96, [L] * B, num_sms=152)
            units = B * S * 2
            assert units <= 38 or eff >= 0.9, (B, L, S, eff)


def test_page_table_check(lib):
    wl = synth.Workload("pt", 3, 5, 2, [70, 200, 5], kv_dtype="bf16")
    b = synth.make_batch(wl, seed=1)
    mla.check_page_table(b.req_to_token, b.seq_lens, None, 5, b.num_slots)
    sh = synth.make_batch(synth.Workload("pt", 3, 5, 2, [70, 200, 9], num_shards=8), seed=1)
    mla.check_page_table(sh.req_to_token, sh.seq_lens, sh.kv_limit, 5, sh.num_slots)

    def bad(r2t=None, sl=None, kl=None, q=5, ns=None):
        with pytest.raises(mla.MlaError) as e:
            mla.check_page_table(b.req_to_token if r2t is None else r2t,
                                 b.seq_lens if sl is None else sl, kl, q,
                                 b.num_slots if ns is None else ns)
        return e.value.code

    r = b.req_to_token.clone()
    r[1, 70] += 1                      # breaks page contiguity
    assert bad(r2t=r) == -5
    r = b.req_to_token.clone()
    r[1, 64:128] += 32                 # page not aligned to 64
    assert bad(r2t=r) == -5
    assert bad(ns=64) == -5            # slots beyond the pool
    sl = b.seq_lens.clone()
    sl[2] = 3                          # shorter than q_len
    assert bad(sl=sl) == -5
    sl[2] = b.req_to_token.shape[1] + 1  # beyond the table
    assert bad(sl=sl) == -5
    kl = torch.full((3, 5), 6, dtype=torch.int32)  # kv_limit > seq_len of req 2
    assert bad(kl=kl) == -5


def _call_partial(lib, **over):
    a = dict(qn=16, qr=16, kv=16, ks=None, dt=0, ns=4096, r2t=16, st=64, sl=16,
             kl=None, B=1, q=5, H=96, shards=1, ps=64, scale=0.07, S=1, O=16,
             L=16, status=None, work=None, nw=0)
    a.update(over)
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.mla_decode_partial(p(a["qn"]), p(a["qr"]), p(a["kv"]), p(a["ks"]),
                                  a["dt"], a["ns"], p(a["r2t"]), a["st"], p(a["sl"]),
                                  p(a["kl"]), a["B"], a["q"], a["H"], a["shards"],
                                  a["ps"], a["scale"], a["S"], None, p(a["work"]),
                                  a["nw"], p(a["O"]), p(a["L"]), p(a["status"]),
                                  None)


def test_bad_arguments_are_rejected_on_the_host(lib):
    assert _call_partial(lib, qn=None) == -1
    assert _call_partial(lib, B=0) == -1
    assert _call_partial(lib, S=0) == -1
    assert _call_partial(lib, ps=32) == -2
    assert _call_partial(lib, dt=1) == -1          # FP8 without a scale
    assert _call_partial(lib, ns=10) == -1         # pool smaller than a page
    assert _call_partial(lib, kv=24) == -3         # misaligned KV
    assert _call_partial(lib, scale=float("nan")) == -1
    # a work list must name every unit: 1 request x 1 split x 2 row units
    assert _call_partial(lib, work=16, nw=1) == -1
    assert _call_partial(lib, work=16, nw=3) == -1
    assert _call_partial(lib, work=None, nw=2) == -1
    assert _call_partial(lib, work=18, nw=2) == -3     # misaligned work list
    assert b"page_size" in lib.mla_last_error_string() or True
    assert lib.mla_lse_combine(None, None, 1, 1, None, None, None) == -1
    assert lib.mla_lse_combine(ctypes.c_void_p(16), ctypes.c_void_p(16), 0, 1,
                               ctypes.c_void_p(16), None, None) == -1
    assert lib.mla_debug_gather(ctypes.c_void_p(16), 0, 4096, ctypes.c_void_p(16),
                                64, ctypes.c_void_p(16), ctypes.c_void_p(16), 1,
                                16, ctypes.c_void_p(16), None) == -2


def test_parts_planner_matches_brute_force(lib):
    rng = random.Random(11)
    cases = [([100_000] * 16, 96, 5, 36, 256), ([100_000] * 4, 96, 5, 36, 256),
             ([400_000] * 20, 96, 5, 36, 256), ([256], 16, 1, 36, 256)]
    for _ in range(12):
        V = rng.randint(1, 12)
        lens = [int(np.exp(rng.uniform(np.log(5), np.log(200_000)))) for _ in range(V)]
        cases.append((lens, rng.choice([16, 96]), rng.randint(1, 5),
                      rng.choice([7, 36, 76]), rng.choice([128, 256])))
    for lens, H, q, slots, rpu in cases:
        c0, lam = rng.choice([(32.0, 1.0), (4.0, 1.0), (0.0, 0.5)])
        S, bnd, eff, ms = mla.plan_parts_ex(lens, q, H, slots, 16, 4, c0, lam,
                                            rows_per_unit=rpu)
        S2, bnd2, eff2, ms2 = ref.plan_parts(lens, H, q, slots, 16, 4, c0, lam,
                                             rows_per_unit=rpu)
        assert (S, ms) == (S2, ms2), (lens[:4], H, q, slots, rpu)
        assert bnd.tolist() == bnd2
        assert eff == pytest.approx(eff2, rel=1e-6)
        # every row partitions the request's pages
        for L, row in zip(lens, bnd.tolist()):
            assert row[0] == 0 and row[-1] == -(-L // 64)
            assert all(a <= b for a, b in zip(row, row[1:]))


def test_parts_planner_fills_idle_slots_at_dp16():
    """16 requests x 100k on 36 cluster slots: the best uniform plan runs 32
    units (4 slots idle); capping the first part and dealing the rest to the
    idle slots shortens the modelled makespan (c0 = 32, lam = 1)."""
    lens = [100_000] * 16
    S_u, _, ms_u = ref.plan(lens, 96, 5, 36, 64, 32.0, 1.0)
    S_p, bnd, _, ms_p = ref.plan_parts(lens, 96, 5, 36, 64, 8, 32.0, 1.0)
    assert S_u == 1 and ms_u == 1563 + 32
    assert S_p >= 2 and ms_p < 0.93 * ms_u
    assert len({tuple(r) for r in bnd}) == 1   # same cut for every request


def test_sched_planner_matches_reference(lib):
    """mla_plan_sched_ex against oracle/planner.plan_sched: the same parts,
    the same longest-first work list and the same modelled makespan."""
    rng = random.Random(13)
    cases = [([100_000] * 16, 96, 5, 36, 256), ([100_000] * 4, 96, 5, 36, 256),
             ([256], 16, 1, 36, 256),
             ([1198, 152649, 2686, 60048, 10681, 170646, 4569], 96, 5, 76, 128)]
    for _ in range(12):
        V = rng.randint(1, 12)
        lens = [int(np.exp(rng.uniform(np.log(5), np.log(200_000)))) for _ in range(V)]
        cases.append((lens, rng.choice([16, 96]), rng.randint(1, 5),
                      rng.choice([7, 36, 76]), rng.choice([128, 256])))
    for lens, H, q, slots, rpu in cases:
        c0, lam = rng.choice([(32.0, 1.0), (4.0, 1.0), (0.0, 0.5)])
        S, bnd, work, eff, ms = mla.plan_sched_ex(lens, q, H, slots, 16, 4, c0,
                                                  lam, rows_per_unit=rpu)
        S2, bnd2, work2, eff2, ms2 = ref.plan_sched(lens, H, q, slots, 16, 4, c0,
                                                    lam, rows_per_unit=rpu)
        assert (S, ms) == (S2, ms2), (lens[:4], H, q, slots, rpu)
        assert bnd.tolist() == bnd2
        assert work.tolist() == work2
        assert eff == pytest.approx(eff2, rel=1e-6)


def test_sched_planner_full_search_matches_reference(lib):
    """The library's own search depth (up to 64 parts, 8 per request), where
    its bounds skip most candidates, against the reference that scores every
    candidate: a ragged batch (FP8 units), dp16 and a DCP-shaped batch."""
    ragged = [1198, 152649, 2686, 60048, 10681, 170646, 4569, 880, 33000,
              7, 199999, 5120, 64, 91000, 2300, 140000, 65, 15000, 700, 120000,
              4000, 77777, 1500, 30000]
    dcp = [(100_000 - s + 7) // 8 for _ in range(32) for s in range(8)]
    cases = [(ragged, 96, 5, 76, 128, 32.0), ([100_000] * 16, 96, 5, 36, 256, 16.0),
             (dcp, 96, 5, 36, 256, 16.0)]
    for lens, H, q, slots, rpu, c0 in cases:
        S, bnd, work, eff, ms = mla.plan_sched_ex(lens, q, H, slots, 64, 8, c0,
                                                  1.0, rows_per_unit=rpu)
        S2, bnd2, work2, eff2, ms2 = ref.plan_sched(lens, H, q, slots, 64, 8, c0,
                                                    1.0, rows_per_unit=rpu)
        assert (S, ms) == (S2, ms2), (len(lens), slots, rpu)
        assert bnd.tolist() == bnd2 and work.tolist() == work2
        assert eff == pytest.approx(eff2, rel=1e-6)
        S, bnd, eff, ms = mla.plan_parts_ex(lens, q, H, slots, 64, 8, c0, 1.0,
                                            rows_per_unit=rpu)
        S2, bnd2, eff2, ms2 = ref.plan_parts(lens, H, q, slots, 64, 8, c0, 1.0,
                                             rows_per_unit=rpu)
        assert (S, ms) == (S2, ms2) and bnd.tolist() == bnd2


def test_sched_planner_defaults_and_capacity(lib):
    lens = [3000, 90_000, 700]
    for kv, U in (("bf16", 2), ("fp8_e4m3", 4)):
        S, bnd, work, eff = mla.plan_sched(3, 5, 96, lens, num_sms=152, kv_dtype=kv)
        assert sorted(work.tolist()) == list(range(3 * S * U))
        assert 0 < eff <= 1
    # too small a work buffer: an error, nothing written
    arr = (ctypes.c_int32 * 3)(*lens)
    bnd = (ctypes.c_int32 * (3 * 17))()
    work = (ctypes.c_int32 * 1)()
    S, n = ctypes.c_int(), ctypes.c_int64()
    rc = lib.mla_plan_sched_ex(3, 5, 96, 256, arr, 38, 16, 4, 32.0, 1.0, bnd,
                               ctypes.byref(S), work, 1, ctypes.byref(n), None, None)
    assert rc == -1 and b"capacity" in lib.mla_last_error_string()
