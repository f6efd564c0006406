"""The BF16 decode with several waves of work units.

Every workload here has more than three times as many work units as the GPU
has resident 4-CTA clusters, so the hardware starts most units as earlier
ones finish and each cluster slot runs many units in turn.  A unit's
arithmetic does not depend on when or where it runs, so the two-launch path
and the fused path (whose clusters also count arrivals and merge) must agree
bit for bit, and both must match the oracle.  Covered: ragged lengths, empty
parts between non-empty ones, the scheduler's parts and order, 8 context
shards (kv_limit), a peaked softmax (rescales), NaN draft tokens, and a work
list with entries that name no unit.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth
from parity import check_close, compact_unsharded, f64, oracle_rows, oracle_rows_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _units(wl, S):
    return wl.B * wl.num_shards * S * (-(-wl.q_len * wl.H // 256))


def _both(batch, S, **kw):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, l1, _ = mla.decode(batch, num_splits=S, status=st, **kw)
    o2, l2, _ = mla.decode(batch, num_splits=S, status=st, fused=True, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o1, l1, o2, l2


def _lens(n, lo, hi, seed):
    g = np.random.default_rng(seed)
    return [int(x) for x in g.integers(lo, hi, size=n)]


CASES = [
    # 40 ragged requests x 2 row units x 3 splits = 240 units
    ("ragged", synth.Workload("pr", 40, 5, 96, _lens(40, 70, 2500, 1)), 3),
    # short requests with 9 splits: many empty parts between non-empty ones
    ("empty_parts", synth.Workload("pe", 24, 5, 96, _lens(24, 1, 700, 2)), 9),
    # peaked rows (rescales) and a request per row-unit count (q_len 7: 3 units)
    ("peaked_q7", synth.Workload("pp", 16, 7, 100, _lens(16, 300, 3000, 3),
                                 q_scale=8.0), 3),
]


@pytest.mark.parametrize("name,wl,S", CASES, ids=[c[0] for c in CASES])
def test_two_launch_equals_fused_and_oracle(name, wl, S):
    assert _units(wl, S) > 3 * mla.cluster_slots()
    batch = synth.make_batch(wl, seed=91, device="cuda")
    o1, l1, o2, l2 = _both(batch, S)
    assert torch.equal(o1, o2) and torch.equal(l1, l2), name
    rows = np.random.default_rng(5).choice(wl.rows, size=min(wl.rows, 1200), replace=False)
    O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), rows)
    check_close(f64(o1).reshape(-1, 512)[rows], f64(l1).reshape(-1)[rows], O_ref, l_ref,
                "bf16", name)


def test_many_units_scheduler_plan():
    """The scheduler's parts and longest-first order over many units."""
    wl = synth.Workload("ps", 48, 5, 96, _lens(48, 100, 6000, 4))
    batch = synth.make_batch(wl, seed=92, device="cuda")
    o1, l1, _ = mla.decode(batch)
    o2, l2, _ = mla.decode(batch, fused=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    rows = np.random.default_rng(6).choice(wl.rows, size=1000, replace=False)
    O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), rows)
    check_close(f64(o1).reshape(-1, 512)[rows], f64(l1).reshape(-1)[rows], O_ref, l_ref,
                "bf16", "scheduler")


def test_many_units_shards_vs_unsharded_oracle():
    wl = synth.Workload("psh", 12, 5, 96, _lens(12, 200, 4000, 7), num_shards=8)
    batch = synth.make_batch(wl, seed=93, device="cuda")
    o1, l1, o2, l2 = _both(batch, 2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    reqs = [0, 5, 11]
    host, Bq = compact_unsharded(batch, reqs)
    O_ref, l_ref = oracle_rows_host(host, Bq, wl, False, None)
    got_o = f64(o1)[reqs].reshape(-1, 512)
    got_l = f64(l1)[reqs].reshape(-1)
    check_close(got_o, got_l, O_ref, l_ref, "bf16", "shards")


def test_many_units_nan_draft_tokens_stay_causal():
    """NaN in draft token j of every request, over several waves: queries
    i < j bitwise unchanged, queries i >= j NaN."""
    wl = synth.Workload("pn", 40, 5, 96, _lens(40, 70, 1500, 8), q_scale=2.0)
    base = synth.make_batch(wl, seed=94, device="cuda")
    o0, l0, _ = mla.decode(base, num_splits=2)
    for j in (1, 4):
        pb = synth.make_batch(wl, seed=94, device="cuda")
        for b in range(wl.B):
            pb.kv[int(pb.req_to_token[b, wl.seq_lens[b] - wl.q_len + j])] = float("nan")
        o1, l1, _ = mla.decode(pb, num_splits=2)
        torch.cuda.synchronize()
        assert torch.equal(o0[:, :j], o1[:, :j]) and torch.equal(l0[:, :j], l1[:, :j])
        assert torch.isnan(o1[:, j:].float()).all() and torch.isnan(l1[:, j:]).all()


def test_many_units_work_list_with_entries_that_name_no_unit():
    """Entries outside [0, units) are skipped with MLA_STATUS_BAD_WORK; every
    other unit still runs (its partial rows equal the clean run's)."""
    wl = synth.Workload("pw", 30, 5, 96, _lens(30, 100, 2000, 9))
    batch = synth.make_batch(wl, seed=95, device="cuda")
    S = 3
    units = _units(wl, S)
    args = (batch.q_nope, batch.q_rope, batch.kv, None, batch.req_to_token,
            batch.seq_lens, None, S, wl.sm_scale)
    good = torch.arange(units, dtype=torch.int32, device="cuda")
    O0, L0 = mla.decode_partial(*args, work=good)
    bad = good.clone()
    bad[7] = -5
    bad[units - 1] = units + 100
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    O1 = torch.full_like(O0, 7.0)
    L1 = torch.full_like(L0, 7.0)
    mla.decode_partial(*args, O_part=O1, LSE_part=L1, status=st, work=bad)
    torch.cuda.synchronize()
    assert int(st.item()) == mla.STATUS_BAD_WORK
    U = -(-wl.q_len * wl.H // 256)
    V = wl.B
    mask = torch.ones_like(L0, dtype=torch.bool)  # [S, 1, B, q, H]
    for unit in (7, units - 1):
        u, rest = unit % U, unit // U
        v, s_ = rest % V, rest // V
        rows = slice(256 * u, min(256 * (u + 1), wl.q_len * wl.H))
        mask[s_, 0, v].view(-1)[rows] = False
    assert torch.equal(L0[mask], L1[mask])
    assert torch.equal(O0[mask], O1[mask])
    assert (L1[~mask] == 7.0).all()
