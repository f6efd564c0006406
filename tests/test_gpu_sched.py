"""GPU tests of the work-balanced scheduler's launch order (the `work` list of
mla_decode_partial / mla_decode, from mla_plan_sched).

Each work unit's result depends only on its own (part, request, row unit), so
any launch order gives the same bits: the natural order, the scheduler's
longest-first list and a random permutation are compared bit for bit, on
ragged batches with empty parts, BF16 and FP8, two launches and fused.  The
scheduled decode is compared with the oracle, and a work-list entry that
names no unit is skipped and reported (MLA_STATUS_BAD_WORK) without touching
any other unit's outputs.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth
from parity import check_close, f64, oracle_rows

pytestmark = pytest.mark.gpu

BAD_WORK = 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _workload(kv_dtype, shards=1):
    # a long request among short ones: equal chunks leave empty parts
    lens = [9000, 700, 64, 2500, 131] if shards == 1 else [60000, 2000]
    return synth.Workload(f"sched_{kv_dtype}_{shards}", len(lens), 5, 96, lens,
                          kv_dtype=kv_dtype, num_shards=shards)


def _plan(batch):
    """The scheduler with a small unit cost (c0 = 4), so these short requests
    get several parts, some of them empty."""
    wl = batch.wl
    fp8 = wl.kv_dtype != "bf16"
    S, bnd, work, _, _ = mla.plan_sched_ex(
        mla.batch_lengths(batch), wl.q_len, wl.H, 76 if fp8 else 38, 16, 8, 4.0,
        0.25, rows_per_unit=128 if fp8 else 256)
    return S, torch.from_numpy(bnd).cuda(), work


def _partials(batch, S, sp, work):
    wl = batch.wl
    st = _status()
    O = torch.full((S, wl.num_shards, wl.B, wl.q_len, wl.H, 512), 7.0,
                   dtype=torch.float32, device="cuda")
    L = torch.full((S, wl.num_shards, wl.B, wl.q_len, wl.H), 7.0,
                   dtype=torch.float32, device="cuda")
    mla.decode_partial(batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
                       batch.req_to_token, batch.seq_lens, batch.kv_limit, S,
                       wl.sm_scale, wl.num_shards, O, L, st, split_pages=sp,
                       work=None if work is None else torch.from_numpy(work).cuda())
    torch.cuda.synchronize()
    return O, L, int(st.item())


@pytest.mark.parametrize("kv_dtype,shards", [("bf16", 1), ("fp8_e4m3", 1), ("bf16", 8)])
def test_launch_order_does_not_change_the_bits(kv_dtype, shards):
    wl = _workload(kv_dtype, shards)
    batch = synth.make_batch(wl, seed=71, device="cuda")
    S, sp, work = _plan(batch)
    assert S > 1
    O0, L0, st0 = _partials(batch, S, sp, None)
    O1, L1, st1 = _partials(batch, S, sp, work)
    perm = np.random.default_rng(3).permutation(len(work)).astype(np.int32)
    O2, L2, st2 = _partials(batch, S, sp, perm)
    assert st0 == st1 == st2 == 0
    assert (L0 != 7.0).all()  # every unit wrote its rows
    for O, L in ((O1, L1), (O2, L2)):
        assert torch.equal(O.view(torch.int32), O0.view(torch.int32))
        assert torch.equal(L.view(torch.int32), L0.view(torch.int32))


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_scheduled_decode_matches_oracle(kv_dtype):
    wl = _workload(kv_dtype)
    batch = synth.make_batch(wl, seed=72, device="cuda")
    hb = synth.host_bits(batch)
    st = _status()
    out, lse, S = mla.decode(batch, status=st)  # plan_sched's parts and order
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, l_ref = oracle_rows(batch, hb, None)
    check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                kv_dtype, f"scheduled decode S={S}")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_bad_work_entry_is_skipped_and_reported(kv_dtype):
    wl = _workload(kv_dtype)
    batch = synth.make_batch(wl, seed=73, device="cuda")
    S, sp, work = _plan(batch)
    O0, L0, _ = _partials(batch, S, sp, work)
    U = -(-wl.q_len * wl.H // (256 if kv_dtype == "bf16" else 128))
    k = 3
    missing = int(work[k])
    bad = work.copy()
    bad[k] = -1
    bad[k + 1] = len(work) + 5  # also out of range: unit work[k + 1] is skipped
    O1, L1, st = _partials(batch, S, sp, bad)
    assert st == BAD_WORK
    # rows of the two skipped units keep the fill; every other row is as before
    keep = torch.ones_like(L1, dtype=torch.bool)
    R = 256 if kv_dtype == "bf16" else 128
    for unit in (missing, int(work[k + 1])):
        u, sv = unit % U, unit // U
        s, v = sv // wl.B, sv % wl.B
        flat = keep[s, 0, v].reshape(-1)
        flat[u * R:(u + 1) * R] = False
    assert (L1[~keep] == 7.0).all() and (O1[~keep] == 7.0).all()
    assert torch.equal(L1[keep], L0[keep]) and torch.equal(O1[keep], O0[keep])


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_fused_decode_in_any_order_gives_the_same_bits(kv_dtype):
    wl = _workload(kv_dtype)
    batch = synth.make_batch(wl, seed=74, device="cuda")
    S, sp, work = _plan(batch)
    perm = np.random.default_rng(9).permutation(len(work)).astype(np.int32)
    res = []
    for w in (None, work, perm):
        st = _status()
        out, lse = mla.decode_fused(
            batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
            batch.req_to_token, batch.seq_lens, batch.kv_limit, S, wl.sm_scale,
            status=st, split_pages=sp,
            work=None if w is None else torch.from_numpy(w).cuda())
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res.append((out.view(torch.int16).clone(), lse.view(torch.int32).clone()))
    for out, lse in res[1:]:
        assert torch.equal(out, res[0][0]) and torch.equal(lse, res[0][1])
