"""GPU checks of the fused decode (mla_decode: partial + LSE combine in one
launch).

The fused merge runs the same per-row arithmetic on the same parts as the
two-launch path (mla_decode_partial + mla_lse_combine), so its outputs must be
bitwise identical to that path's; they are also compared with the oracle
under the stated tolerances.  The arrival counters must be zero again after
every call, so one counter tensor serves consecutive calls.
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


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _run_both(batch, S, split_pages=None):
    """(fused out, fused lse, two-launch out, two-launch lse, counters)."""
    wl = batch.wl
    st = _status()
    counters = mla.fused_counters(wl.B, wl.q_len, wl.H, "cuda")
    args = (batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
            batch.req_to_token, batch.seq_lens, batch.kv_limit, S, wl.sm_scale)
    out_f, lse_f = mla.decode_fused(*args, num_shards=wl.num_shards,
                                    counters=counters, status=st,
                                    split_pages=split_pages)
    O_part, LSE_part = mla.decode_partial(*args, num_shards=wl.num_shards,
                                          split_pages=split_pages)
    out_u, lse_u = mla.lse_combine(O_part, LSE_part)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out_f, lse_f, out_u.view_as(out_f), lse_u.view_as(lse_f), counters


CASES = [
    ("tiny", synth.config("tiny"), 1),
    ("bf16_small", synth.Workload("fs", 3, 5, 96, [1000, 257, 5]), 3),
    ("bf16_rows_200", synth.Workload("fr", 2, 2, 100, [700, 640]), 2),
    ("bf16_empty_splits", synth.Workload("fe", 2, 5, 32, [64, 200]), 9),
    ("fp8_small", synth.Workload("f8", 3, 5, 96, [1000, 257, 5], kv_dtype="fp8_e4m3"), 3),
    ("fp8_empty_splits", synth.Workload("f8e", 2, 5, 32, [64, 200], kv_dtype="fp8_e4m3"), 9),
    # 700 rows per request: 3 BF16 units, 6 FP8 units, each with its counter
    ("bf16_rows_700_q7", synth.Workload("f7", 2, 7, 100, [900, 450]), 2),
    ("fp8_rows_700_q7", synth.Workload("f78", 2, 7, 100, [900, 450], kv_dtype="fp8_e4m3"), 2),
]


@pytest.mark.parametrize("name,wl,S", CASES, ids=[c[0] for c in CASES])
def test_fused_equals_two_launches_and_matches_oracle(name, wl, S):
    batch = synth.make_batch(wl, seed=41, device="cuda")
    out_f, lse_f, out_u, lse_u, counters = _run_both(batch, S)
    assert torch.equal(out_f, out_u) and torch.equal(lse_f, lse_u), name
    assert int(counters.abs().sum().item()) == 0
    O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), None)
    m = check_close(f64(out_f).reshape(-1, 512), f64(lse_f).reshape(-1), O_ref,
                    l_ref, wl.kv_dtype, name)
    print(name, m)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_fused_shards_match_unsharded_oracle(kv_dtype):
    """8 token-interleaved shards x 2 splits: the last of 16 parts merges."""
    sh = synth.Workload("fdcp", 3, 5, 96, [517, 64, 9], num_shards=8,
                        kv_dtype=kv_dtype)
    batch = synth.make_batch(sh, seed=42, device="cuda")
    out_f, lse_f, out_u, lse_u, counters = _run_both(batch, 2)
    assert torch.equal(out_f, out_u) and torch.equal(lse_f, lse_u)
    assert int(counters.abs().sum().item()) == 0
    host, Bq = compact_unsharded(batch, [0, 1, 2])
    O_ref, l_ref = oracle_rows_host(host, Bq, sh, kv_dtype != "bf16", None)
    check_close(f64(out_f).reshape(-1, 512), f64(lse_f).reshape(-1), O_ref, l_ref,
                kv_dtype, f"fused sharded {kv_dtype}")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_fused_with_split_table_and_repeated_calls(kv_dtype):
    """Per-request parts from a random split table (some empty); three calls
    on one counter tensor give identical results and leave it zero."""
    wl = synth.Workload("ftb", 3, 5, 96, [3000, 700, 90], kv_dtype=kv_dtype)
    batch = synth.make_batch(wl, seed=43, device="cuda")
    rng = np.random.default_rng(5)
    S = 4
    rows = []
    for L in wl.seq_lens:
        P = -(-L // 64)
        rows.append([0] + sorted(rng.integers(0, P + 1, size=S - 1).tolist()) + [P])
    sp = torch.tensor(rows, dtype=torch.int32, device="cuda")
    out_f, lse_f, out_u, lse_u, counters = _run_both(batch, S, split_pages=sp)
    assert torch.equal(out_f, out_u) and torch.equal(lse_f, lse_u)
    args = (batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
            batch.req_to_token, batch.seq_lens, batch.kv_limit, S, wl.sm_scale)
    for _ in range(2):
        o2, l2 = mla.decode_fused(*args, counters=counters, split_pages=sp)
        torch.cuda.synchronize()
        assert torch.equal(o2, out_f) and torch.equal(l2, lse_f)
        assert int(counters.abs().sum().item()) == 0
    O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), None)
    check_close(f64(out_f).reshape(-1, 512), f64(lse_f).reshape(-1), O_ref, l_ref,
                kv_dtype, f"fused split table {kv_dtype}")


def test_fused_full_size_dp16_equals_two_launches():
    """16 requests x q_len 5 x 96 heads x 100k tokens with the planner's
    per-request parts, the configuration bench.py times: fused and two-launch
    outputs are bitwise identical (the two-launch path is checked against
    the oracle at this size in test_gpu_tc.py)."""
    wl = synth.config("dp16")
    batch = synth.make_batch(wl, seed=0, device="cuda")
    S, bnd, _ = mla.plan_parts(wl.B, wl.q_len, wl.H, mla.batch_lengths(batch), 1)
    sp = torch.from_numpy(bnd).cuda()
    out_f, lse_f, out_u, lse_u, counters = _run_both(batch, S, split_pages=sp)
    assert torch.equal(out_f, out_u) and torch.equal(lse_f, lse_u)
    assert int(counters.abs().sum().item()) == 0


def test_fused_rejects_missing_outputs():
    wl = synth.Workload("fx", 1, 1, 16, [64])
    batch = synth.make_batch(wl, seed=44, device="cuda")
    O_part, LSE_part = mla.decode_partial(
        batch.q_nope, batch.q_rope, batch.kv, None, batch.req_to_token,
        batch.seq_lens, None, 1, wl.sm_scale)
    lib = mla.library()
    p = mla._ptr
    rc = lib.mla_decode(p(batch.q_nope), p(batch.q_rope), p(batch.kv), None, 0,
                        batch.kv.shape[0], p(batch.req_to_token),
                        batch.req_to_token.stride(0), p(batch.seq_lens), None, 1,
                        1, 16, 1, 64, wl.sm_scale, 1, None, None, 0, p(O_part),
                        p(LSE_part), None, None, None, None, mla._stream(None))
    assert rc == -1
