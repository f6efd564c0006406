"""GPU parity of the tensor-core decode path (mla_decode_partial) vs the oracle.

Small cases span several tiles, ragged tails, empty splits, shards and the
rescale path (peaked softmax); the full-size 16 x 5 x 96 x 100k workload is
checked on sampled rows in the launch configuration bench.py times.  Bitwise
properties (page-permutation invariance, causality, determinism) need no
oracle.  Expected values come only from oracle/.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth
from parity import (check_close, compact_unsharded, f64, oracle_rows,
                    oracle_rows_host, split_range)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


CASES = [
    ("tiny", synth.config("tiny"), 1),
    ("one_token", synth.Workload("one", 1, 1, 16, [1]), 1),
    ("small_bf16", synth.Workload("s", 3, 5, 96, [1000, 257, 5]), 3),
    ("heads16_q3", synth.Workload("h", 2, 3, 16, [130, 3]), 7),
    ("rows_200", synth.Workload("r", 2, 2, 100, [700, 640]), 2),
    ("peaked", synth.Workload("p", 2, 5, 96, [3000, 333], q_scale=8.0), 4),
    ("long_one_split", synth.Workload("l", 1, 5, 96, [20_000]), 1),
    ("empty_splits", synth.Workload("e", 2, 5, 32, [64, 200]), 9),
    # more rows per request than the 480 of the pages' shape: 700 rows are 3
    # units of 256 (the last 188), 1024 rows exactly 4; q_len 7 and 8
    ("rows_700_q7", synth.Workload("r7", 2, 7, 100, [900, 450]), 2),
    ("rows_1024_q8", synth.Workload("r1k", 1, 8, 128, [1300]), 2),
]


@pytest.mark.parametrize("name,wl,S", CASES, ids=[c[0] for c in CASES])
def test_tc_decode_matches_oracle(name, wl, S):
    batch = synth.make_batch(wl, seed=3, device="cuda")
    hb = synth.host_bits(batch)
    st = _status()
    out, lse, _ = mla.decode(batch, num_splits=S, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, l_ref = oracle_rows(batch, hb, None)
    m = check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                    wl.kv_dtype, name)
    print(name, m)


def test_tc_partials_match_oracle_per_split():
    wl = synth.Workload("parts", 2, 5, 40, [1000, 100], q_scale=2.0)
    batch = synth.make_batch(wl, seed=4, device="cuda")
    hb = synth.host_bits(batch)
    S = 5
    O_part, LSE_part = mla.decode_partial(
        batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale, batch.req_to_token,
        batch.seq_lens, batch.kv_limit, S, wl.sm_scale)
    torch.cuda.synchronize()
    rows = np.arange(wl.rows)
    b_of = rows // (wl.q_len * wl.H)
    for s in range(S):
        lo = np.array([split_range(wl.seq_lens[b], S, s)[0] for b in b_of])
        hi = np.array([split_range(wl.seq_lens[b], S, s)[1] for b in b_of])
        O_ref, l_ref = oracle_rows(batch, hb, rows, lo=lo, hi=hi)
        check_close(f64(O_part[s, 0]).reshape(-1, 512), f64(LSE_part[s, 0]).reshape(-1),
                    O_ref, l_ref, "bf16", f"split {s}")


@pytest.mark.parametrize("lens,splits", [([517, 64, 9], 2), ([5, 300, 7], None)],
                         ids=["short", "empty_shards_scheduled"])
def test_tc_shards_match_unsharded_oracle(lens, splits):
    """8 token-interleaved shards vs the unsharded oracle.  With 5- and
    7-token requests some shards hold no token at all (their parts are
    empty: O = 0, LSE = -inf) and shard-local lengths fall below q_len; the
    second case takes the scheduler's parts and launch order."""
    sh = synth.Workload("dcp", 3, 5, 96, lens, num_shards=8)
    base = synth.Workload("dcp", 3, 5, 96, lens)
    b_sh = synth.make_batch(sh, seed=5, device="cuda")
    b_un = synth.make_batch(base, seed=5, device="cuda")
    st = _status()
    out_s, lse_s, _ = mla.decode(b_sh, num_splits=splits, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, l_ref = oracle_rows(b_un, synth.host_bits(b_un), None)
    check_close(f64(out_s).reshape(-1, 512), f64(lse_s).reshape(-1), O_ref, l_ref,
                "bf16", "sharded")


def test_tc_agrees_with_cuda_core_path():
    wl = synth.Workload("x", 4, 5, 96, [2000, 1500, 64, 777], q_scale=3.0)
    batch = synth.make_batch(wl, seed=6, device="cuda")
    a, la, _ = mla.decode(batch, num_splits=3)
    b, lb, _ = mla.decode(batch, num_splits=3, simt=True)
    torch.cuda.synchronize()
    check_close(f64(a).reshape(-1, 512), f64(la).reshape(-1), f64(b).reshape(-1, 512),
                f64(lb).reshape(-1), "bf16", "tc vs simt")


def test_tc_page_permutation_and_determinism_are_bitwise():
    wl = synth.Workload("perm", 3, 5, 96, [900, 4000, 130])
    a = synth.make_batch(wl, seed=7, device="cuda")
    b = synth.make_batch(wl, seed=7, device="cuda", page_seed=999)
    assert not torch.equal(a.req_to_token, b.req_to_token)
    oa, la, _ = mla.decode(a, num_splits=4)
    oa2, la2, _ = mla.decode(a, num_splits=4)
    ob, lb, _ = mla.decode(b, num_splits=4)
    torch.cuda.synchronize()
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    assert torch.equal(oa, oa2) and torch.equal(la, la2)


def test_tc_draft_tokens_are_causal():
    """Zero queries make the softmax flat (O = mean of the visible c_kv rows),
    so adding 1 to draft token j's c_kv must move every row of query i >= j by
    exactly 1/n_i and leave the rows of queries i < j bitwise unchanged
    (checked on the fp32 partial output of a single split)."""
    q_len, H = 5, 96
    wl = synth.Workload("causal", 2, q_len, H, [300, 77], q_scale=0.0)

    def run(batch):
        O, L = mla.decode_partial(batch.q_nope, batch.q_rope, batch.kv, None,
                                  batch.req_to_token, batch.seq_lens, None, 1,
                                  wl.sm_scale)
        torch.cuda.synchronize()
        return O[0, 0], L[0, 0]

    base = synth.make_batch(wl, seed=8, device="cuda")
    o0, l0 = run(base)
    for j in range(q_len):
        pb = synth.make_batch(wl, seed=8, device="cuda")
        delta = {}
        for b in range(2):
            slot = int(pb.req_to_token[b, wl.seq_lens[b] - q_len + j])
            pb.kv[slot, :512] += 1
            # the stored shift is 1 up to the bf16 rounding of the new row
            delta[b] = (pb.kv[slot, :512].double() - base.kv[slot, :512].double()).cpu().numpy()
        o1, l1 = run(pb)
        assert torch.equal(o0[:, :j], o1[:, :j]) and torch.equal(l0[:, :j], l1[:, :j])
        for b in range(2):
            assert np.abs(delta[b] - 1).max() <= 2 ** -4
            for i in range(j, q_len):
                n = wl.seq_lens[b] - q_len + 1 + i
                d = (o1[b, i].double() - o0[b, i].double()).cpu().numpy()
                assert np.abs(d - delta[b][None, :] / n).max() < 2e-6, (b, i, j)


def test_tc_full_size_dp16_sampled_rows():
    """16 requests x q_len 5 x 96 heads x 100k tokens, planner splits (the
    configuration bench.py times), checked on rows sampled across requests,
    queries, heads and row groups."""
    wl = synth.config("dp16")
    batch = synth.make_batch(wl, seed=0, device="cuda")
    st = _status()
    out, lse, S = mla.decode(batch, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    hb = synth.host_bits(batch)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([
        rng.choice(wl.rows, 40, replace=False),
        [0, wl.rows - 1, 127, 128, 383, 384, 479]]))  # row-group edges
    O_ref, l_ref = oracle_rows(batch, hb, rows)
    got = f64(out).reshape(-1, 512)[rows]
    m = check_close(got, f64(lse).reshape(-1)[rows], O_ref, l_ref, "bf16",
                    f"dp16 S={S}")
    print("dp16", S, m)


def test_tc_full_size_dcp_sampled_rows_vs_unsharded_oracle():
    """128 requests x q_len 5 x 96 heads x 100k tokens in 8 token-interleaved
    shards (12.5k local tokens each, 14.7 GB of KV), planner splits, one
    launch over all shards, then the LSE combine over 8 x S parts.  Sampled
    rows of three requests are compared with the unsharded oracle on the
    same bytes."""
    wl = synth.config("dcp")
    batch = synth.make_batch(wl, seed=0, device="cuda")
    st = _status()
    out, lse, S = mla.decode(batch, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    reqs = [0, 77, 127]
    host, Bq = compact_unsharded(batch, reqs)
    R = wl.q_len * wl.H
    rng = np.random.default_rng(1)
    local = np.unique(np.concatenate([rng.choice(Bq * R, 30, replace=False),
                                      [0, R - 1, R, 2 * R + 479]]))
    O_ref, l_ref = oracle_rows_host(host, Bq, wl, False, local)
    flat_out = f64(out).reshape(wl.B * R, 512)
    flat_lse = f64(lse).reshape(wl.B * R)
    glob = np.array([reqs[r // R] * R + r % R for r in local])
    m = check_close(flat_out[glob], flat_lse[glob], O_ref, l_ref, "bf16",
                    f"dcp S={S}")
    print("dcp", S, m)


@pytest.mark.parametrize("name", ["sweep_B1_L400000", "sweep8_B1_L400000"])
def test_tc_longest_context_sampled_rows(name):
    """One request of 400k tokens (6250 pages), BF16 or FP8 KV, with the
    scheduler's parts (18 for BF16): the longest context of the sweep, checked
    on sampled rows and the row-group edges."""
    wl = synth.config(name)
    batch = synth.make_batch(wl, seed=3, device="cuda")
    st = _status()
    out, lse, S = mla.decode(batch, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and S > 1
    hb = synth.host_bits(batch)
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([rng.choice(wl.rows, 30, replace=False),
                                     [0, 127, 128, 255, 256, 383, 384, 479]]))
    O_ref, l_ref = oracle_rows(batch, hb, rows)
    m = check_close(f64(out).reshape(-1, 512)[rows], f64(lse).reshape(-1)[rows],
                    O_ref, l_ref, wl.kv_dtype, f"{name} S={S}")
    print(name, S, m)


# ----------------------------------------------------------- FP8 E4M3 KV ----
FP8_CASES = [
    ("fp8_tiny", synth.Workload("t8", 1, 1, 16, [256], kv_dtype="fp8_e4m3"), 1),
    ("fp8_small", synth.Workload("s8", 3, 5, 96, [1000, 257, 5], kv_dtype="fp8_e4m3"), 3),
    ("fp8_heads16_q3", synth.Workload("h8", 2, 3, 16, [130, 3], kv_dtype="fp8_e4m3"), 7),
    ("fp8_peaked", synth.Workload("p8", 2, 5, 96, [3000, 333], kv_dtype="fp8_e4m3",
                                  q_scale=8.0), 4),
    ("fp8_empty_splits", synth.Workload("e8", 2, 5, 32, [64, 200], kv_dtype="fp8_e4m3"), 9),
    # 700 rows: 6 units of 128 (the last 60); 1024 rows: exactly 8
    ("fp8_rows_700_q7", synth.Workload("r78", 2, 7, 100, [900, 450], kv_dtype="fp8_e4m3"), 2),
    ("fp8_rows_1024_q8", synth.Workload("r1k8", 1, 8, 128, [1300], kv_dtype="fp8_e4m3"), 2),
]


@pytest.mark.parametrize("name,wl,S", FP8_CASES, ids=[c[0] for c in FP8_CASES])
def test_tc_fp8_decode_matches_oracle(name, wl, S):
    batch = synth.make_batch(wl, seed=13, device="cuda")
    hb = synth.host_bits(batch)
    st = _status()
    out, lse, _ = mla.decode(batch, num_splits=S, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, l_ref = oracle_rows(batch, hb, None)
    m = check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                    "fp8_e4m3", name)
    print(name, m)


def _rescale_tokens(batch, fn):
    """kv_scale[slot of token t of request b] *= fn(b, t) (in place, B x L)."""
    for b, L in enumerate(batch.wl.seq_lens):
        t = torch.arange(L, device="cuda")
        slots = batch.req_to_token[b, :L].long()
        batch.kv_scale[slots] *= fn(b, t).to(torch.float32)


FP8_SCALE_CASES = [
    # (name, kv scale factor per token, query factor, output factor).
    # Scales growing along the context: the running max |scale| crosses
    # powers of two inside a split (O and l change units mid-stream).
    ("growing", lambda b, t: torch.pow(2.0, (t // 300).float() - 9.0), 1.0, 1.0),
    # neighbouring pages 2^18 apart: most of a tile's P' sits far below its max
    ("alternating", lambda b, t: torch.pow(2.0, -18.0 * ((t // 64) % 2).float()),
     1.0, 1.0),
    # scales far from 1 with the query scaled the other way: the scores (and
    # the LSE) are unchanged and O scales exactly by the factor
    ("tiny", lambda b, t: torch.full_like(t, 2.0 ** -40, dtype=torch.float32),
     2.0 ** 40, 2.0 ** -40),
    ("large", lambda b, t: torch.full_like(t, 2.0 ** 12, dtype=torch.float32),
     2.0 ** -12, 2.0 ** 12),
]


@pytest.mark.parametrize("name,fn,qf,of", FP8_SCALE_CASES,
                         ids=[c[0] for c in FP8_SCALE_CASES])
def test_tc_fp8_scale_magnitudes_match_oracle(name, fn, qf, of):
    wl = synth.Workload("sc8", 2, 5, 96, [2500, 700], kv_dtype="fp8_e4m3", q_scale=2.0)
    batch = synth.make_batch(wl, seed=31, device="cuda")
    _rescale_tokens(batch, fn)
    batch.q_nope.mul_(qf)
    batch.q_rope.mul_(qf)
    hb = synth.host_bits(batch)
    st = _status()
    out, lse, _ = mla.decode(batch, num_splits=2, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, l_ref = oracle_rows(batch, hb, None)
    m = check_close(f64(out).reshape(-1, 512) / of, f64(lse).reshape(-1), O_ref / of,
                    l_ref, "fp8_e4m3", f"fp8 scales {name}")
    print(name, m)


def test_tc_fp8_query_dynamic_range_matches_oracle():
    """Query rows with one element 64 times the rest, and rows scaled by
    2^-60: the row scale 2^e of the FP8 path keeps every element at least
    2^-9 of the row's largest exact."""
    wl = synth.Workload("qd8", 2, 5, 96, [900, 300], kv_dtype="fp8_e4m3")
    batch = synth.make_batch(wl, seed=32, device="cuda")
    batch.q_nope[:, :, ::3, 7] *= 64.0
    batch.q_rope[:, :, 1::3, 5] *= 64.0
    batch.q_nope[:, :, 2::7, :] *= 2.0 ** -60
    batch.q_rope[:, :, 2::7, :] *= 2.0 ** -60
    hb = synth.host_bits(batch)
    st = _status()
    out, lse, _ = mla.decode(batch, num_splits=1, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, l_ref = oracle_rows(batch, hb, None)
    m = check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                    "fp8_e4m3", "fp8 q dynamic range")
    print(m)


@pytest.mark.parametrize("lens,splits", [([517, 64, 9], 2), ([5, 300, 7], None)],
                         ids=["short", "empty_shards_scheduled"])
def test_tc_fp8_shards_match_unsharded_oracle(lens, splits):
    sh = synth.Workload("dcp8", 3, 5, 96, lens, num_shards=8,
                        kv_dtype="fp8_e4m3")
    batch = synth.make_batch(sh, seed=5, device="cuda")
    st = _status()
    out, lse, _ = mla.decode(batch, num_splits=splits, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    host, Bq = compact_unsharded(batch, [0, 1, 2])
    O_ref, l_ref = oracle_rows_host(host, Bq, sh, True, None)
    check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                "fp8_e4m3", "fp8 sharded")


def test_tc_fp8_agrees_with_cuda_core_path():
    wl = synth.Workload("x8", 4, 5, 96, [2000, 1500, 64, 777], q_scale=3.0,
                        kv_dtype="fp8_e4m3")
    batch = synth.make_batch(wl, seed=6, device="cuda")
    a, la, _ = mla.decode(batch, num_splits=3)
    b, lb, _ = mla.decode(batch, num_splits=3, simt=True)
    torch.cuda.synchronize()
    check_close(f64(a).reshape(-1, 512), f64(la).reshape(-1), f64(b).reshape(-1, 512),
                f64(lb).reshape(-1), "fp8_e4m3", "fp8 tc vs simt")


def test_tc_fp8_full_size_ragged_sampled_rows():
    """24 requests x q_len 5 x 96 heads, contexts log-uniform in [1k, 200k],
    E4M3 KV with per-token scales, planner splits; rows sampled across
    requests (short and long) compared with the oracle on the stored bytes."""
    wl = synth.config("ragged_fp8")
    batch = synth.make_batch(wl, seed=0, device="cuda")
    st = _status()
    out, lse, S = mla.decode(batch, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    order = np.argsort(wl.seq_lens)
    reqs = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    host, Bq = compact_unsharded(batch, reqs)
    R = wl.q_len * wl.H
    rng = np.random.default_rng(2)
    local = np.unique(np.concatenate([rng.choice(Bq * R, 30, replace=False),
                                      [0, R - 1, Bq * R - 1]]))
    O_ref, l_ref = oracle_rows_host(host, Bq, wl, True, local)
    glob = np.array([reqs[r // R] * R + r % R for r in local])
    m = check_close(f64(out).reshape(-1, 512)[glob], f64(lse).reshape(-1)[glob],
                    O_ref, l_ref, "fp8_e4m3", f"ragged_fp8 S={S}")
    print("ragged_fp8", S, [wl.seq_lens[r] for r in reqs], m)


# ------------------------------------------------- per-request split tables ----
def _ragged_table(wl, S, seed):
    """Random non-decreasing boundaries 0 = b0 <= ... <= bS = P per request,
    with some empty parts."""
    rng = np.random.default_rng(seed)
    rows = []
    for L in (wl.seq_lens * wl.num_shards if wl.num_shards == 1 else
              [synth.shard_lengths(L, wl.q_len, wl.num_shards, s)[0]
               for s in range(wl.num_shards) for L in wl.seq_lens]):
        P = -(-L // 64)
        cuts = sorted(rng.integers(0, P + 1, size=S - 1).tolist())
        rows.append([0] + cuts + [P])
    return np.array(rows, dtype=np.int32)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_tc_split_table_parts_and_combine_match_oracle(kv_dtype):
    wl = synth.Workload("tbl", 3, 5, 96, [3000, 700, 90], kv_dtype=kv_dtype)
    batch = synth.make_batch(wl, seed=21, device="cuda")
    hb = synth.host_bits(batch)
    S = 4
    table = _ragged_table(wl, S, 3)
    sp = torch.from_numpy(table).cuda()
    st = _status()
    O_part, LSE_part = mla.decode_partial(
        batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale, batch.req_to_token,
        batch.seq_lens, batch.kv_limit, S, wl.sm_scale, status=st, split_pages=sp)
    out, lse = mla.lse_combine(O_part, LSE_part)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = np.arange(wl.rows)
    b_of = rows // (wl.q_len * wl.H)
    for s in range(S):
        lo = np.array([min(table[b][s] * 64, wl.seq_lens[b]) for b in b_of])
        hi = np.array([min(table[b][s + 1] * 64, wl.seq_lens[b]) for b in b_of])
        O_ref, l_ref = oracle_rows(batch, hb, rows, lo=lo, hi=hi)
        check_close(f64(O_part[s, 0]).reshape(-1, 512), f64(LSE_part[s, 0]).reshape(-1),
                    O_ref, l_ref, kv_dtype, f"part {s}")
    O_ref, l_ref = oracle_rows(batch, hb, None)
    check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                kv_dtype, "combined")


def test_simt_split_table_matches_tensor_core():
    wl = synth.Workload("tbl2", 2, 5, 96, [1500, 333], num_shards=8)
    batch = synth.make_batch(wl, seed=22, device="cuda")
    S = 3
    sp = torch.from_numpy(_ragged_table(wl, S, 4)).cuda()
    a, la = mla.decode_partial(batch.q_nope, batch.q_rope, batch.kv, None,
                               batch.req_to_token, batch.seq_lens, batch.kv_limit,
                               S, wl.sm_scale, num_shards=8, split_pages=sp)
    b, lb = mla.decode_partial(batch.q_nope, batch.q_rope, batch.kv, None,
                               batch.req_to_token, batch.seq_lens, batch.kv_limit,
                               S, wl.sm_scale, num_shards=8, split_pages=sp, simt=True)
    torch.cuda.synchronize()
    fa, fb = f64(a).reshape(-1, 512), f64(b).reshape(-1, 512)
    check_close(fa, f64(la).reshape(-1), fb, f64(lb).reshape(-1), "bf16",
                "tc vs simt, split table")
