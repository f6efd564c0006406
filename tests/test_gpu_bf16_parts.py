"""GPU checks of the bf16 partial outputs (mla_decode_partial_bf16_parts and
mla_lse_combine_bf16_parts), BF16 and FP8 KV.

Each part is the fp32 path's normalised O rounded once to bf16, so:
- every part matches the oracle's part under the BF16 tolerances;
- the bf16 merge equals, bit for bit, the fp32 merge of the same parts
  widened to fp32 (the widening is exact and the arithmetic the same);
- the merged decode matches the oracle under the BF16 tolerances, with the
  parts' extra rounding (at most 2^-9 relative) inside them;
- the LSE parts are the fp32 path's, bit for bit.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth
from parity import check_close, compact_unsharded, f64, oracle_rows, oracle_rows_host, split_range

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _args(batch, S):
    wl = batch.wl
    return (batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale, batch.req_to_token,
            batch.seq_lens, batch.kv_limit, S, wl.sm_scale)


def _plan(batch):
    wl = batch.wl
    S, bnd, wk, _ = mla.plan_sched(wl.B, wl.q_len, wl.H, mla.batch_lengths(batch),
                                   wl.num_shards, kv_dtype=wl.kv_dtype)
    dev = batch.q_nope.device
    return S, torch.from_numpy(bnd).to(dev), torch.from_numpy(wk).to(dev)


CASES = [
    ("small", synth.Workload("s", 3, 5, 96, [1000, 257, 5])),
    ("rows_200", synth.Workload("r", 2, 2, 100, [700, 640])),
    ("heads16_q3", synth.Workload("h", 2, 3, 16, [130, 3])),
    ("peaked", synth.Workload("p", 2, 5, 96, [3000, 333], q_scale=8.0)),
    ("rows_700_q7", synth.Workload("r7", 2, 7, 100, [900, 450])),
    ("sharded", synth.Workload("d", 3, 5, 96, [517, 64, 9], num_shards=8)),
]


@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_bf16_parts_decode_matches_oracle_and_fp32_merge(name, wl):
    batch = synth.make_batch(wl, seed=51, device="cuda")
    S, sp, wk = _plan(batch)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Ob, Lb = mla.decode_partial(*_args(batch, S), num_shards=wl.num_shards,
                                status=st, split_pages=sp, work=wk,
                                part_dtype=torch.bfloat16)
    Of, Lf = mla.decode_partial(*_args(batch, S), num_shards=wl.num_shards,
                                status=st, split_pages=sp, work=wk)
    out_b, lse_b = mla.lse_combine(Ob, Lb)
    out_w, lse_w = mla.lse_combine(Ob.float(), Lb)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert Ob.dtype == torch.bfloat16
    # the parts: the fp32 path's, rounded once; the LSE parts identical
    assert torch.equal(Ob, Of.to(torch.bfloat16)), name
    assert torch.equal(Lb, Lf), name
    # the bf16 merge is the fp32 merge of the widened parts
    assert torch.equal(out_b, out_w) and torch.equal(lse_b, lse_w), name
    if wl.num_shards == 1:
        O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), None)
    else:
        host, Bq = compact_unsharded(batch, list(range(wl.B)))
        O_ref, l_ref = oracle_rows_host(host, Bq, wl, False, None)
    check_close(f64(out_b).reshape(-1, 512), f64(lse_b).reshape(-1), O_ref, l_ref,
                "bf16", name)


def test_bf16_parts_per_split_match_oracle():
    """Every part, empty ones included (O = 0, LSE = -inf), against the
    oracle's ranged rows."""
    wl = synth.Workload("parts", 2, 5, 40, [1000, 100], q_scale=2.0)
    batch = synth.make_batch(wl, seed=52, device="cuda")
    hb = synth.host_bits(batch)
    S = 5
    O_part, LSE_part = mla.decode_partial(*_args(batch, S), part_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    rows = np.arange(wl.rows)
    b_of = rows // (wl.q_len * wl.H)
    for s in range(S):
        lo = np.array([split_range(wl.seq_lens[b], S, s)[0] for b in b_of])
        hi = np.array([split_range(wl.seq_lens[b], S, s)[1] for b in b_of])
        O_ref, l_ref = oracle_rows(batch, hb, rows, lo=lo, hi=hi)
        check_close(f64(O_part[s, 0]).reshape(-1, 512), f64(LSE_part[s, 0]).reshape(-1),
                    O_ref, l_ref, "bf16", f"split {s}")


def test_bf16_parts_empty_splits_are_zero():
    wl = synth.Workload("e", 2, 5, 32, [64, 200])
    batch = synth.make_batch(wl, seed=53, device="cuda")
    O_part, LSE_part = mla.decode_partial(*_args(batch, 9), part_dtype=torch.bfloat16)
    O_f, L_f = mla.decode_partial(*_args(batch, 9))
    torch.cuda.synchronize()
    empty = torch.isinf(L_f) & (L_f < 0)
    assert bool(empty.any())
    assert torch.equal(O_part[empty], torch.zeros_like(O_part[empty]))
    assert torch.equal(O_part, O_f.to(torch.bfloat16))


FP8_CASES = [
    ("fp8_small", synth.Workload("f8", 3, 5, 96, [1000, 257, 5], kv_dtype="fp8_e4m3")),
    ("fp8_rows_700_q7", synth.Workload("f87", 2, 7, 100, [900, 450], kv_dtype="fp8_e4m3")),
    ("fp8_sharded", synth.Workload("f8d", 3, 5, 96, [517, 64, 9], num_shards=8,
                                   kv_dtype="fp8_e4m3")),
]


@pytest.mark.parametrize("name,wl", FP8_CASES, ids=[c[0] for c in FP8_CASES])
def test_bf16_parts_fp8_kv(name, wl):
    """The FP8 kernel's bf16 parts: the fp32 parts rounded once, the LSE
    parts bit for bit, and the merge within the FP8 tolerances."""
    batch = synth.make_batch(wl, seed=54, device="cuda")
    S, sp, wk = _plan(batch)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Ob, Lb = mla.decode_partial(*_args(batch, S), num_shards=wl.num_shards,
                                status=st, split_pages=sp, work=wk,
                                part_dtype=torch.bfloat16)
    Of, Lf = mla.decode_partial(*_args(batch, S), num_shards=wl.num_shards,
                                status=st, split_pages=sp, work=wk)
    out_b, lse_b = mla.lse_combine(Ob, Lb)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(Ob, Of.to(torch.bfloat16)), name
    assert torch.equal(Lb, Lf), name
    if wl.num_shards == 1:
        O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), None)
    else:
        host, Bq = compact_unsharded(batch, list(range(wl.B)))
        O_ref, l_ref = oracle_rows_host(host, Bq, wl, True, None)
    check_close(f64(out_b).reshape(-1, 512), f64(lse_b).reshape(-1), O_ref, l_ref,
                "fp8_e4m3", name)


@pytest.mark.parametrize("P,rows", [(7, 1000), (40, 300), (3, 20000)])
def test_bf16_combine_matches_oracle_and_widened_fp32_merge(P, rows):
    """The bf16 merge over more than 32 parts (two rounds of LSE loads) and
    over many rows (one warp per row), with empty parts and all-empty rows:
    bitwise the fp32 merge of the widened parts, and within one bf16
    rounding of the fp64 merge of those parts."""
    import oracle
    g = torch.Generator(device="cuda").manual_seed(P + rows)
    O = torch.randn((P, rows, 512), generator=g, device="cuda").to(torch.bfloat16)
    L = torch.randn((P, rows), generator=g, device="cuda") * 3
    L[P // 2, :100] = -float("inf")   # empty parts
    L[:, 100:110] = -float("inf")     # all parts empty
    out, lse = mla.lse_combine(O, L)
    out_w, lse_w = mla.lse_combine(O.float(), L)
    torch.cuda.synchronize()
    assert torch.equal(out, out_w) and torch.equal(lse, lse_w)
    O_ref, l_ref = oracle.lse_combine(f64(O), f64(L))
    got = f64(out)
    assert np.array_equal(got[100:110], np.zeros((10, 512)))
    assert np.isneginf(f64(lse)[100:110]).all()
    np.testing.assert_allclose(got, O_ref, rtol=2 ** -8, atol=1e-6)
    np.testing.assert_allclose(f64(lse), l_ref, rtol=0, atol=1e-5)
