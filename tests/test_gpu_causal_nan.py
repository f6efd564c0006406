"""Causality among the draft tokens under non-finite KV, on the GPU.

Query i of a request sees tokens t <= L - q_len + i (or t < kv_limit[v, i]
on a context shard), so filling draft token j = L - q_len + j with NaN must
leave the rows of queries i < j bitwise unchanged and make the rows of
queries i >= j NaN, exactly as the oracle does (the pin is
tests/test_oracle.py::test_draft_tokens_are_causal).  The masked token must
add nothing to the rows that may not see it, not 0 * NaN.

Covered: BF16 KV (NaN and infinite rows) and FP8 KV (a row of NaN codes),
partial outputs per split, the two-launch and the fused decode, the
scheduler's plan, 8 token-interleaved context shards (kv_limit), draft
tokens straddling a page and a split boundary, and q_len 8.

A FP8 token's scale must be finite.  It also takes part in the split's
shared power-of-two unit for the probabilities, so changing a draft token's
scale may move the last bits of earlier queries' rows (through the rounding
of tiny probabilities) but never more: with a NaN or infinite scale on a
draft token the earlier queries' rows still match the oracle of the clean
batch within the FP8 tolerances.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth
from parity import (check_close, compact_unsharded, f64, oracle_rows,
                    oracle_rows_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _slot(batch, b, p):
    wl = batch.wl
    S = wl.num_shards
    if S == 1:
        return int(batch.req_to_token[b, p])
    return int(batch.req_to_token[(p % S) * wl.B + b, p // S])


def _poison(batch, j, how):
    """Poison draft token j of every request (logical position L - q + j)."""
    wl = batch.wl
    for b in range(wl.B):
        slot = _slot(batch, b, wl.seq_lens[b] - wl.q_len + j)
        if how == "nan":
            if batch.kv_is_fp8:
                batch.kv[slot] = synth.E4M3_NAN_BYTE
            else:
                batch.kv[slot] = float("nan")
        elif how == "inf":
            batch.kv[slot] = float("inf")
        elif how == "scale_nan":
            batch.kv_scale[slot] = float("nan")
        elif how == "scale_inf":
            batch.kv_scale[slot] = float("inf")
        else:
            raise ValueError(how)


def _run(batch, mode, S):
    """(out, lse) with rows [B, q, H, ...], plus the partials (or None)."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if mode == "partial":
        O, L = mla.decode_partial(
            batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
            batch.req_to_token, batch.seq_lens, batch.kv_limit, S,
            batch.wl.sm_scale, num_shards=batch.wl.num_shards, status=st)
        out, lse = mla.lse_combine(O, L)
        parts = (O, L)
    else:
        out, lse, _ = mla.decode(batch, num_splits=S, status=st,
                                 fused=(mode == "fused"))
        parts = None
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out, lse, parts


def _check(wl, mode, S, how, seed, oracle_j=None):
    base = synth.make_batch(wl, seed=seed, device="cuda")
    o0, l0, p0 = _run(base, mode, S)
    assert torch.isfinite(o0).all() and torch.isfinite(l0).all()
    for j in range(wl.q_len):
        pb = synth.make_batch(wl, seed=seed, device="cuda")
        _poison(pb, j, how)
        o1, l1, p1 = _run(pb, mode, S)
        # queries i < j never see the poisoned token: bitwise unchanged
        assert torch.equal(o0[:, :j], o1[:, :j]), (how, j)
        assert torch.equal(l0[:, :j], l1[:, :j]), (how, j)
        if p0 is not None:  # every split's partial rows of queries i < j too
            assert torch.equal(p0[0][:, :, :, :j], p1[0][:, :, :, :j]), (how, j)
            assert torch.equal(p0[1][:, :, :, :j], p1[1][:, :, :, :j]), (how, j)
        if how in ("nan", "scale_nan"):
            # queries i >= j see it: their rows are NaN, O and LSE
            assert torch.isnan(o1[:, j:].float()).all(), (how, j)
            assert torch.isnan(l1[:, j:]).all(), (how, j)
        if oracle_j == j:
            if wl.num_shards > 1:  # the unsharded definition
                host, Bq = compact_unsharded(pb, list(range(wl.B)))
                O_ref, l_ref = oracle_rows_host(host, Bq, wl, pb.kv_is_fp8, None)
            else:
                O_ref, l_ref = oracle_rows(pb, synth.host_bits(pb), None)
            got_o = o1.float().cpu().numpy().reshape(-1, 512)
            got_l = l1.cpu().numpy().reshape(-1)
            assert np.array_equal(np.isnan(O_ref), np.isnan(got_o))
            assert np.array_equal(np.isnan(l_ref), np.isnan(got_l))


# lengths: 300 (draft tokens inside the last page), 130 (they straddle pages
# 1 and 2), 66 (with 2 uniform splits they straddle the split boundary)
LENS = [300, 130, 66]


@pytest.mark.parametrize("mode", ["partial", "two_launch", "fused"])
def test_bf16_nan_draft_token_is_causal(mode):
    wl = synth.Workload("cnan", 3, 5, 96, LENS, q_scale=2.0)
    _check(wl, mode, 2, "nan", seed=61, oracle_j=2 if mode == "two_launch" else None)


def test_bf16_inf_draft_token_leaves_earlier_queries_bitwise():
    wl = synth.Workload("cinf", 3, 5, 96, LENS, q_scale=2.0)
    _check(wl, "partial", 2, "inf", seed=62)


def test_bf16_nan_draft_token_scheduler_plan():
    wl = synth.Workload("csch", 3, 5, 96, [4000, 300, 130], q_scale=2.0)
    _check(wl, "two_launch", None, "nan", seed=63)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_nan_draft_token_q_len_8(kv_dtype):
    wl = synth.Workload("c8", 2, 8, 16, [200, 70], kv_dtype=kv_dtype, q_scale=2.0)
    _check(wl, "partial", 2, "nan", seed=64)


@pytest.mark.parametrize("mode", ["partial", "fused"])
def test_fp8_nan_draft_token_is_causal(mode):
    wl = synth.Workload("cnan8", 3, 5, 96, LENS, kv_dtype="fp8_e4m3", q_scale=2.0)
    _check(wl, mode, 2, "nan", seed=65, oracle_j=3 if mode == "partial" else None)


@pytest.mark.parametrize("how", ["scale_nan", "scale_inf"])
def test_fp8_non_finite_scale_of_draft_token(how):
    """Outside the contract (scales must be finite), but a non-finite scale
    on draft token j still leaves the rows of queries i < j finite and within
    the FP8 tolerances of the clean batch's oracle; with NaN the rows of
    queries i >= j are NaN."""
    wl = synth.Workload("cscl8", 3, 5, 96, LENS, kv_dtype="fp8_e4m3", q_scale=2.0)
    base = synth.make_batch(wl, seed=67, device="cuda")
    O_ref, l_ref = oracle_rows(base, synth.host_bits(base), None)
    O_ref = O_ref.reshape(wl.B, wl.q_len, wl.H, 512)
    l_ref = l_ref.reshape(wl.B, wl.q_len, wl.H)
    for j in range(1, wl.q_len):
        pb = synth.make_batch(wl, seed=67, device="cuda")
        _poison(pb, j, how)
        o1, l1, _ = _run(pb, "partial", 2)
        check_close(f64(o1[:, :j]).reshape(-1, 512), f64(l1[:, :j]).reshape(-1),
                    O_ref[:, :j].reshape(-1, 512), l_ref[:, :j].reshape(-1),
                    "fp8_e4m3", f"{how} j={j}")
        if how == "scale_nan":
            assert torch.isnan(o1[:, j:].float()).all()
            assert torch.isnan(l1[:, j:]).all()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("mode", ["partial", "fused"])
def test_sharded_nan_draft_token_is_causal(kv_dtype, mode):
    """8 token-interleaved shards: draft token j lives in shard (L-q+j) % 8,
    where kv_limit hides it from the queries i < j."""
    wl = synth.Workload("cnans", 2, 5, 96, [300, 130], kv_dtype=kv_dtype,
                        num_shards=8, q_scale=2.0)
    _check(wl, mode, 2, "nan", seed=66, oracle_j=1 if mode == "partial" else None)
