"""Pins for the fp64 CPU oracle, each against something other than the oracle.

* storage decoders: every bit pattern against torch's own conversions and the
  OCP E4M3 spec values;
* attention: an independent formulation (torch SDPA in float64 over the
  densely gathered K/V with the offset-causal mask) on tiny inputs;
* closed forms: one-token context, constant rows, zero query;
* invariants: split-KV and 8-way interleaved-shard merges equal the unsplit
  result, causality among the draft tokens, page-permutation invariance,
  NaN in unused slots never leaks.

Definitions followed: "Resident VRAM: weights and KV cache", KV ledger section
(576-d latent row = 512 c_kv + 64 RoPE key, no head dimension); "Kimi K3
decode on 2x8 B200: DP16 vs DP2 x DCP8", MLA section ((O, LSE) per shard and
an LSE merge) and "the problem" section (slot p on rank p % 8).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mla_latent_decode_gb300 import synth

SCALE = 1.0 / math.sqrt(192.0)


def _rows_of(b, i, h, q_len, H):
    return (b * q_len + i) * H + h


def _dense_kv_f64(hb, b, L, fp8):
    """Dense [L, 576] float64 rows of request b via numpy fancy indexing."""
    slots = hb["req_to_token"][b, :L].astype(np.int64)
    if fp8:
        raw = torch.from_numpy(hb["kv"][slots].copy()).view(torch.float8_e4m3fn)
        return raw.to(torch.float64).numpy() * hb["kv_scale"][slots].astype(np.float64)[:, None]
    raw = torch.from_numpy(hb["kv"][slots].view(np.int16).copy()).view(torch.bfloat16)
    return raw.to(torch.float64).numpy()


def _q_f64(hb, name):
    return torch.from_numpy(hb[name].view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def _run_oracle(hb, wl, rows=None, lo=None, hi=None, kv_limit=None, B=None):
    return oracle.mla_decode_rows(
        hb["q_nope"], hb["q_rope"], hb["kv"], wl.kv_dtype != "bf16", hb["kv_scale"],
        hb["req_to_token"], hb["seq_lens"], kv_limit if kv_limit is not None else hb["kv_limit"],
        B or wl.B, wl.q_len, wl.H, wl.sm_scale, rows, lo, hi)


# ---------------------------------------------------------------- decoders --
def test_bf16_decode_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    # sign of zero is kept
    assert math.copysign(1.0, oracle.bf16_to_f64(0x8000)) == -1.0


def test_e4m3_decode_every_byte_and_spec_values():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    # OCP FP8 E4M3: bias 7, no infinities, S.1111.111 NaN, max 448,
    # smallest subnormal 2^-9, smallest normal 2^-6.
    spec = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
            0x38: 1.0, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0, 0x40: 2.0}
    for byte, val in spec.items():
        assert oracle.e4m3_to_f64(byte) == val, hex(byte)
    assert math.isnan(oracle.e4m3_to_f64(0x7F)) and math.isnan(oracle.e4m3_to_f64(0xFF))
    assert int(nan.sum()) == 2


# ---------------------------------------------------------- brute force ----
def _sdpa_reference(hb, wl, b):
    """torch SDPA (float64) over request b's dense K/V: MQA, one KV head."""
    fp8 = wl.kv_dtype != "bf16"
    L = int(hb["seq_lens"][b])
    K = torch.from_numpy(_dense_kv_f64(hb, b, L, fp8))
    V = K[:, :512].clone()
    qn = torch.from_numpy(_q_f64(hb, "q_nope")[b])  # [q, H, 512]
    qr = torch.from_numpy(_q_f64(hb, "q_rope")[b])
    Q = torch.cat([qn, qr], dim=-1).reshape(wl.q_len * wl.H, 576)
    qi = torch.arange(wl.q_len).repeat_interleave(wl.H)
    n_vis = L - wl.q_len + 1 + qi
    mask = torch.arange(L)[None, :] < n_vis[:, None]
    O = torch.nn.functional.scaled_dot_product_attention(
        Q[None, None], K[None, None], V[None, None], attn_mask=mask[None, None],
        scale=wl.sm_scale)[0, 0]
    s = (Q @ K.T) * wl.sm_scale
    lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=1)
    return O.numpy(), lse.numpy()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_matches_sdpa_on_tiny_inputs(kv_dtype, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 4))
    q_len = int(rng.integers(1, 6))
    H = int(rng.integers(1, 5))
    lens = [int(x) for x in rng.integers(q_len, 300, size=B)]
    wl = synth.Workload("t", B, q_len, H, lens, kv_dtype=kv_dtype, q_scale=2.0)
    hb = synth.host_bits(synth.make_batch(wl, seed=seed))
    O, lse = _run_oracle(hb, wl)
    for b in range(B):
        Oref, lref = _sdpa_reference(hb, wl, b)
        sl = slice(b * q_len * H, (b + 1) * q_len * H)
        np.testing.assert_allclose(O[sl], Oref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[sl], lref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------- closed forms ---
def test_one_token_context_returns_its_own_row():
    wl = synth.Workload("one", 1, 1, 3, [1])
    hb = synth.host_bits(synth.make_batch(wl, seed=5))
    O, lse = _run_oracle(hb, wl)
    K = _dense_kv_f64(hb, 0, 1, False)[0]
    x = np.concatenate([_q_f64(hb, "q_nope")[0, 0], _q_f64(hb, "q_rope")[0, 0]], axis=-1)
    for h in range(3):
        np.testing.assert_array_equal(O[h], K[:512])
        assert lse[h] == pytest.approx(SCALE * float(np.dot(x[h], K)), rel=1e-14)


def test_constant_rows_return_the_constant():
    wl = synth.Workload("const", 2, 3, 2, [70, 131])
    batch = synth.make_batch(wl, seed=6)
    row = torch.randn(576, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    for b in range(2):
        L = wl.seq_lens[b]
        batch.kv[batch.req_to_token[b, :L].long()] = row
    hb = synth.host_bits(batch)
    O, lse = _run_oracle(hb, wl)
    r = row.to(torch.float64).numpy()
    x = np.concatenate([_q_f64(hb, "q_nope"), _q_f64(hb, "q_rope")], axis=-1)
    for b in range(2):
        L = wl.seq_lens[b]
        for i in range(3):
            for h in range(2):
                k = _rows_of(b, i, h, 3, 2)
                np.testing.assert_allclose(O[k], r[:512], rtol=1e-13, atol=1e-15)
                n = L - 3 + 1 + i
                s = SCALE * float(np.dot(x[b, i, h], r))
                assert lse[k] == pytest.approx(s + math.log(n), rel=1e-13, abs=1e-13)


def test_zero_query_gives_the_mean_of_visible_rows():
    wl = synth.Workload("zero", 2, 4, 2, [9, 200], q_scale=0.0)
    hb = synth.host_bits(synth.make_batch(wl, seed=7))
    O, lse = _run_oracle(hb, wl)
    for b in range(2):
        L = wl.seq_lens[b]
        K = _dense_kv_f64(hb, b, L, False)
        for i in range(4):
            n = L - 4 + 1 + i
            for h in range(2):
                k = _rows_of(b, i, h, 4, 2)
                np.testing.assert_allclose(O[k], K[:n, :512].mean(axis=0), rtol=1e-12, atol=1e-14)
                assert lse[k] == pytest.approx(math.log(n), abs=1e-14)


# ------------------------------------------------------------ invariants ---
def _page_split_ranges(L, S, s, page=64):
    P = -(-L // page)
    p0 = s * P // S
    p1 = (s + 1) * P // S
    return p0 * page, p1 * page


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_split_merge_equals_unsplit(kv_dtype):
    wl = synth.Workload("split", 2, 5, 3, [1000, 333], kv_dtype=kv_dtype, q_scale=3.0)
    hb = synth.host_bits(synth.make_batch(wl, seed=11))
    O, lse = _run_oracle(hb, wl)
    rows = np.arange(wl.rows, dtype=np.int64)
    b_of = rows // (wl.q_len * wl.H)
    for S in (1, 2, 3, 7, 32):
        parts_O, parts_l = [], []
        for s in range(S):
            lo = np.array([_page_split_ranges(wl.seq_lens[b], S, s)[0] for b in b_of])
            hi = np.array([_page_split_ranges(wl.seq_lens[b], S, s)[1] for b in b_of])
            Op, lp = _run_oracle(hb, wl, rows, lo, hi)
            parts_O.append(Op)
            parts_l.append(lp)
        if S == 32:  # 333 tokens = 6 pages: most splits of request 1 are empty
            assert np.isneginf(np.stack(parts_l)).any()
        Oc, lc = oracle.lse_combine(np.stack(parts_O), np.stack(parts_l))
        np.testing.assert_allclose(Oc, O, rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(lc, lse, rtol=1e-13, atol=1e-13)


def test_interleaved_shard_merge_equals_unsharded():
    base = synth.Workload("dcp", 3, 5, 2, [517, 64, 9])
    hb = synth.host_bits(synth.make_batch(base, seed=13))
    O, lse = _run_oracle(hb, base)
    sh = synth.Workload("dcp", 3, 5, 2, [517, 64, 9], num_shards=8)
    hs = synth.host_bits(synth.make_batch(sh, seed=13))
    B = 3
    parts_O, parts_l = [], []
    for s in range(8):
        sub = dict(hs)
        sub["req_to_token"] = hs["req_to_token"][s * B:(s + 1) * B]
        sub["seq_lens"] = hs["seq_lens"][s * B:(s + 1) * B]
        Op, lp = _run_oracle(sub, base, kv_limit=hs["kv_limit"][s * B:(s + 1) * B])
        parts_O.append(Op)
        parts_l.append(lp)
    # request 2 (9 tokens, q_len 5): shards 5..7 hold one token that only the
    # last queries see, so some shard parts are empty
    assert np.isneginf(np.stack(parts_l)).any()
    Oc, lc = oracle.lse_combine(np.stack(parts_O), np.stack(parts_l))
    np.testing.assert_allclose(Oc, O, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(lc, lse, rtol=1e-13, atol=1e-13)


def test_shard_lengths_follow_the_interleave_rule():
    # brute force over positions p < L: shard s holds p % S == s
    for L in (1, 5, 9, 64, 100, 517):
        for q in (1, 5):
            if q > L:
                continue
            for s in range(8):
                pos = [p for p in range(L) if p % 8 == s]
                loc, lim = synth.shard_lengths(L, q, 8, s)
                assert loc == len(pos)
                for i in range(q):
                    assert lim[i] == sum(1 for p in pos if p <= L - q + i)
    assert synth.shard_lengths(100_000, 5, 8, 3)[0] == 12_500


@pytest.mark.parametrize("poison", ["perturb", "nan"])
def test_draft_tokens_are_causal(poison):
    q_len, H = 5, 2
    wl = synth.Workload("causal", 2, q_len, H, [300, 77], q_scale=2.0)
    batch = synth.make_batch(wl, seed=17)
    hb0 = synth.host_bits(batch)
    O0, l0 = _run_oracle(hb0, wl)
    for j in range(q_len):
        pb = synth.make_batch(wl, seed=17)
        for b in range(2):
            slot = int(pb.req_to_token[b, wl.seq_lens[b] - q_len + j])
            if poison == "nan":
                pb.kv[slot] = float("nan")
            else:
                pb.kv[slot] = pb.kv[slot] * 3 + 1
        O1, l1 = _run_oracle(synth.host_bits(pb), wl)
        for b in range(2):
            for i in range(q_len):
                for h in range(H):
                    k = _rows_of(b, i, h, q_len, H)
                    if i < j:
                        assert np.array_equal(O0[k], O1[k]) and l0[k] == l1[k]
                    elif poison == "nan":
                        assert np.isnan(O1[k]).all()
                    else:
                        assert not np.array_equal(O0[k], O1[k])


def test_page_permutation_does_not_change_the_result():
    wl = synth.Workload("perm", 3, 5, 2, [200, 640, 65], kv_dtype="fp8_e4m3")
    a = synth.host_bits(synth.make_batch(wl, seed=19))
    b = synth.host_bits(synth.make_batch(wl, seed=19, page_seed=1234))
    assert not np.array_equal(a["req_to_token"], b["req_to_token"])
    Oa, la = _run_oracle(a, wl)
    Ob, lb = _run_oracle(b, wl)
    assert np.array_equal(Oa, Ob) and np.array_equal(la, lb)


def test_unused_slots_are_nan_and_do_not_leak():
    wl = synth.Workload("nan", 2, 5, 2, [70, 129])
    hb = synth.host_bits(synth.make_batch(wl, seed=23))
    # the dummy page and the tails of the last pages hold NaN
    assert np.all(hb["kv"][:64] == synth.BF16_NAN_BITS)
    last = hb["req_to_token"][0, 69]
    assert np.all(hb["kv"][last + 1] == synth.BF16_NAN_BITS)
    O, lse = _run_oracle(hb, wl)
    assert np.isfinite(O).all() and np.isfinite(lse).all()


# ---------------------------------------------------------------- combine --
def test_combine_special_cases():
    rng = np.random.default_rng(3)
    O1 = rng.standard_normal((1, 4, 512))
    l1 = rng.standard_normal((1, 4))
    Oc, lc = oracle.lse_combine(O1, l1)
    np.testing.assert_array_equal(Oc, O1[0])
    np.testing.assert_array_equal(lc, l1[0])
    # two parts with equal LSE: the plain average, LSE + ln 2
    O2 = rng.standard_normal((2, 3, 512))
    l2 = np.full((2, 3), 0.75)
    Oc, lc = oracle.lse_combine(O2, l2)
    np.testing.assert_allclose(Oc, O2.mean(axis=0), rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(lc, 0.75 + math.log(2.0), rtol=1e-15)
    # an empty part (LSE = -inf) is ignored; all-empty gives 0 and -inf
    l3 = np.array([[0.5, -np.inf], [-np.inf, -np.inf]])
    O3 = np.stack([np.ones((2, 512)), np.full((2, 512), np.nan)])
    Oc, lc = oracle.lse_combine(O3, l3)
    np.testing.assert_array_equal(Oc[0], np.ones(512))
    assert lc[0] == 0.5
    np.testing.assert_array_equal(Oc[1], np.zeros(512))
    assert np.isneginf(lc[1])
    # weights follow exp(LSE): the merge of (a, la) and (b, lb)
    la, lb = 1.0, -2.0
    a, b = rng.standard_normal(512), rng.standard_normal(512)
    Oc, lc = oracle.lse_combine(np.stack([a[None], b[None]]), np.array([[la], [lb]]))
    wa, wb = math.exp(la), math.exp(lb)
    np.testing.assert_allclose(Oc[0], (wa * a + wb * b) / (wa + wb), rtol=1e-14)
    assert lc[0] == pytest.approx(math.log(wa + wb), rel=1e-15)


def test_gather_matches_fancy_indexing():
    wl = synth.Workload("g", 3, 2, 1, [5, 130, 64], kv_dtype="bf16")
    hb = synth.host_bits(synth.make_batch(wl, seed=29))
    got = oracle.gather(hb["kv"], hb["req_to_token"], hb["seq_lens"])
    want = np.concatenate([hb["kv"][hb["req_to_token"][b, :L]] for b, L in enumerate(wl.seq_lens)])
    assert got.dtype == np.uint16 and np.array_equal(got, want)


# --------------------------------------------------- dims from the pages --
def test_model_dimensions_match_the_pages():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mla_dimensions.json")))
    H, qk, ql = g["q_b_proj_shape"]
    assert H * qk * ql / 1e6 == pytest.approx(g["q_b_proj_fp8_MB"], abs=0.05)
    Hk, nope, rank = g["w_kc_shape"]
    assert Hk * nope * rank * 2 / 1e6 == pytest.approx(g["w_kc_bf16_MB"], abs=0.05)
    total = g["mla_layers"] * (H * qk * ql + Hk * nope * rank * 2) / 2 ** 30
    assert total == pytest.approx(g["replicated_q_proj_total_GiB_24_layers"], abs=0.005)
    assert qk == g["qk_nope_head_dim"] + g["qk_rope_head_dim"]
    assert rank == g["kv_lora_rank"]
    # the latent row: kv_lora_rank + qk_rope_head_dim, 1 B per element in FP8
    assert g["kv_lora_rank"] + g["qk_rope_head_dim"] == g["kv_bytes_per_token_per_layer_fp8"] == synth.ROW_DIM
    wl = synth.config("dp16")
    assert wl.H == H and wl.q_len == g["q_len"]
    assert wl.sm_scale == pytest.approx(1.0 / math.sqrt(qk), rel=1e-15)
    assert synth.VALUE_DIM == g["kv_lora_rank"]
