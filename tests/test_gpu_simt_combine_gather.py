"""GPU parity of the CUDA-core decode path, the LSE combine and the TMA gather.

Every expected value comes from the fp64 oracle (oracle/) on the same seeded
inputs; nothing expected is produced by the CUDA path itself.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
import oracle
from mla_latent_decode_gb300 import build, synth
from parity import check_close, f64, oracle_rows, split_range

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


CASES = [
    ("tiny", synth.config("tiny"), 1),
    ("small_bf16", synth.Workload("s", 3, 5, 96, [1000, 257, 5]), 3),
    ("small_fp8", synth.Workload("s8", 2, 5, 96, [700, 64], kv_dtype="fp8_e4m3"), 2),
    ("heads16_q3", synth.Workload("h", 2, 3, 16, [130, 3]), 7),
    ("peaked", synth.Workload("p", 2, 5, 32, [900, 333], q_scale=8.0), 4),
]


@pytest.mark.parametrize("name,wl,S", CASES, ids=[c[0] for c in CASES])
def test_simt_decode_matches_oracle(name, wl, S):
    batch = synth.make_batch(wl, seed=3, device="cuda")
    hb = synth.host_bits(batch)
    st = _status()
    out, lse, _ = mla.decode(batch, num_splits=S, simt=True, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, l_ref = oracle_rows(batch, hb, None)
    check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                wl.kv_dtype, name)


def test_simt_partials_match_oracle_per_split():
    wl = synth.Workload("parts", 2, 5, 8, [1000, 100], q_scale=2.0)
    batch = synth.make_batch(wl, seed=4, device="cuda")
    hb = synth.host_bits(batch)
    S = 5
    O_part, LSE_part = mla.decode_partial(
        batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale, batch.req_to_token,
        batch.seq_lens, batch.kv_limit, S, wl.sm_scale, simt=True)
    torch.cuda.synchronize()
    rows = np.arange(wl.rows)
    b_of = rows // (wl.q_len * wl.H)
    for s in range(S):
        lo = np.array([split_range(wl.seq_lens[b], S, s)[0] for b in b_of])
        hi = np.array([split_range(wl.seq_lens[b], S, s)[1] for b in b_of])
        O_ref, l_ref = oracle_rows(batch, hb, rows, lo=lo, hi=hi)
        check_close(f64(O_part[s, 0]).reshape(-1, 512), f64(LSE_part[s, 0]).reshape(-1),
                    O_ref, l_ref, "bf16", f"split {s}")
    # request 1 has 2 pages dealt floor(s*2/5): splits 0, 1 and 3 are empty
    for s in range(S):
        lo, hi = split_range(wl.seq_lens[1], S, s)
        empty = bool(torch.isneginf(LSE_part[s, 0, 1]).all()) and bool((O_part[s, 0, 1] == 0).all())
        assert empty == (hi <= lo), s
    assert [s for s in range(S) if split_range(100, S, s)[1] <= split_range(100, S, s)[0]] == [0, 1, 3]


def test_simt_shards_combine_to_unsharded():
    base = synth.Workload("dcp", 3, 5, 16, [517, 64, 9])
    sh = synth.Workload("dcp", 3, 5, 16, [517, 64, 9], num_shards=8)
    b_un = synth.make_batch(base, seed=5, device="cuda")
    b_sh = synth.make_batch(sh, seed=5, device="cuda")
    out_u, lse_u, _ = mla.decode(b_un, num_splits=2, simt=True)
    out_s, lse_s, _ = mla.decode(b_sh, num_splits=2, simt=True)
    torch.cuda.synchronize()
    hb = synth.host_bits(b_un)
    O_ref, l_ref = oracle_rows(b_un, hb, None)
    check_close(f64(out_s).reshape(-1, 512), f64(lse_s).reshape(-1), O_ref, l_ref, "bf16", "sharded")
    check_close(f64(out_u).reshape(-1, 512), f64(lse_u).reshape(-1), O_ref, l_ref, "bf16", "unsharded")


def test_combine_matches_oracle():
    g = torch.Generator(device="cuda").manual_seed(8)
    P, rows = 7, 1000
    O = torch.randn((P, rows, 512), generator=g, device="cuda")
    L = torch.randn((P, rows), generator=g, device="cuda") * 3
    L[2, :100] = -float("inf")          # empty parts
    L[:, 100:110] = -float("inf")       # all parts empty
    O[2, :100] = float("nan")           # never read
    out, lse = mla.lse_combine(O, L)
    torch.cuda.synchronize()
    O_ref, l_ref = oracle.lse_combine(f64(O), f64(L))
    got = f64(out)
    assert np.array_equal(got[100:110], np.zeros((10, 512)))
    assert np.isneginf(f64(lse)[100:110]).all()
    # bf16 output: within one bf16 rounding of the fp64 merge
    np.testing.assert_allclose(got, O_ref, rtol=2 ** -8, atol=1e-6)
    np.testing.assert_allclose(f64(lse), l_ref, rtol=0, atol=1e-5)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_gather_is_bit_exact(kv_dtype):
    wl = synth.Workload("g", 4, 5, 1, [1, 64, 65, 1000], kv_dtype=kv_dtype)
    batch = synth.make_batch(wl, seed=9, device="cuda")
    hb = synth.host_bits(batch)
    lens = wl.seq_lens
    off = torch.tensor(np.concatenate([[0], np.cumsum(lens)[:-1]]), dtype=torch.int64,
                       device="cuda")
    dense = mla.debug_gather(batch.kv, batch.req_to_token, batch.seq_lens, off, sum(lens))
    torch.cuda.synchronize()
    want = oracle.gather(hb["kv"], hb["req_to_token"], hb["seq_lens"])
    got = dense.contiguous().view(torch.uint8).cpu().numpy().reshape(want.shape[0], -1)
    assert np.array_equal(got, want.view(np.uint8).reshape(want.shape[0], -1))
