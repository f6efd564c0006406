"""GPU parity of the cache write (mla_kv_write) against the oracle.

BF16 rows are copied bit for bit; FP8 codes and scales must equal the
oracle's quantiser (oracle_kv_quantize) byte for byte: both take the same
binary32 divisions and the same round-to-nearest-even E4M3 decision.  Rows
cover ordinary, tiny, huge, zero and one-outlier magnitudes and values near
E4M3 midpoints; slots are scattered; a bad slot is skipped and reported; a
decode over a cache written this way matches the oracle.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
import oracle
from mla_latent_decode_gb300 import build, synth
from parity import check_close, f64, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _rows(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 576)).astype(np.float32)
    x[1] *= 1e-25
    x[2] *= 1e20
    x[3] = 0.0
    x[4, 100] = 1000.0
    x[5, :] = -0.0
    x[5, 7] = 3.0
    # values whose quotient by the scale lands on E4M3 midpoints: row amax
    # 448 makes the scale exactly 1 (midpoints of the value set are exact)
    x[6, 0] = 448.0
    x[6, 1:9] = [1.0625, 1.1875, -2.125, 0.0029296875, 300.0, -13.0, 0.75, 15.5]
    # a row maximum small enough (scale under 2^-90) for the direct division
    x[7] *= 1e-30
    # E4M3 midpoints and the 2^-10 boundary at a power-of-two scale 2^-60
    x[8, :] = 0.0
    x[8, 0] = 448.0 * 2.0 ** -60
    x[8, 1:8] = np.array([1.0625, -2.125, 2.0 ** -10, -(2.0 ** -10), 3 * 2.0 ** -11,
                          208.0, 0.0029296875]) * 2.0 ** -60
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t, t.to(torch.float32).numpy()  # the bf16 values, widened exactly


@pytest.mark.parametrize("n", [9, 300])
def test_fp8_write_matches_oracle_bytes(n):
    rows, exact = _rows(n, seed=n)
    num_slots = 4096
    slots = torch.randperm(num_slots)[:n].to(torch.int32)
    kv = torch.full((num_slots, 576), 0x7F, dtype=torch.uint8, device="cuda")
    scale = torch.full((num_slots,), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.kv_write(rows.cuda(), slots.cuda(), kv, scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    codes, scales = oracle.kv_quantize(exact)
    got = kv.cpu().numpy()[slots.numpy()]
    np.testing.assert_array_equal(got, codes)
    np.testing.assert_array_equal(scale.cpu().numpy()[slots.numpy()], scales)
    # untouched slots keep their bytes
    mask = np.ones(num_slots, bool)
    mask[slots.numpy()] = False
    assert (kv.cpu().numpy()[mask] == 0x7F).all()


def test_write_quotients_equal_ieee_division_exhaustively():
    """The write divides by a row's scale through one correctly rounded
    reciprocal and one Markstein correction: over every positive finite
    bf16 row maximum and every bf16 element it meets, its quotients equal
    the IEEE binary32 division bit for bit wherever they can set a code
    (|q| >= 2^-11), and every E4M3 code is the same."""
    counters = torch.zeros(2, dtype=torch.int64, device="cuda")
    mla.debug_quotients(counters)
    torch.cuda.synchronize()
    assert counters.tolist() == [0, 0]


def test_bf16_write_is_a_copy_and_bad_slot_is_reported():
    rows, _ = _rows(9, seed=2)
    num_slots = 256
    slots = torch.tensor([5, 200, 17, -1, 3, 300, 0, 255, 64], dtype=torch.int32)
    kv = torch.zeros((num_slots, 576), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.kv_write(rows.cuda(), slots.cuda(), kv, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 4  # MLA_STATUS_BAD_SLOT
    for r, sl in enumerate(slots.tolist()):
        if 0 <= sl < num_slots:
            assert torch.equal(kv[sl].cpu().view(torch.int16),
                               rows[r].view(torch.int16)), r
    written = {s for s in slots.tolist() if 0 <= s < num_slots}
    for sl in range(num_slots):
        if sl not in written:
            assert not kv[sl].any()


def test_decode_over_a_written_fp8_cache_matches_oracle():
    """Write a request's rows token by token into a permuted paged pool with
    mla_kv_write, then decode: the result matches the oracle on the written
    bytes and scales."""
    wl = synth.Workload("kvw", 2, 5, 96, [700, 130], kv_dtype="fp8_e4m3")
    batch = synth.make_batch(wl, seed=61, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(62)
    for b, L in enumerate(wl.seq_lens):
        rows = torch.randn((L, 576), generator=gen, device="cuda").to(torch.bfloat16)
        mla.kv_write(rows, batch.req_to_token[b, :L].contiguous(), batch.kv,
                     batch.kv_scale)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _ = mla.decode(batch, num_splits=2, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), None)
    check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                "fp8_e4m3", "decode over written cache")
