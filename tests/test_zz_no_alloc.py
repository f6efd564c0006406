"""mla_decode_scratch: the fused decode with its workspace in the library's
static device scratch (no allocation, no workspace argument).

Collected last (file name) and independent of the other tests' state: every
call clears the scratch counters before its decode, whatever ran before.
CPU tests cover the size rule and the size limit (checked before any other
argument, so nothing is launched); GPU tests compare with mla_decode on
caller workspace bit for bit and check that repeated calls allocate no
device memory.
"""
import ctypes

import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth

MLA_ERR_SCRATCH = -6
SCRATCH_BYTES = 256 << 20


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mla.library()


def _r256(x):
    return (x + 255) // 256 * 256


def test_scratch_size_rule(lib):
    for B, q, H, sh, S in [(1, 1, 16, 1, 1), (16, 5, 96, 1, 2), (3, 5, 100, 8, 3),
                           (24, 5, 96, 1, 8)]:
        rows, parts = B * q * H, sh * S
        want = (_r256(B * (-(-q * H // 128)) * 4) + _r256(parts * rows * 4)
                + _r256(parts * rows * 512 * 4))
        assert mla.scratch_bytes(B, q, H, sh, S) == want
    with pytest.raises(mla.MlaError):
        mla.scratch_bytes(0, 5, 96, 1, 1)


def test_scratch_limit_is_checked_first(lib):
    """An oversized call fails with MLA_ERR_SCRATCH even with NULL data
    pointers: the limit is checked before anything else, nothing launches."""
    B, q, H, S = 128, 5, 96, 3  # 3 x 61440 partial rows of 2 KB > 256 MiB
    assert mla.scratch_bytes(B, q, H, 1, S) > SCRATCH_BYTES
    rc = lib.mla_decode_scratch(None, None, None, None, 0, 1 << 20, None, 64,
                                None, None, B, q, H, 1, 64, 0.07, S, None, None,
                                0, None, None, None, None)
    assert rc == MLA_ERR_SCRATCH
    msg = lib.mla_last_error_string().decode()
    assert str(mla.scratch_bytes(B, q, H, 1, S)) in msg and str(SCRATCH_BYTES) in msg
    # within the limit, the same NULL pointers are an ordinary argument error
    rc = lib.mla_decode_scratch(None, None, None, None, 0, 1 << 20, None, 64,
                                None, None, 1, 1, 16, 1, 64, 0.07, 1, None, None,
                                0, None, None, None, None)
    assert rc == -1


def _cases():
    return [
        ("bf16", synth.Workload("na", 3, 5, 96, [1000, 257, 5]), 3),
        ("fp8", synth.Workload("na8", 2, 5, 96, [700, 70], kv_dtype="fp8_e4m3"), 2),
        ("bf16_shards", synth.Workload("nas", 2, 5, 96, [300, 65], num_shards=8), 2),
    ]


@pytest.mark.gpu
@pytest.mark.parametrize("name,wl,S", _cases(), ids=[c[0] for c in _cases()])
def test_scratch_decode_equals_workspace_decode(lib, name, wl, S):
    batch = synth.make_batch(wl, seed=51, device="cuda")
    args = (batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
            batch.req_to_token, batch.seq_lens, batch.kv_limit, S, wl.sm_scale)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, l1 = mla.decode_scratch(*args, num_shards=wl.num_shards, status=st)
    o2, l2 = mla.decode_fused(*args, num_shards=wl.num_shards)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2), name


@pytest.mark.gpu
def test_scratch_decode_allocates_nothing_and_repeats(lib):
    """After one call (which loads the library's device code and with it the
    static scratch), further calls change neither the device's free memory
    nor their results; the full-size 16 x 5 x 96 x 100k step fits."""
    wl = synth.config("dp16")
    batch = synth.make_batch(wl, seed=0, device="cuda")
    S, bnd, _ = mla.plan_parts(wl.B, wl.q_len, wl.H, mla.batch_lengths(batch), 1)
    sp = torch.from_numpy(bnd).cuda()
    args = (batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
            batch.req_to_token, batch.seq_lens, batch.kv_limit, S, wl.sm_scale)
    out = torch.empty((wl.B, wl.q_len, wl.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.B, wl.q_len, wl.H), dtype=torch.float32, device="cuda")
    out0 = torch.empty_like(out)
    lse0 = torch.empty_like(lse)
    mla.decode_scratch(*args, out=out0, lse_out=lse0, split_pages=sp)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        mla.decode_scratch(*args, out=out, lse_out=lse, split_pages=sp)
        torch.cuda.synchronize()
        assert torch.equal(out, out0) and torch.equal(lse, lse0)
    assert torch.cuda.mem_get_info()[0] == free0
    ref_o, ref_l = mla.decode_fused(*args, split_pages=sp)
    torch.cuda.synchronize()
    assert torch.equal(ref_o, out0) and torch.equal(ref_l, lse0)


@pytest.mark.gpu
def test_scratch_decode_recovers_after_bad_work_list(lib):
    """A work list with an entry that names no unit sets MLA_STATUS_BAD_WORK
    and leaves that unit's arrival count short in the static scratch; the
    next call must not inherit it (each call clears the counters first)."""
    wl = synth.Workload("nab", 3, 5, 96, [1000, 257, 70])
    batch = synth.make_batch(wl, seed=52, device="cuda")
    S = 3  # three arrivals per (request, row unit): a missing one leaves 2
    args = (batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
            batch.req_to_token, batch.seq_lens, batch.kv_limit, S, wl.sm_scale)
    units = S * wl.B * (-(-wl.q_len * wl.H // 256))
    good = torch.arange(units, dtype=torch.int32, device="cuda")
    bad = good.clone()
    bad[0] = 1 << 30  # names no unit: that cluster does nothing
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.decode_scratch(*args, work=bad, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 8  # MLA_STATUS_BAD_WORK
    for _ in range(2):
        st.zero_()
        o1, l1 = mla.decode_scratch(*args, work=good, status=st)
        o2, l2 = mla.decode_fused(*args, work=good)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
