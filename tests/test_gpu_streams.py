"""The decode entry points run on the stream they are given, torch's current
stream or an explicit `stream=`, with bitwise the results of the default
stream; and two decodes in flight at once on two streams, each with its own
buffers, give the bits each gives alone: the library keeps no state between
calls (the end-to-end loop in bench.py overlaps steps this way).
"""
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _plan(batch):
    wl = batch.wl
    S, bnd, wk, _ = mla.plan_sched(wl.B, wl.q_len, wl.H, mla.batch_lengths(batch),
                                   wl.num_shards, kv_dtype=wl.kv_dtype)
    dev = batch.q_nope.device
    return S, torch.from_numpy(bnd).to(dev), torch.from_numpy(wk).to(dev)


def _buffers(batch, S):
    wl = batch.wl
    dev = batch.q_nope.device
    O = torch.full((S, wl.num_shards, wl.B, wl.q_len, wl.H, 512), 7.0,
                   dtype=torch.float32, device=dev)
    L = torch.full((S, wl.num_shards, wl.B, wl.q_len, wl.H), 7.0,
                   dtype=torch.float32, device=dev)
    out = torch.zeros((wl.B, wl.q_len, wl.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((wl.B, wl.q_len, wl.H), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    counters = mla.fused_counters(wl.B, wl.q_len, wl.H, dev)
    return O, L, out, lse, st, counters


def _launch(batch, plan, bufs, stream=None, fused=False):
    """Enqueue one decode step; the buffers were made ready beforehand."""
    wl = batch.wl
    S, sp, wk = plan
    O, L, out, lse, st, counters = bufs
    if fused:
        mla.decode_fused(batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
                         batch.req_to_token, batch.seq_lens, batch.kv_limit, S,
                         wl.sm_scale, wl.num_shards, O, L, counters, out, lse, st,
                         stream=stream, split_pages=sp, work=wk)
        return
    mla.decode_partial(batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
                       batch.req_to_token, batch.seq_lens, batch.kv_limit, S,
                       wl.sm_scale, wl.num_shards, O, L, st, stream=stream,
                       split_pages=sp, work=wk)
    mla.lse_combine(O, L, out, lse, stream=stream)


def _bits(bufs):
    O, L, out, lse, st, _ = bufs
    assert int(st.item()) == 0
    return out.view(torch.int16).clone(), lse.view(torch.int32).clone()


def _same(a, b):
    return torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_side_stream_gives_the_default_stream_bits(kv_dtype):
    wl = synth.Workload(f"st_{kv_dtype}", 3, 5, 96, [3000, 700, 90], kv_dtype=kv_dtype)
    batch = synth.make_batch(wl, seed=81, device="cuda")
    plan = _plan(batch)
    side = torch.cuda.Stream()
    ref = _buffers(batch, plan[0])
    explicit = _buffers(batch, plan[0])
    current = _buffers(batch, plan[0])
    torch.cuda.synchronize()  # inputs and buffers ready for every stream
    _launch(batch, plan, ref)
    _launch(batch, plan, explicit, stream=side)
    with torch.cuda.stream(side):
        _launch(batch, plan, current)
    torch.cuda.synchronize()
    r = _bits(ref)
    assert _same(_bits(explicit), r) and _same(_bits(current), r)


@pytest.mark.parametrize("fused", [False, True], ids=["two_launches", "fused"])
def test_two_decodes_in_flight_match_each_alone(fused):
    a = synth.make_batch(synth.Workload("sa", 3, 5, 96, [5000, 64, 1200]),
                         seed=82, device="cuda")
    b = synth.make_batch(synth.Workload("sb", 2, 5, 96, [2500, 9000],
                                        kv_dtype="fp8_e4m3"), seed=83, device="cuda")
    pa, pb = _plan(a), _plan(b)
    alone_a, alone_b = _buffers(a, pa[0]), _buffers(b, pb[0])
    both_a, both_b = _buffers(a, pa[0]), _buffers(b, pb[0])
    torch.cuda.synchronize()
    _launch(a, pa, alone_a, fused=fused)
    torch.cuda.synchronize()
    _launch(b, pb, alone_b, fused=fused)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    _launch(a, pa, both_a, stream=s1, fused=fused)
    _launch(b, pb, both_b, stream=s2, fused=fused)
    torch.cuda.synchronize()
    assert _same(_bits(both_a), _bits(alone_a))
    assert _same(_bits(both_b), _bits(alone_b))
