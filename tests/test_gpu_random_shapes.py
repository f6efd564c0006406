"""Seeded random shapes through the tensor-core decode, against the fp64
oracle.

Each case draws the batch size, q_len, the head count (including counts that
leave a 256-row unit or a 32-row store block partly filled), ragged lengths
(some shorter than a page, some shorter than q_len in a shard), the KV type,
the context-shard count and the split count (or the scheduler's plan).  The
two-launch path (partial decode + combine) is compared element by element
with the oracle under the stated tolerances; the fused launch, whose partial
outputs take the plain-store path where the two-launch path stores by TMA,
must give the same bits.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth
from parity import check_close, compact_unsharded, f64, oracle_rows, oracle_rows_host

pytestmark = pytest.mark.gpu

HEADS = [1, 3, 16, 32, 48, 96, 100, 128]


def _case(i):
    rng = np.random.default_rng(1000 + i)
    B = int(rng.integers(1, 5))
    q_len = int(rng.integers(1, 9))
    H = int(rng.choice(HEADS))
    while q_len * H > 1024:
        H = int(rng.choice(HEADS))
    lens = []
    for _ in range(B):
        kind = rng.integers(0, 3)
        hi = 70 if kind == 0 else (700 if kind == 1 else 2500)
        lens.append(int(rng.integers(q_len, hi + 1)))
    kv_dtype = "fp8_e4m3" if i % 2 else "bf16"
    shards = 8 if i % 4 == 3 else 1
    splits = None if rng.random() < 0.5 else int(rng.integers(1, 10))
    q_scale = float(rng.choice([1.0, 4.0]))
    wl = synth.Workload(f"r{i}", B, q_len, H, lens, kv_dtype=kv_dtype,
                        num_shards=shards, q_scale=q_scale)
    return wl, splits


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


@pytest.mark.parametrize("i", range(16))
def test_random_shape_matches_oracle_and_fused_bits(i):
    wl, S = _case(i)
    batch = synth.make_batch(wl, seed=2000 + i, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, S_used = mla.decode(batch, num_splits=S, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, (i, wl)
    if wl.num_shards == 1:
        O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), None)
    else:
        host, Bq = compact_unsharded(batch, list(range(wl.B)))
        O_ref, l_ref = oracle_rows_host(host, Bq, wl, wl.kv_dtype != "bf16", None)
    check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                wl.kv_dtype, f"case {i}: {wl}")

    # the fused launch on the same uniform deal
    counters = mla.fused_counters(wl.B, wl.q_len, wl.H, "cuda")
    args = (batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
            batch.req_to_token, batch.seq_lens, batch.kv_limit, S_used, wl.sm_scale)
    out_f, lse_f = mla.decode_fused(*args, num_shards=wl.num_shards,
                                    counters=counters, status=st)
    O_part, LSE_part = mla.decode_partial(*args, num_shards=wl.num_shards)
    out_u, lse_u = mla.lse_combine(O_part, LSE_part)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out_f, out_u.view_as(out_f)), i
    assert torch.equal(lse_f, lse_u.view_as(lse_f)), i
    assert int(counters.abs().sum().item()) == 0
