"""FP8 KV decode with outlier channels in the query, vs the oracle.

The FP8 kernel represents a query row as 2^e (Qhi + Qlo), two E4M3 parts,
exact for elements within 2^9 of the row's largest.  A channel far above the
rest of its row (an outlier feature of the absorbed query, the same channel
in every row) would set e and push the other elements under that floor, so
such channels (up to 4 per 128-row group) leave the split and their products
with the key bytes are added in fp32.  These tests put single-channel
outliers of 256x, 1000x and 4096x the typical |q| into q_nope and q_rope
(and two at once, and at the kernel's 128-dim block boundaries) and check
the decode against the oracle at the FP8 tolerances.  Expected values come
only from oracle/.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth
from parity import check_close, f64, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _with_outliers(batch, channels, factor):
    """Multiply query channel c (0..511: q_nope, 512..575: q_rope) of every
    row by `factor` (the bf16 rounding of the product is the input)."""
    for c in channels:
        if c < 512:
            batch.q_nope[..., c] = (batch.q_nope[..., c].float() * factor).to(torch.bfloat16)
        else:
            batch.q_rope[..., c - 512] = (batch.q_rope[..., c - 512].float()
                                          * factor).to(torch.bfloat16)


def _decode_vs_oracle(wl, channels, factor, S, seed, what):
    batch = synth.make_batch(wl, seed=seed, device="cuda")
    _with_outliers(batch, channels, factor)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _ = mla.decode(batch, num_splits=S, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), None)
    m = check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                    wl.kv_dtype, what)
    print(what, m)
    return m


@pytest.mark.parametrize("factor", [256.0, 1000.0, 4096.0])
@pytest.mark.parametrize("channel", [77, 300, 512 + 13], ids=["nope77", "nope300", "rope13"])
def test_fp8_single_channel_outlier(channel, factor):
    wl = synth.Workload("out8", 2, 5, 96, [3000, 333], kv_dtype="fp8_e4m3")
    _decode_vs_oracle(wl, [channel], factor, 3, seed=81,
                      what=f"fp8 channel {channel} x{factor:g}")


@pytest.mark.parametrize("channels", [[127, 128], [511, 512], [575], [5, 530]],
                         ids=["block_edge", "nope_rope_edge", "last", "nope_and_rope"])
def test_fp8_outlier_channels_at_block_edges(channels):
    wl = synth.Workload("oute8", 2, 5, 96, [700, 130], kv_dtype="fp8_e4m3")
    _decode_vs_oracle(wl, channels, 1000.0, 2, seed=82,
                      what=f"fp8 channels {channels} x1000")


def test_fp8_outliers_peaked_rows_and_fused():
    """Larger queries (a peaked softmax) with an outlier channel, through the
    fused decode and the scheduler's plan."""
    wl = synth.Workload("outp8", 3, 5, 96, [4000, 1000, 77], kv_dtype="fp8_e4m3",
                        q_scale=4.0)
    batch = synth.make_batch(wl, seed=83, device="cuda")
    _with_outliers(batch, [200], 1000.0)
    out, lse, _ = mla.decode(batch, fused=True)
    torch.cuda.synchronize()
    O_ref, l_ref = oracle_rows(batch, synth.host_bits(batch), None)
    print(check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                      "fp8_e4m3", "fp8 peaked fused x1000"))


def test_bf16_single_channel_outlier():
    """BF16 KV with a 256x outlier channel (no query split there).  Beyond
    that the BF16 tensor-core path keeps no exception channels: the outlier
    products dominate the MMA's fp32 partial sums, and at 4096x the rounding
    of those sums moves the LSE by up to ~4e-3."""
    wl = synth.Workload("out16", 2, 5, 96, [3000, 333])
    _decode_vs_oracle(wl, [300], 256.0, 3, seed=85, what="bf16 channel 300 x256")
