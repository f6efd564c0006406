"""Page-table entries outside the pool and lengths past the table, through
the decode kernels (tensor-core BF16 and FP8 KV, and the CUDA-core path):
the recovery the header states, against the oracle.

- A page whose base slot is negative, not a multiple of the page size, or
  whose 64 slots run past the pool is read as zeros and
  MLA_STATUS_BAD_SLOT is set: its tokens score 0 and add zero value rows.
  The oracle sees the same inputs with that page's tokens pointed at a page
  of zeros.  Bad pages are put at the start of a split (the first tile of a
  unit) and inside one.
- A length past the page table's stride is clamped to the stride and
  MLA_STATUS_BAD_LENGTH is set.  The oracle sees the clamped length.

Expected values come only from oracle/.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth
from parity import check_close, f64, oracle_rows

pytestmark = pytest.mark.gpu

PAGE = 64
BAD_SLOT, BAD_LENGTH = 4, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _zero_page0(hb, fp8):
    """Page 0 of the pool (slots 0..63) is never a request's page; make it a
    page of zeros for the oracle."""
    hb["kv"][:PAGE] = 0
    if fp8:
        hb["kv_scale"][:PAGE] = 1.0


@pytest.mark.parametrize("kv_dtype,simt", [("bf16", False), ("fp8_e4m3", False),
                                           ("bf16", True)],
                         ids=["tc_bf16", "tc_fp8", "simt_bf16"])
@pytest.mark.parametrize("where", ["split_start", "inside"])
@pytest.mark.parametrize("kind", ["past_pool", "negative", "misaligned"])
def test_bad_page_reads_zeros(kv_dtype, simt, where, kind):
    wl = synth.Workload("bad", 2, 5, 96, [1000, 700], kv_dtype=kv_dtype)
    batch = synth.make_batch(wl, seed=61, device="cuda")
    num_slots = batch.kv.shape[0]
    # request 0: 16 pages in 2 splits of 8 (pages 0..7, 8..15)
    page = 8 if where == "split_start" else 5
    t0 = page * PAGE
    good = int(batch.req_to_token[0, t0].item())
    bad = {"past_pool": num_slots, "negative": -PAGE, "misaligned": good + 1}[kind]
    batch.req_to_token[0, t0] = bad

    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _ = mla.decode(batch, num_splits=2, simt=simt, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == BAD_SLOT

    hb = synth.host_bits(batch)
    fp8 = kv_dtype != "bf16"
    _zero_page0(hb, fp8)
    hb["req_to_token"][0, t0:t0 + PAGE] = np.arange(PAGE, dtype=np.int32)
    O_ref, l_ref = oracle_rows(batch, hb, None)
    check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                kv_dtype, f"{kv_dtype} simt={simt} {where} {kind}")

    # the context stays usable: the same decode on a good table reports nothing
    batch.req_to_token[0, t0] = good
    st.zero_()
    mla.decode(batch, num_splits=2, simt=simt, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


@pytest.mark.parametrize("kv_dtype,simt", [("bf16", False), ("fp8_e4m3", False),
                                           ("bf16", True)],
                         ids=["tc_bf16", "tc_fp8", "simt_bf16"])
def test_length_past_table_is_clamped(kv_dtype, simt):
    # request 0 holds 1000 tokens in 16 pages, so the table's stride is 1024;
    # a length of 1100 is clamped to 1024.  Tokens 1000..1023 lie in the
    # request's last page, whose unwritten slots are zeros here (scale 1 for
    # FP8), and the oracle reads the same slots.
    wl = synth.Workload("len", 2, 5, 96, [1000, 700], kv_dtype=kv_dtype)
    batch = synth.make_batch(wl, seed=62, device="cuda", nan_fill=False)
    stride = batch.req_to_token.shape[1]
    assert stride == 1024
    base = int(batch.req_to_token[0, 960].item()) - 960 % PAGE
    fp8 = kv_dtype != "bf16"
    if fp8:
        batch.kv_scale[base + 1000 % PAGE:base + PAGE] = 1.0
    batch.seq_lens[0] = 1100

    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _ = mla.decode(batch, num_splits=2, simt=simt, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == BAD_LENGTH

    hb = synth.host_bits(batch)
    hb["seq_lens"][0] = stride
    t = np.arange(1000, stride)
    hb["req_to_token"][0, t] = base + t % PAGE
    O_ref, l_ref = oracle_rows(batch, hb, None)
    check_close(f64(out).reshape(-1, 512), f64(lse).reshape(-1), O_ref, l_ref,
                kv_dtype, f"{kv_dtype} simt={simt} clamped length")
