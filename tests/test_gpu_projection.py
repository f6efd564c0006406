"""GPU parity of the per-head projections (mla_absorb_q, mla_project_out)
against the fp64 oracle.

Bound (from the arithmetic): the result is the fp32-accumulated sum rounded
once to bf16, so |got - y| <= 2^-8 |y| + 1.01 * 2 K 2^-24 sum_k |x_k w_k|
(half a bf16 step of 8 significant bits, plus a generous fp32 accumulation
term).  Shapes cover one row, a ragged tail across two 128-row tiles, the
dp16 (80 rows) and DCP (640 rows) row counts, and few heads.
"""
import numpy as np
import pytest
import torch

import mla_latent_decode_gb300 as mla
import oracle
from mla_latent_decode_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    mla.library()


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _check(got, x, w):
    y = oracle.head_projection(_bits(x), _bits(w))
    xa = np.abs(x.cpu().float().numpy().astype(np.float64))
    wa = np.abs(w.cpu().float().numpy().astype(np.float64))
    acc = np.einsum("mhk,hkn->mhn", xa, wa)
    K = x.shape[-1]
    bound = 2.0 ** -8 * np.abs(y) + 1.01 * 2 * K * 2.0 ** -24 * acc
    g = got.cpu().float().numpy().astype(np.float64)
    err = np.abs(g - y)
    assert (err <= bound).all(), float((err - bound).max())
    return float(err.max())


@pytest.mark.parametrize("M,H", [(1, 96), (80, 96), (130, 3), (640, 96)])
def test_absorb_q_matches_oracle(M, H):
    g = torch.Generator(device="cuda").manual_seed(M + H)
    q = torch.randn((M, 1, H, 128), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((H, 128, 512), generator=g, device="cuda") / 11.3).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mla.absorb_q(q, w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    print(M, H, _check(out.view(M, H, 512), q.view(M, H, 128), w))


@pytest.mark.parametrize("M,H", [(1, 96), (80, 96), (130, 3), (640, 96)])
def test_project_out_matches_oracle(M, H):
    g = torch.Generator(device="cuda").manual_seed(1000 + M + H)
    o = torch.randn((M, 1, H, 512), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((H, 512, 128), generator=g, device="cuda") / 22.6).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mla.project_out(o, w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    print(M, H, _check(out.view(M, H, 128), o.view(M, H, 512), w))


def test_projection_argument_errors():
    lib = mla.library()
    assert lib.mla_absorb_q(None, None, None, 1, 96, None, None) == -1
    x = torch.zeros((1, 1, 96, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((96, 128, 512), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, 1, 96, 512), dtype=torch.bfloat16, device="cuda")
    assert lib.mla_absorb_q(mla._ptr(x), mla._ptr(w), mla._ptr(y), 0, 96, None, None) == -1


def test_chained_launches_read_what_the_previous_launch_wrote():
    """Both projections let the stream's next kernel start early and prefetch
    its weights before waiting: a launch whose activations and weights are
    the output of the launch just before it (no synchronisation between
    them) must read the written values."""
    H = 96
    g = torch.Generator(device="cuda").manual_seed(7)
    o = torch.randn((512, 1, H, 512), generator=g, device="cuda").to(torch.bfloat16)
    w_vc = (torch.randn((H, 512, 128), generator=g, device="cuda") / 22.6).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full((512, 1, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    z = torch.empty((80, 1, H, 512), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        mla.project_out(o, w_vc, y, status=st)
        mla.absorb_q(y[:80], y.view(H, 128, 512), z, status=st)
        y.fill_(float("nan"))
        mla.project_out(o, w_vc, y, status=st)
        mla.absorb_q(y[:80], y.view(H, 128, 512), z, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check(y.view(512, H, 128), o.view(512, H, 512), w_vc)
    _check(z.view(80, H, 512), y[:80].view(80, H, 128), y.view(H, 128, 512))
