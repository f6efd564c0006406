"""The bounded pipeline wait gives up and returns (failure detection).

Every wait of the decode kernels is bounded: after 2 s of %globaltimer, or as
soon as another warp of the CTA has given up, it returns false and the
kernel ORs MLA_STATUS_WAIT_TIMEOUT into the status word instead of spinning
forever.  mla_debug_wait runs that same wait on a barrier phase that nothing
completes (or that another warp aborts or completes late), with no TMA,
tensor-core or tensor-memory work in flight, so the kernel ends cleanly; a
decode afterwards must still be bitwise the one before.  The argument checks
run on the host (CPU tests).
"""
import pytest
import torch

import mla_latent_decode_gb300 as mla
from mla_latent_decode_gb300 import build, synth

LIMIT_NS = 2_000_000_000


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mla.library()


def test_wait_probe_arguments_checked_on_host(lib):
    """Bad arguments fail before any CUDA call (no GPU needed)."""
    assert lib.mla_debug_wait(3, 0, None, None, None) == -1
    assert lib.mla_debug_wait(0, -1, None, None, None) == -1
    assert lib.mla_debug_wait(1, 2_000_000, None, None, None) == -1
    assert lib.mla_debug_wait(0, 0, None, None, None) == -1
    assert "required" in lib.mla_last_error_string().decode()


def _wait(mode, delay_us):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ns = torch.zeros(1, dtype=torch.int64, device="cuda")
    mla.debug_wait(mode, delay_us, st, ns)
    torch.cuda.synchronize()
    return int(st.item()), int(ns.item())


@pytest.mark.gpu
def test_wait_gives_up_after_its_limit_and_context_stays_usable(lib):
    wl = synth.Workload("wt", 2, 5, 96, [700, 130])
    batch = synth.make_batch(wl, seed=71, device="cuda")
    o0, l0, _ = mla.decode(batch, num_splits=2)
    torch.cuda.synchronize()
    st, ns = _wait(0, 0)  # nothing ever completes the phase
    assert st == mla.STATUS_WAIT_TIMEOUT
    assert LIMIT_NS <= ns < LIMIT_NS + 500_000_000, ns
    o1, l1, _ = mla.decode(batch, num_splits=2)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


@pytest.mark.gpu
def test_wait_gives_up_when_the_cta_aborts(lib):
    st, ns = _wait(1, 3000)  # another warp raises the abort flag after 3 ms
    assert st == mla.STATUS_WAIT_TIMEOUT
    assert 3_000_000 <= ns < 200_000_000, ns


@pytest.mark.gpu
def test_wait_returns_when_the_phase_completes_late(lib):
    st, ns = _wait(2, 3000)  # another warp completes the phase after 3 ms
    assert st == 0
    assert 3_000_000 <= ns < 200_000_000, ns
