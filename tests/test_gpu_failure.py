"""Failure detection on the GPU without a fault: a kernel waits, with the same
bounded wait the GEMM pipelines use, on an mbarrier that nothing arrives on.
The wait runs out after a short limit, the kernel returns and reports
DG_DEVFLAG_TIMEOUT through the device status word; the context stays usable
and the next GEMM still matches the oracle bit for bit."""
import time

import numpy as np
import pytest
import torch

import moe_grouped_gemm_x128_gb300 as dg
import oracle
from helpers import exact_dense

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    dg.load()
    dg.dg_read_device_status()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_bounded_wait_runs_out_and_reports_timeout():
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dg.dg_selftest_wait_timeout(2_000_000)          # about a millisecond of SM cycles
    flags = dg.dg_read_device_status()              # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert flags & dg.DG_DEVFLAG_TIMEOUT
    assert elapsed < 5.0
    # the C entry point maps the flag to DG_ERR_DEVICE_TIMEOUT, and reading clears it
    dg.dg_selftest_wait_timeout(1000)
    import ctypes
    out = ctypes.c_int(0)
    assert dg.load().dg_read_device_status(ctypes.byref(out), None) == dg.DG_ERR_DEVICE_TIMEOUT
    assert out.value & dg.DG_DEVFLAG_TIMEOUT
    assert dg.dg_read_device_status() == 0


@pytest.mark.parametrize("force", ["", "256"], ids=["one_sm", "pair256"])
def test_next_gemm_after_a_timeout_is_exact(force, monkeypatch):
    monkeypatch.setenv("DG_FORCE_BN", force)
    dg.dg_selftest_wait_timeout(100_000)
    assert dg.dg_read_device_status() & dg.DG_DEVFLAG_TIMEOUT
    a, sfa, b, sfb = exact_dense(300, 520, 640, seed=77)
    d = torch.empty((300, 520), dtype=torch.bfloat16, device="cuda")
    dg.dg_fp8_gemm_nt(dev(a), dev(sfa), dev(b), dev(sfb), d)
    torch.cuda.synchronize()
    got = d.view(torch.int16).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got, oracle.gemm_nt(a, sfa, b, sfb))
    assert dg.dg_read_device_status() == 0


def test_limit_outside_the_allowed_range_is_rejected():
    with pytest.raises(dg.DgError):
        dg.dg_selftest_wait_timeout(10)
    with pytest.raises(dg.DgError):
        dg.dg_selftest_wait_timeout(10 ** 12)
