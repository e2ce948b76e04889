"""Device-side failure detection without a fault: a barrier that nothing
arrives on makes the bounded wait run out; the kernel records
PKV_DEVERR_WAIT_TIMEOUT, frees what it holds and returns, and the context
stays usable (the next append + decode still matches the oracle)."""

import time

import numpy as np
import pytest

import paged_kv_cache_222_gb300 as pkv
import workloads as W
from tests import gpu_support as S

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PKV_DEVERR_WAIT_TIMEOUT = 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_222_gb300 import build
    build.build()
    pkv.library()
    assert pkv.device_error(DEV) == 0
    yield
    assert pkv.device_error(DEV) == 0


@pytest.mark.parametrize("which", [0, 1])
def test_wait_runs_out_and_is_reported(which):
    t0 = time.perf_counter()
    assert pkv.selftest_wait_timeout(which, limit_us=20000, device=DEV) == PKV_DEVERR_WAIT_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.015 < elapsed < 5.0, elapsed
    assert pkv.device_error(DEV) == 0                     # read clears it


def test_context_usable_after_time_out():
    for which in (1, 1, 0):                               # tensor memory is freed each time
        assert pkv.selftest_wait_timeout(which, limit_us=5000, device=DEV) == PKV_DEVERR_WAIT_TIMEOUT
    spec = dict(B=3, H_q=16, H_kv=2, D=128, bs=16, kv="bf16", free_frac=0.25, steps=1, seed=4242,
                q_mult=1.0, ctx=(1, 200, 777))
    case = W.make_case(spec, device=DEV)
    S.poison_unused(case)
    snaps = {(b, h): S.snapshot_sequence(case, b, h) for b in range(3) for h in range(2)}
    out = S.run_step(case, 0).cpu().numpy()
    assert pkv.device_error(DEV) == 0
    G = 8
    for b in range(3):
        for h in range(2):
            ref = S.oracle_unit(case, b, h, 0, snaps[(b, h)])
            assert np.max(np.abs(out[b, h * G:(h + 1) * G] - ref)) <= 2e-3
