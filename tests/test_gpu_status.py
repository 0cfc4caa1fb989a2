"""A wait that runs out is reported, and leaves the context usable.

The schedule's test hook (REM_TEST_SKIP_FIRST_STAGE) makes each CTA's
producer issue no copy for its first pipeline stage, with a 2 ms bound on
every wait: the consumers' wait for that stage runs out, the producer's
wait for its release runs out, and on the tensor-core engine the MMA warp's
wait for the first unit runs out too.  Nothing is left in flight (no copy
was issued for the skipped stage; the others land before the CTA exits), so
the kernel returns: every output it could not finish is NaN, and
rem_device_status reports the event until it is cleared.  A normal call on
the same context then matches the oracle.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import quantized_few_row_gb300 as rem
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rem.build()
    rem.load()
    torch.cuda.init()


# (format, engine, m): on the tensor cores m picks the tile width and who
# converts the inputs -- 1 (MP 1, the MMA warps, the early accumulator read),
# 3 (MP 4, the MMA warps), 8 (MP 8, the consumer warps), 16 (MP 16, the
# consumer warps)
CASES = [("q8_0", rem.ENGINE_SIMT, 3), ("q8_0", rem.ENGINE_TC, 3), ("q6_K", rem.ENGINE_TC, 3), ("f16", rem.ENGINE_SIMT, 3),
         ("q4_K", rem.ENGINE_SIMT, 3), ("q6_K", rem.ENGINE_TC, 1), ("q6_K", rem.ENGINE_TC, 8),
         ("q5_0", rem.ENGINE_TC, 16)]


@pytest.mark.parametrize("fmt,engine,m", CASES, ids=[f"{f}-{'tc' if e else 'simt'}-m{m}" for f, e, m in CASES])
def test_wait_that_runs_out_is_reported(fmt, engine, m):
    assert rem.rem_device_status(True) in (rem.REM_OK, rem.REM_ECUDA)   # start clean
    assert rem.rem_device_status(False) == rem.REM_OK
    n, k = 300, 2048
    w, x = H.contiguous(fmt, n, k, m, 770, 771)
    hook = rem.Schedule(engine=engine, wait_ns=2_000_000, test_flags=rem.TEST_SKIP_FIRST_STAGE)
    y = H.run_sched(w, fmt, n, k, 1, x, m, k, 0, n, 0, m * n, hook)
    assert np.all(np.isnan(y)), int(np.isnan(y).sum())
    assert rem.rem_device_status(False) == rem.REM_ECUDA
    assert "bounded wait" in rem.rem_last_error()
    assert rem.rem_device_status(True) == rem.REM_ECUDA       # reported once more, then cleared
    assert rem.rem_device_status(False) == rem.REM_OK
    y_ref, a_ref = oracle.matvec(w, fmt, n, k, 1, x, m, k, 0)
    y = H.run_sched(w, fmt, n, k, 1, x, m, k, 0, n, 0, m * n, rem.Schedule(engine=engine))
    H.assert_close_to_oracle(y.reshape(1, m, n), y_ref, a_ref, f"{fmt} after the timeout")
    assert rem.rem_device_status(False) == rem.REM_OK
