"""Failure detection on the GPU without a fault: a pipeline wait that nothing
completes must expire within its limit, stop the other waiting role through
the shared abort flag, and leave MOE_ERR_TIMEOUT in the workspace's status
word, with the CUDA context still usable afterwards (the next launches run and
give correct results)."""
import time

import numpy as np
import pytest

import oracle as O
from tests._util import assert_close, dev, dev_bf16, f64
from workloads import normal_bf16

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 6


@pytest.mark.parametrize("timeout_ns", [20_000, 2_000_000])
def test_bounded_wait_expires_and_reports_timeout(timeout_ns):
    import moe_routed_expert_gb300 as M
    ws = M.Workspace(256)
    ws.reset()
    assert M.read_status(ws) == 0
    t0 = time.perf_counter()
    M.check_wait_timeout(ws, timeout_ns=timeout_ns)
    assert M.read_status(ws) == MOE_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 1.0          # the second waiter stopped on the flag, not its own limit
    # the status is sticky until cleared, and the context keeps working
    M.check_wait_timeout(ws, timeout_ns=timeout_ns)
    assert M.read_status(ws) == MOE_ERR_TIMEOUT
    ws.reset()
    assert M.read_status(ws) == 0
    rng = np.random.default_rng(3)
    gl = np.array([100, 0, 156], np.int64)
    x = normal_bf16(rng, (256, 128))
    w = normal_bf16(rng, (3, 128, 256), 1 / np.sqrt(128))
    y = M.gmm_forward(dev_bf16(x), dev_bf16(w), dev(gl), ws=ws)
    assert M.read_status(ws) == 0
    assert_close("y", y, O.gmm_forward(f64(x), f64(w), gl))
