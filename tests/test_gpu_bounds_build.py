"""The bounds-checking build (libmoe_gb300_bounds.so, MOE_BOUNDS_CHECK=1).

Its kernels check each index they derive from their own arithmetic (a row
from group offsets and tile numbers, a permuted row from a rank) before the
access, and record MOE_ERR_BOUNDS and skip the access when it falls outside
the tensor, in place of a memory checker, which this GPU pool does not run.
Here: the check itself fires in that build (and not in the release build),
and the GPU parity suites of the permute, the combine, the grouped matmuls
(one-CTA, pairs, fused forms, MX) and the layer pass unchanged on it: every
one of those tests reads the status word, so no derived index left its
tensor on any of their inputs."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_permute.py", "tests/test_gpu_combine.py", "tests/test_gpu_gmm.py",
          "tests/test_gpu_fused.py", "tests/test_gpu_mx.py", "tests/test_gpu_layer.py"]


def _run(args, timeout):
    env = dict(os.environ, MOE_GB300_BOUNDS_CHECK="1")
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


@pytest.mark.gpu
def test_bounds_check_fires_only_in_the_bounds_build():
    import moe_routed_expert_gb300 as M
    from moe_routed_expert_gb300 import build
    build.build(bounds=True)
    # release library in this process: the check compiles to nothing
    ws = M.Workspace(256)
    M.check_bounds(ws)
    assert M.read_status(ws) == 0
    # bounds build in a child process
    code = ("import moe_routed_expert_gb300 as M; M.load(); assert M.bounds_checking(); "
            "assert M.lib_path().endswith('libmoe_gb300_bounds.so'); "
            "ws = M.Workspace(256); M.check_bounds(ws); print(M.read_status(ws))")
    r = _run(["-c", code], timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert r.stdout.strip().splitlines()[-1] == "7"   # MOE_ERR_BOUNDS


@pytest.mark.gpu
def test_gpu_suites_pass_on_the_bounds_build():
    from moe_routed_expert_gb300 import build
    build.build(bounds=True)
    r = _run(["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *SUITES], timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
