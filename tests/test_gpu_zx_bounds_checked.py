"""The bounds-checked build, libnvfp4_checked.so (the library compiled with
NVFP4_CHECK_BOUNDS): before every access its kernels test shared-memory
destinations and operands against the CTA's dynamic shared memory, TMEM
column ranges against the 512 columns, tensor-map x coordinates for 16-byte
alignment, and every plain global load and store against the byte range the
call's arguments grant that tensor; a failed test is counted and its access
skipped, so a wrong index shows up as a recorded site instead of a fault.

test_selftest_counts_the_skipped_stores shows the checks fire (a kernel told
that only part of a caller buffer is its own: the checked build skips and
counts exactly the stores past that part, the normal build makes them all;
every store lies inside the buffer either way).  The last test runs the GPU
suite (parity against the oracle on every route and shape class, edge cases,
failure detection) under the checked build, where tests/conftest.py fails any
test after which a failed address test was recorded."""
import os
import subprocess
import sys

import pytest
import torch

import nvfp4_block_scaled_30_b300 as nv
from conftest import ROOT

pytestmark = pytest.mark.gpu
INNER = os.environ.get("NVFP4_LIB") == "checked"


def test_selftest_counts_the_skipped_stores():
    span = 4096
    buf = torch.zeros(span + 64 + 32, dtype=torch.uint8, device="cuda")
    checked = nv.bounds_checked()
    if checked:
        nv.bounds_record(clear=True)
    nv.bounds_selftest(buf, span)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    if checked:
        n, where, value, limit = nv.bounds_record(clear=True)
        assert n == 64, n
        assert where.startswith("diag_bounds.cu:"), where
        assert span <= value < span + 64 and limit == span
        assert (host[:span] == 1).all() and (host[span:] == 0).all()
    else:
        assert (host[:span + 64] == 1).all() and (host[span + 64:] == 0).all()


@pytest.mark.skipif(INNER, reason="this test starts the checked run itself")
def test_gpu_suite_under_the_bounds_checked_build():
    from nvfp4_block_scaled_30_b300 import build
    build.build(checked=True)
    # all GPU tests but the exhaustive 2^32-pattern conversion check (one
    # flat grid-stride kernel) and the oracle's eight-layer chain (CPU-bound)
    cmd = [sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider",
           "--ignore=tests/test_gpu_2_probe.py", "-k", "not chain_error_vs_oracle"]
    env = dict(os.environ, NVFP4_LIB="checked")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout[-4000:] + "\n" + r.stderr[-2000:]).strip()
    print(tail.splitlines()[-1] if tail else "")
    assert r.returncode == 0, tail
