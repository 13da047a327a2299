"""The bounds-checked build (include/mhcpb.h, mhcpb_debug_checked_sites): the
library compiled with -DMHCPB_CHECKED checks every global access its kernels
make at a computed address against its buffer.  In a child process that loads
that build first (tests/checked_run.py), every entry point runs over the
tests' edge shapes, the full training profile included: no access falls
outside its buffer, and the results still match the oracles.  This stands in
for a device-side sanitizer, which this library's tests cannot use."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_finds_no_out_of_range_access():
    run = subprocess.run([sys.executable, os.path.join(HERE, "checked_run.py")], capture_output=True,
                         text=True, timeout=1800)
    assert run.returncode == 0, f"{run.stdout[-3000:]}\n{run.stderr[-3000:]}"
    assert "checked build ok" in run.stdout
