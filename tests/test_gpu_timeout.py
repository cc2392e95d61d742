"""The decode kernel's bounded waits: a wait that runs out is reported, and the
GPU context stays usable.

A test-only build of the library (macro KVATTN_TEST_STALL, compiled into its
own directory, never the library that ships) lets a call ask, through a bit
of its status word, that every decode warp first wait, with a limit of about a
millisecond, on a shared-memory barrier that nothing arrives at and that no
copy is ever issued to.  The wait runs out, the warp records
KVATTN_DEV_TIMEOUT, stops consuming, lets the tile copies it already issued
land, and leaves.  A child process that loads only that build (two copies of
the library, each with its own static CUDA runtime, do not share a process
well) checks that the bit reaches kvattn_read_device_status, then
re-initialises the workspace and decodes without the request on the same
context: the result must match the oracle.  No GPU fault, trap or hang is
involved: every wait ends.
"""
import os
import subprocess
import sys

import pytest

from decode_phase_gqa_gb300 import build as B

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    path = B.build(variant="teststall", extra_flags=["-DKVATTN_TEST_STALL"])
    r = subprocess.run([sys.executable, "-m", "tests.stall_child", path], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "stall-child ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
