"""The index-checked debug build (libfp8fg_debug.so, compiled with
FP8FG_DEBUG): every kernel store first checks its index against the extent of
the buffer it writes, records ERR_BOUNDS and skips the store when it falls
outside -- an out-of-bounds write check that needs no memory-checker tool.

Its self-test plants a store past a claimed extent (inside a real allocation)
and must see ERR_BOUNDS with the store skipped; the release build's self-test
writes through with status OK.  Then the small-shape GPU parity suite -- every
kernel family, ragged tails, empty groups and tokens, output leading
dimensions, the guard bands of every output -- runs again in a child process
on the debug build and must pass unchanged: no store of those cases falls
outside its buffer, and the checks do not change a single output."""
import os
import re
import subprocess
import sys

import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
from gpu_helpers import assert_status_ok

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Left out of the debug rerun: the full-size and exhaustive cases (minutes of
# oracle time, the same kernels and code paths as the small cases), the
# bounded-wait self-test, and this file's rerun itself.
_DEBUG_RERUN_EXCLUDE = ("full_size", "headline", "sampled", "mlp_size", "every_bf16", "every_scale",
                        "wait_times_out", "debug_build_rerun")


def test_selftest_bounds_in_the_loaded_build():
    buf = torch.zeros(1000, dtype=torch.float32, device="cuda")
    fg.selftest_bounds(buf, 1000)               # the whole buffer claimed: no error in either build
    assert_status_ok()
    assert bool((buf == 1).all())
    buf.zero_()
    fg.selftest_bounds(buf, 600)                # 400 stores past the claimed extent
    st = fg.device_status()
    if fg.debug_build():
        assert st == fg.ERR_BOUNDS
        assert bool((buf[:600] == 1).all()) and bool((buf[600:] == 0).all())
    else:
        assert st == fg.OK
        assert bool((buf == 1).all())
    fg.selftest_bounds(buf, 0)                  # nothing claimed
    st = fg.device_status()
    assert st == (fg.ERR_BOUNDS if fg.debug_build() else fg.OK)


def test_selftest_bounds_rejects_bad_extents():
    buf = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(fg.Fp8Error) as e:
        fg.selftest_bounds(buf, 17)
    assert e.value.code == fg.ERR_INVALID_ARG
    with pytest.raises(fg.Fp8Error):
        fg.selftest_bounds(buf, -1)


def test_debug_build_rerun_of_small_parity_suite():
    if fg.debug_build():
        pytest.skip("already running on the debug build")
    from fp8_fine_grained_x128_gb300 import build as b
    b.build(debug=True)
    env = dict(os.environ, FP8FG_DEBUG="1")
    sel = " and ".join(f"not {k}" for k in _DEBUG_RERUN_EXCLUDE)
    cmd = [sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
           "-k", sel, "--ignore=tests/test_gpu_mlp_step.py", "--ignore=tests/test_gpu_division_exhaustive.py"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = "\n".join((p.stdout + p.stderr).splitlines()[-40:])
    assert p.returncode == 0, f"debug-build rerun failed:\n{tail}"
    m = re.search(r"(\d+) passed", tail)
    assert m and int(m.group(1)) >= 120 and " failed" not in tail, tail
