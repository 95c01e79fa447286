"""The bounded wait of the TMA-staged reduce pass, made to run out: an mbarrier
phase that nothing completes.  The wait must give up by itself, set the abort
flag and the error word (which the step status turns into ZERO_ETIMEOUT), end
the kernel within seconds, and leave the context usable for the next step."""
import ctypes
import os
import subprocess
import sys
import time

import numpy as np
import pytest

import harness as H

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
POLLS = 4096                   # the helper's limit
LIBRARY_POLLS = 1 << 20        # ZERO_TMA_WAIT_LIMIT in the library


@pytest.fixture(scope="module")
def helper(tmp_path_factory):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = tmp_path_factory.mktemp("bw") / "libbounded_wait_check.so"
    csrc = os.path.join(ROOT, "zero_sharded_mixed_02_gb300", "csrc")
    # a short limit (4096 polls) keeps the test quick whatever one poll takes; the
    # time per poll it measures bounds the library's own limit
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    f"-DZERO_TMA_WAIT_LIMIT={POLLS}u",
                    "-shared", "-Xcompiler", "-fPIC", "-I", csrc,
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "bounded_wait_check.cu"), "-o", str(out)],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(str(out))
    lib.bounded_wait_on_nothing.restype = ctypes.c_int
    return torch, lib


def test_wait_on_an_uncompleted_phase_gives_up(helper):
    torch, lib = helper
    ret, err, abort = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
    cycles = ctypes.c_longlong(0)
    t0 = time.monotonic()
    rc = lib.bounded_wait_on_nothing(ctypes.byref(ret), ctypes.byref(err), ctypes.byref(cycles),
                                     ctypes.byref(abort))
    elapsed = time.monotonic() - t0
    assert rc == 0                                       # no CUDA error: the kernel ended
    assert ret.value == 1 and err.value == 1 and abort.value == 1
    assert cycles.value > 0 and elapsed < 30.0
    # the library's limit, at the measured cycles per poll and 2 GHz, gives up within 10 s
    assert cycles.value / POLLS * LIBRARY_POLLS / 2.0e9 < 10.0, cycles.value


def test_context_usable_after_the_wait_gave_up(helper):
    torch, lib = helper
    ret, err, abort = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
    cycles = ctypes.c_longlong(0)
    assert lib.bounded_wait_on_nothing(ctypes.byref(ret), ctypes.byref(err),
                                       ctypes.byref(cycles), ctypes.byref(abort)) == 0
    sys.path.insert(0, os.path.join(ROOT))
    from zero_sharded_mixed_02_gb300 import build
    build.build()
    import zero_sharded_mixed_02_gb300 as z
    c = H.Case(shapes=[(5000,)], nd=4, clip=1.0, steps=2)
    gpu = H.run_gpu(z, c)
    assert [r["t"] for r in gpu.results] == [1, 2]
    assert np.all(np.isfinite(gpu.master))
