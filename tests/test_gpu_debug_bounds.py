"""The bounds-checked build of the library (TQ_DEBUG_BOUNDS, libtq_debug.so).

In that build every index the kernels compute into shared or global memory is
checked against the extent of the buffer it addresses; an index outside sets
TQ_ERR_DEVICE_BOUNDS in the device error word and the access is redirected
inside the buffer (a copy is dropped).  Nothing faults, traps or waits forever.

The test runs the quantize, append and decode parity suites (tiny and odd
shapes among them: 1, 2 and 31 tokens, lengths one token either side of a
split boundary, windows spread over several splits, QJL and Direct Sign keys,
multi-query decode) in a child process that loads the debug library.  Every
case reads the error word back and expects TQ_OK, except the cases that
provoke a bounds error on purpose, which expect exactly that error.
("TurboQuant KV 캐시 압축 for llama.cpp", v1.1.0 bug fixes: a __syncthreads
race on the query-WHT shared memory is the kind of fault such checks expose.)
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_parity_suites_pass_on_the_bounds_checked_library():
    if os.environ.get("TQ_LIB_VARIANT") == "debug":
        pytest.skip("already inside the bounds-checked run")
    env = dict(os.environ, TQ_LIB_VARIANT="debug")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "gpu",
           "tests/test_gpu_quantize.py", "tests/test_gpu_decode.py",
           "tests/test_gpu_debug_bounds.py::test_child_loads_the_debug_library"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=3600)
    tail = r.stdout[-4000:] + "\n" + r.stderr[-2000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail


@pytest.mark.gpu
def test_child_loads_the_debug_library():
    """Runs inside the child above: the binding loaded libtq_debug.so."""
    if os.environ.get("TQ_LIB_VARIANT") != "debug":
        pytest.skip("only meaningful inside the bounds-checked run")
    from kv_cache_quantization_random_gb300 import binding as B
    B.load(build_if_missing=True)
    assert B.lib_path().endswith("libtq_debug.so")
    assert os.path.exists(B.lib_path())
