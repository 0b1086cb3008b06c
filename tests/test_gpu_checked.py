"""The bounds-checked build of the library (compiled with -DMTP_CHECKED).

compute-sanitizer is not available here, so out-of-bounds writes are looked
for in two other ways: the guard bands that every GPU test places around the
buffers it hands to the library (tests/gpu_util.py), and this build, in which
every output store of the draft, verify and KV kernels is checked against the
extent of its buffer for the call; a store outside is skipped and reported as
MTP_ERR_BOUNDS through the error word.  The GPU tests (all but the full-size
ones) run again in a child process that loads the checked build (the binding
loads the library named by MTP_LIBRARY); each of them asserts a clean error
word after its calls, so any store outside its extent fails it."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

SUITE = ["tests/test_gpu_draft.py", "tests/test_gpu_verify_kv.py", "tests/test_gpu_quant.py",
         "tests/test_gpu_loop.py", "tests/test_gpu_dynamic.py", "tests/test_gpu_tree.py", "tests/test_zz_no_alloc.py"]


def _checked_library() -> str:
    import importlib.util
    spec = importlib.util.spec_from_file_location("_mtp_build_checked",
                                                  os.path.join(ROOT, "mtp_self_speculative_gb300", "_build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(checked=True)


def _run_child(args, timeout):
    env = dict(os.environ, MTP_LIBRARY=_checked_library())
    return subprocess.run([sys.executable] + args, cwd=ROOT, env=env, stdout=subprocess.PIPE,
                          stderr=subprocess.STDOUT, text=True, timeout=timeout)


def test_checked_build_skips_and_reports_an_out_of_range_store():
    """The checked build's self-test sends one store one element past a
    4-element extent through the check: nothing is written, the error word
    reads MTP_ERR_BOUNDS once, then the context drafts cleanly."""
    code = r'''
import sys
sys.path.insert(0, "tests")
import mtp_self_speculative_gb300 as M
assert M._lib.LIB_PATH.endswith("libmtp_checked.so"), M._lib.LIB_PATH
import synth
from gpu_util import F32_LOGIT_TOL
from test_gpu_draft import Case, check_forced
case = Case(synth.TINY_F32)
M.mtp_selftest_bounds(case.ctx)
assert M.mtp_get_device_error(case.ctx) == M.MTP_ERR_BOUNDS
assert M.mtp_get_device_error(case.ctx) == 0
check_forced(case, [0], F32_LOGIT_TOL)
print("checked self-test ok")
'''
    r = _run_child(["-c", code], timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "checked self-test ok" in r.stdout


def test_gpu_suite_runs_clean_on_the_checked_build():
    r = _run_child(["-m", "pytest", "-q", "-x", "-m", "gpu and not slow", "-p", "no:cacheprovider"] + SUITE,
                   timeout=2400)
    assert r.returncode == 0, r.stdout[-4000:]
