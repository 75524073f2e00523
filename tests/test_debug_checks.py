"""The build with device bounds checks (MOE_DEBUG_CHECKS=1): it compiles for
sm_103a and exports the same C ABI (CPU), and on a GPU it runs the smoke
layers clean -- every table entry the checks read is in range, so the status
stays MOE_OK and both paths match the oracle (subprocesses: the variable
selects the library when the package is imported)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(code, timeout):
    env = dict(os.environ, MOE_DEBUG_CHECKS="1")
    return subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True,
                          timeout=timeout)


def test_debug_checks_library_builds_and_exports_the_abi():
    code = ("import __graft_entry__ as g; g.build(); import expert_routed_ffn_moe_gb300 as m; L = m.lib(); "
            "missing = [n for n in m.header_functions() if not hasattr(L, n)]; "
            "print(m.LIB); print('missing', missing)")
    r = _run(code, timeout=1800)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = r.stdout.strip().splitlines()
    assert lines[-2].endswith("libmoe_gb300_debug.so")
    assert lines[-1] == "missing []"


@pytest.mark.gpu
def test_debug_checks_smoke_runs_clean():
    r = _run("import __graft_entry__ as g; g.smoke()", timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
