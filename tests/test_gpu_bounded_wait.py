"""The bounded mbarrier wait that every pipeline wait of the library uses (csrc/iq_common.cuh),
exercised on the GPU without a fault or a hang: a phase that nothing completes (an mbarrier that
no thread arrives on) makes the wait return false once its limit has passed, a completed phase
returns true at once, and the context stays usable, since the second launch runs after the first.
The kernels turn such a false into IQ_STATUS_TIMEOUT."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_after_its_limit_and_the_context_stays_usable(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    here = os.path.dirname(os.path.abspath(__file__))
    exe = str(tmp_path / "bounded_wait")
    subprocess.run([nvcc, "-O2", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-o", exe,
                    os.path.join(here, "bounded_wait.cu")], check=True, capture_output=True, timeout=900)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = {ln.split()[0]: ln.split()[1:] for ln in r.stdout.splitlines() if ln.strip()}
    ok, ns, limit = (int(x) for x in lines["never-completed"])
    assert ok == 0
    assert limit <= ns < limit + 1_000_000_000
    ok2, ns2 = (int(x) for x in lines["completed"])
    assert ok2 == 1 and ns2 < 1_000_000_000
