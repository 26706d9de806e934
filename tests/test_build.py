"""The build driver: processes that build at once (the ranks of one job each
call build()) take turns on a lock file and end with the same library."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="needs the CUDA toolkit")
def test_concurrent_builds_share_the_lock():
    code = ("import sys; sys.path.insert(0, %r); "
            "from fp8_packed_reduced_gb300 import build as b; print(b.build())" % ROOT)
    procs = [subprocess.Popen([sys.executable, "-c", code], stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for _ in range(3)]
    outs = [p.communicate(timeout=900) for p in procs]
    assert [p.returncode for p in procs] == [0, 0, 0], [e for _, e in outs]
    libs = {o.strip().splitlines()[-1] for o, _ in outs}
    assert len(libs) == 1
    lib = libs.pop()
    assert os.path.exists(lib) and os.path.exists(lib + ".sha256")
