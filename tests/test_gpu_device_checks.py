"""The checked build of the library on valid inputs.

Built with FCP_DEVICE_CHECKS=1, every index the kernels read from a plan's
device tables (work order, tiles, pieces, key segments, backward units,
preprocess row chunks, gather runs) is checked on the device against the
table sizes and against the rows of the tensor it addresses before it is used;
a failed check sets an error bit that fcp_get_device_status reports as
FCP_ERR_INVALID_ARG, and the kernel skips that work unit instead of trapping.
This test builds that library and runs the GPU parity suites of the attention
kernels, the ring-order forward, the online-softmax rescale cases and the
closed-form edge cases through it, in a child process that selects it with
FCP_DEVICE_CHECKS=1: every case must pass with no error bit set (those tests
read the device status after their calls). Corrupt tables are never fed to the
GPU; the host rejects corrupted plan handles before any launch
(test_cabi_validation.py).
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_passes_the_parity_suites(cuda):
    from context_document_masked_gb300 import build as b
    lib = b.build(checked=True)
    assert os.path.exists(lib) and "_lib_checked" in lib
    env = dict(os.environ, FCP_DEVICE_CHECKS="1")
    probe = subprocess.run([sys.executable, "-c",
                            "from context_document_masked_gb300 import fcp; print(fcp.CHECKED, fcp.LIB_PATH)"],
                           env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert probe.returncode == 0 and probe.stdout.split()[0] == "True" and "_lib_checked" in probe.stdout
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        "tests/test_gpu_attention.py", "tests/test_gpu_ring.py", "tests/test_gpu_rescale.py",
                        "tests/test_gpu_edges.py"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1800)
    tail = r.stdout[-3000:] + r.stderr[-2000:]
    print(tail)
    assert r.returncode == 0, tail
