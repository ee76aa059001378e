"""The binding has no fallback: importing it where libfcp.so has not been
built raises (a copy of the binding in a temporary package with no _lib/),
so no code path can silently run without the CUDA library."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_import_without_library_raises(tmp_path):
    pkg = tmp_path / "fcp_copy"
    pkg.mkdir()
    (pkg / "__init__.py").write_text("")
    shutil.copy(os.path.join(ROOT, "context_document_masked_gb300", "fcp.py"), pkg / "fcp.py")
    code = ("import sys\n"
            "try:\n"
            "    import fcp_copy.fcp\n"
            "except ImportError as e:\n"
            "    print('ImportError:', e); sys.exit(0)\n"
            "sys.exit(3)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True,
                       env={**os.environ, "PYTHONPATH": str(tmp_path)}, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "not built" in r.stdout


def test_checked_build_selection_without_library_raises(tmp_path):
    """FCP_DEVICE_CHECKS=1 selects _lib_checked/: missing, it raises too."""
    pkg = tmp_path / "fcp_copy"
    pkg.mkdir()
    (pkg / "__init__.py").write_text("")
    shutil.copy(os.path.join(ROOT, "context_document_masked_gb300", "fcp.py"), pkg / "fcp.py")
    (pkg / "_lib").mkdir()   # the plain build present, the checked one not
    src = os.path.join(ROOT, "context_document_masked_gb300", "_lib", "libfcp.so")
    if not os.path.exists(src):
        pytest.skip("plain library not built here")
    shutil.copy(src, pkg / "_lib" / "libfcp.so")
    code = ("import sys\n"
            "try:\n"
            "    import fcp_copy.fcp as f\n"
            "except ImportError as e:\n"
            "    print('ImportError:', e); sys.exit(0)\n"
            "sys.exit(3)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True,
                       env={**os.environ, "PYTHONPATH": str(tmp_path), "FCP_DEVICE_CHECKS": "1"}, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "_lib_checked" in r.stdout
