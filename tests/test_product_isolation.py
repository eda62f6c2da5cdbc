"""The product path stands apart from the oracle (CPU): importing the package
and its modules loads nothing under oracle/, the CUDA library's sources
include nothing of the oracle, and a missing library makes the binding fail
loudly instead of computing anything another way."""
import glob
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(code):
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    return r.stdout


def test_package_imports_no_oracle_module():
    out = _run(
        "import sys\n"
        "import bit_plane_kv_gb300, bit_plane_kv_gb300.binding, bit_plane_kv_gb300.synth\n"
        "import bit_plane_kv_gb300.fidelity, bit_plane_kv_gb300.build\n"
        "print(sorted(m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')))\n")
    assert out.strip() == "[]"


def test_cuda_sources_share_nothing_with_the_oracle():
    for path in glob.glob(os.path.join(ROOT, "bit_plane_kv_gb300", "csrc", "*")) + \
            glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path, encoding="utf-8").read()
        assert "oracle" not in text.lower(), path
    text = open(os.path.join(ROOT, "oracle", "fathom_oracle.c"), encoding="utf-8").read()
    assert "#include \"" not in text          # only system headers


def test_missing_library_fails_loudly():
    out = _run(
        "from bit_plane_kv_gb300 import binding as B\n"
        "B.LIB_PATH = '/nonexistent/libfathom.so'\n"
        "B._lib = None\n"
        "try:\n"
        "    B.lib()\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n")
    assert out.startswith("raised: libfathom is not built")
