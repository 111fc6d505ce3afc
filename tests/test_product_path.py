"""The product path on a host without a GPU: the binding raises when the
library has not been built (there is no fallback), and neither the binding
nor the library reaches the oracle, which is test infrastructure only."""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_84_gb300")


def test_missing_library_raises(monkeypatch, tmp_path):
    import paged_kv_cache_84_gb300 as pkv
    monkeypatch.setattr(pkv, "_lib", None)
    monkeypatch.setattr(pkv, "LIB_PATH", str(tmp_path / "libpkv.so"))
    with pytest.raises(ImportError, match="no fallback"):
        pkv.plan_request_kernels([0, 1], [5], 8, 4, 64)
    with pytest.raises(ImportError):
        pkv.attention_workspace_bytes(1, 1, 8, 64, 16)


def test_binding_and_library_do_not_reach_the_oracle():
    code = ("import sys; import paged_kv_cache_84_gb300 as p; from paged_kv_cache_84_gb300 import build; "
            "build.build(); p.plan_request_kernels([0, 3, 4], [9, 42], 8, 4, 48); "
            "p.plan_attention([0, 3, 4], [9, 42], 8, 4, 48, num_sms=152); "
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]; "
            "assert not bad, bad")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    # no source of the package or its library names the oracle in code (comments aside)
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if not f.endswith((".py", ".cu", ".cuh", ".h", ".cpp", ".c")):
                continue
            text = open(os.path.join(dirpath, f)).read()
            includes = re.findall(r"^\s*#\s*include\s*[<\"]([^>\"]+)", text, flags=re.M)
            assert not any("oracle" in inc for inc in includes), f"{f} includes the oracle"
            text = re.sub(r"/\*.*?\*/|//[^\n]*|#[^\n]*|\"\"\".*?\"\"\"", "", text, flags=re.S)
            assert not re.search(r"\boracle\b", text), f"{f} refers to the oracle"
