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


def test_binding_checks_device_metadata_sizes():
    """The library sees only pointers, so the binding checks that the device
    metadata has an entry for every request before anything is passed on
    (here with host tensors: the size check comes before the device check)."""
    import torch

    import paged_kv_cache_84_gb300 as pkv
    from paged_kv_cache_84_gb300 import build
    build.build()
    q = torch.zeros(4, 8, 64, dtype=torch.bfloat16)
    pool = torch.zeros(9, 16, 4, 64, dtype=torch.bfloat16)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    qsl_h, sl_h = [0, 3, 4], [9, 42]
    good = dict(qsl=torch.tensor(qsl_h, dtype=torch.int32), sl=torch.tensor(sl_h, dtype=torch.int32),
                bt=torch.zeros(2, 3, dtype=torch.int32))
    bad = [dict(good, bt=torch.zeros(1, 3, dtype=torch.int32)),      # one table row for two requests
           dict(good, bt=torch.zeros(6, dtype=torch.int32)),         # not [num_reqs, width]
           dict(good, qsl=torch.tensor([0, 3], dtype=torch.int32)),  # query_start_loc too short
           dict(good, sl=torch.tensor([9], dtype=torch.int32))]      # seq_lens too short
    for m in bad:
        with pytest.raises(ValueError):
            pkv.ragged_paged_attention(torch.empty_like(q), q, pool, pool, m["qsl"], m["sl"], m["bt"],
                                       qsl_h, sl_h, 3, 42, 0.125, ws)
        with pytest.raises(ValueError):
            pkv.paged_kv_write_attention(torch.zeros(4, 4, 64, dtype=torch.bfloat16),
                                         torch.zeros(4, 4, 64, dtype=torch.bfloat16), pool, pool,
                                         torch.zeros(4, dtype=torch.int64), torch.empty_like(q), q,
                                         m["qsl"], m["sl"], m["bt"], qsl_h, sl_h, 3, 42, 0.125, ws)
    with pytest.raises(TypeError):                                   # sizes fine: host tensors refused
        pkv.ragged_paged_attention(torch.empty_like(q), q, pool, pool, good["qsl"], good["sl"], good["bt"],
                                   qsl_h, sl_h, 3, 42, 0.125, ws)
