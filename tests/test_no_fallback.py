"""The product path has no CPU fallback: the binding fails loudly without its
CUDA library, and neither the package nor the CUDA sources reach the oracle."""
import os
import re
import subprocess
import sys

import pytest

import speculative_decoding_draft_round_gb300 as ds

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_decoding_draft_round_gb300")


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(ds, "LIB_PATH", str(tmp_path / "libdspark.so"))
    monkeypatch.setattr(ds, "_lib", None)
    with pytest.raises(RuntimeError, match="libdspark.so is missing"):
        ds.lib()


def test_package_sources_do_not_reach_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle\b|from\s+oracle\b)|dspark_oracle|oracle/", re.M)
    hits = []
    for dirpath, _, files in os.walk(PKG):
        if "__pycache__" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp", ".c")):
                path = os.path.join(dirpath, f)
                if pat.search(open(path, encoding="utf-8").read()):
                    hits.append(os.path.relpath(path, ROOT))
    assert hits == []


def test_importing_the_package_loads_no_oracle():
    code = ("import sys; import speculative_decoding_draft_round_gb300 as ds; "
            "from speculative_decoding_draft_round_gb300 import workloads; "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "False"
