"""The oracle and the CUDA path share no code and neither imports the other.

Static checks over the source trees: no file under oracle/ names the CUDA
package or its sources, and no file of the package names the oracle. Only
the input generators (workload/) serve both, and they hold none of the
layer's arithmetic.
"""
from __future__ import annotations

import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PACKAGE = "mxfp4_weight_mxfp8_gb300"


def sources(folder, suffixes=(".py", ".c", ".h", ".cu", ".cuh", ".cpp")):
    base = os.path.join(ROOT, folder)
    for dirpath, dirnames, files in os.walk(base):
        dirnames[:] = [d for d in dirnames if not d.startswith("_build") and d != "__pycache__"]
        for f in files:
            if f.endswith(suffixes):
                yield os.path.join(dirpath, f)


def test_oracle_does_not_reference_the_cuda_path():
    for path in sources("oracle"):
        text = open(path, encoding="utf-8").read()
        assert PACKAGE not in text.replace(f"under {PACKAGE}/", ""), path
        assert not re.search(r"#include\s+[<\"].*(csrc|include/)", text), path


def test_cuda_path_does_not_reference_the_oracle():
    for path in list(sources(PACKAGE)) + list(sources("include")):
        text = open(path, encoding="utf-8").read()
        assert not re.search(r"\boracle\b", text), path


def test_workload_imports_neither_side():
    for path in sources("workload"):
        text = open(path, encoding="utf-8").read()
        assert not re.search(r"^\s*(from|import)\s+(oracle|%s)" % PACKAGE, text, re.M), path
