"""The product and the oracle stay apart, and the product has no fallback:
the package never imports the oracle, the CUDA sources include nothing of it
(nor it of them), and a library that cannot be built makes every call raise."""
import os
import re

import pytest

import grouped_query_decode_gb300 as gq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "grouped_query_decode_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "_build" in d or "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_package_never_imports_the_oracle():
    for path in _files(PKG, (".py",)):
        src = open(path).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), path


def test_cuda_sources_and_oracle_share_no_code():
    for path in _files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h")):
        for inc in re.findall(r'#include\s+"([^"]+)"', open(path).read()):
            assert "oracle" not in inc, (path, inc)
    csrc_names = {os.path.basename(p) for p in _files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h"))}
    for path in _files(ORACLE, (".c", ".h", ".py")):
        src = open(path).read()
        for inc in re.findall(r'#include\s+"([^"]+)"', src):
            assert os.path.basename(inc) not in csrc_names, (path, inc)
        assert not re.search(r"^\s*(import|from)\s+grouped_query_decode_gb300\b", src, re.M), path


def test_a_library_that_cannot_be_built_raises(monkeypatch):
    def broken(*a, **k):
        raise RuntimeError("nvcc failed")

    monkeypatch.setattr(gq, "_lib", None)
    monkeypatch.setattr(gq._build, "build", broken)
    with pytest.raises(RuntimeError):
        gq.load()
    with pytest.raises(RuntimeError):
        gq.gqa_decode_workspace_bytes(1, 1, 8, 2, 128, 64)
