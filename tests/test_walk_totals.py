"""The walks' closed-form lengths (KvWalk::total, QWalk::total in ring.cuh),
which the kernels use instead of stepping through every ring step at CTA
start, equal the number of tiles the walks visit, for many mesh geometries
and step ranges.  The check is a host program compiled from ring.cuh."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "head_context_attention_gb300", "csrc")


def test_walk_totals_match_walked_lengths(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "walk_totals"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "native", "walk_totals.cpp"),
                    "-o", str(exe)], check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout
    assert "0 mismatches" in r.stdout
