"""Host side of the library's two builds, without a GPU: the trace build
(libw4a16_trace.so, decode timeline stamps compiled in) compiles and exports
every symbol the header declares, the default build is what the binding
loads unless W4A16_LIBRARY=trace, and unknown variants are refused."""
import ctypes
import os
import re

import pytest

from w4a16_group_quantised_gb300 import binding
from w4a16_group_quantised_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_path_follows_the_variant(monkeypatch):
    monkeypatch.delenv("W4A16_LIBRARY", raising=False)
    assert os.path.basename(binding.library_path()) == "libw4a16.so"
    monkeypatch.setenv("W4A16_LIBRARY", "trace")
    assert os.path.basename(binding.library_path()) == "libw4a16_trace.so"
    monkeypatch.setenv("W4A16_LIBRARY", "fast")
    with pytest.raises(ValueError):
        binding.library_path()


def test_unknown_build_variant_is_refused():
    with pytest.raises(ValueError):
        libbuild.build(variant="debug")


def test_trace_build_exports_the_boundary():
    path = libbuild.build(variant="trace")
    assert os.path.basename(path) == "libw4a16_trace.so"
    assert path != libbuild.build()
    header = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "w4a16.h")).read(), flags=re.S)
    names = sorted(set(re.findall(r"\bint\s+(w4a16_\w+)\s*\(", header)))
    assert "w4a16_debug_decode_trace" in names
    lib = ctypes.CDLL(path)
    for n in names:
        assert hasattr(lib, n), n
