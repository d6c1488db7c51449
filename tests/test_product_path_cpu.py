"""The product path stands apart from the oracle and has no fallback: nothing in the
package imports, includes or links the oracle, and the binding raises when the CUDA
library has not been built instead of computing anything itself."""
import glob
import os
import re

import pytest

from quantized_attention_layer_gb300 import hfa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "quantized_attention_layer_gb300")


def test_package_sources_never_reach_the_oracle():
    py = glob.glob(os.path.join(PKG, "*.py"))
    native = glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*"))
    assert py and native
    for path in py:
        text = open(path).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), path
        assert "liborc" not in text, path
    for path in native:
        text = open(path, errors="replace").read()
        assert not re.search(r'#include\s+[<"][^>"]*oracle', text), path
        assert "liborc" not in text, path


def test_binding_raises_when_the_library_is_missing(monkeypatch):
    monkeypatch.setattr(hfa, "_lib", None)
    monkeypatch.setattr(hfa, "LIB_PATH", os.path.join(PKG, "no_such_libhfa.so"))
    with pytest.raises(RuntimeError, match="missing"):
        hfa.lib()
