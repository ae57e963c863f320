"""The oracle and the CUDA path share no code: neither imports, includes or
loads anything of the other, and the only module both use is the seeded input
generator `synth` (tested here statically, on the sources)."""

import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp8_quantized_moe_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _sources(top, exts):
    for d, dirs, files in os.walk(top):
        dirs[:] = [x for x in dirs if not x.startswith(("_build", "__pycache__"))]
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def _code(path):
    text = open(path, encoding="utf-8").read()
    if path.endswith(".py"):
        text = re.sub(r'"""(.*?)"""', "", text, flags=re.S)  # docstrings may name the other side
        text = re.sub(r"#.*", "", text)
    else:
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//.*", "", text)
    return text


def test_product_path_never_references_the_oracle():
    for path in _sources(PKG, (".py", ".cu", ".cuh", ".h")):
        code = _code(path)
        assert not re.search(r"\boracle\b", code), path
    for path in _sources(os.path.join(ROOT, "include"), (".h",)):
        assert not re.search(r"\boracle\b", _code(path)), path


def test_oracle_never_references_the_product_path():
    for path in _sources(ORACLE, (".py", ".c", ".h")):
        code = _code(path)
        assert "fp8_quantized_moe_gb300" not in code, path
        assert "moefp8" not in code and "csrc" not in code, path
        assert not re.search(r"#\s*include\s*\"", code), path  # system headers only


def test_the_shared_input_generator_holds_no_method_arithmetic():
    code = _code(os.path.join(ROOT, "synth", "__init__.py"))
    for word in ("e4m3", "absmax", "quantize", "silu", "swiglu", "fp8"):
        assert word not in code.lower(), word
