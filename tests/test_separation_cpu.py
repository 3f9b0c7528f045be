"""The CUDA path and the oracle share no code and neither loads the other.

The package (`mixture_experts_ffn_gemm_gb300/`: the binding, the build, the kernels) must not
import, include or open anything under `oracle/`, and the oracle must not include or import the
package's sources.  The one shared module is `synthetic.py`, which draws seeded tensors and holds
none of the layer's arithmetic; it must not reach either side."""
import ast
import os
import re

from conftest import ROOT

PKG = os.path.join(ROOT, "mixture_experts_ffn_gemm_gb300")
ORC = os.path.join(ROOT, "oracle")


def _files(root, exts):
    for dirpath, dirnames, names in os.walk(root):
        dirnames[:] = [d for d in dirnames if not d.startswith(("_build", "__pycache__"))]
        for n in names:
            if n.endswith(exts):
                yield os.path.join(dirpath, n)


def _imports(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            yield from (a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            yield ("." * node.level) + (node.module or "")


def _includes(path):
    return re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', open(path).read(), re.M)


def test_package_python_never_imports_the_oracle():
    for path in _files(PKG, (".py",)):
        for mod in _imports(path):
            assert not mod.split(".")[0] == "oracle", (path, mod)
        assert "oracle/" not in open(path).read().replace("\\", "/"), path


def test_kernels_never_include_the_oracle():
    for path in _files(PKG, (".cu", ".cuh", ".h", ".cpp")):
        for inc in _includes(path):
            assert "oracle" not in inc, (path, inc)


def test_oracle_never_includes_or_imports_the_package():
    for path in _files(ORC, (".c", ".h")):
        for inc in _includes(path):
            assert "mixture_experts_ffn_gemm_gb300" not in inc and "csrc" not in inc, (path, inc)
            assert inc not in ("moe.h", "common.cuh", "internal.h", "sched.cuh"), (path, inc)
    for path in _files(ORC, (".py",)):
        for mod in _imports(path):
            top = mod.split(".")[0]
            assert top != "mixture_experts_ffn_gemm_gb300" or mod.endswith("synthetic"), (path, mod)


def test_input_generator_reaches_neither_side():
    path = os.path.join(PKG, "synthetic.py")
    for mod in _imports(path):
        top = mod.lstrip(".").split(".")[0]
        assert top not in ("oracle", "binding", "build"), mod
        assert not mod.startswith(".binding") and not mod.startswith(".build"), mod
