"""The oracle and the CUDA path are independent, and the product has no CPU
fallback (checked on the CPU, without a GPU)."""

import ast
import glob
import os
import subprocess
import sys

from conftest import ROOT

PKG = "speculative_decoding_verify_bf16_gb300"


def _imports(path, top_level_only=False):
    tree = ast.parse(open(path).read(), filename=path)
    nodes = tree.body if top_level_only else list(ast.walk(tree))
    names = set()
    for node in nodes:
        if isinstance(node, ast.Import):
            names |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def test_oracle_imports_neither_the_library_nor_the_input_generators():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        assert not _imports(path) & {PKG, "workloads", "bench"}, path


def test_cpp_oracle_includes_only_the_standard_library():
    """oracle/verify_ref.cpp shares no header with the CUDA library."""
    import re
    src = open(os.path.join(ROOT, "oracle", "verify_ref.cpp")).read()
    includes = re.findall(r'^\s*#\s*include\s*([<"][^>"]+[>"])', src, flags=re.M)
    assert includes and all(i.startswith("<") for i in includes), includes
    assert "cuda" not in " ".join(includes).lower() and "spec_" not in src


def test_library_and_input_generators_never_import_the_oracle():
    paths = glob.glob(os.path.join(ROOT, PKG, "*.py")) + glob.glob(os.path.join(ROOT, "workloads", "*.py"))
    for path in paths:
        assert "oracle" not in _imports(path), path
    for path in glob.glob(os.path.join(ROOT, PKG, "csrc", "*")):
        assert "oracle" not in open(path).read().lower(), path


def test_bench_imports_the_oracle_only_in_its_cpu_legs():
    """bench.py may run the oracle for the CPU baseline and the reference arm:
    never at module level, never on the GPU path."""
    path = os.path.join(ROOT, "bench.py")
    assert "oracle" not in _imports(path, top_level_only=True)
    tree = ast.parse(open(path).read())
    users = {node.name for node in ast.walk(tree) if isinstance(node, ast.FunctionDef)
             and any(isinstance(n, (ast.Import, ast.ImportFrom)) and "oracle" in
                     ({a.name.split(".")[0] for a in n.names} if isinstance(n, ast.Import) else {(n.module or "").split(".")[0]})
                     for n in ast.walk(node))}
    assert users and all(("cpu" in u or "reference" in u) for u in users), users


def test_missing_library_raises_instead_of_falling_back(tmp_path):
    code = (f"import {PKG} as sv\n"
            f"sv.LIB_PATH = {str(tmp_path / 'absent.so')!r}\n"
            "try:\n"
            "    sv.spec_row_budget(3, 8, 1)\n"
            "except RuntimeError as e:\n"
            "    assert 'no CPU fallback' in str(e), e\n"
            "    print('raised')\n")
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert res.returncode == 0 and res.stdout.strip() == "raised", res.stdout + res.stderr
