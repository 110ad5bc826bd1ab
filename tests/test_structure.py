"""Structural checks (no GPU): the product path never reaches the oracle, the
oracle and the CUDA path share no code, and every committed profiler command
leaves the GPU clocks alone."""
import ast
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "quantized_kv_cache_tq_gb300")


def _imported_modules(path):
    tree = ast.parse(open(path).read(), filename=path)
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            mods.add(node.module.split(".")[0])
    return mods


def test_package_never_imports_the_oracle_or_the_generators():
    for path in glob.glob(os.path.join(PKG, "*.py")):
        mods = _imported_modules(path)
        assert "oracle" not in mods and "workloads" not in mods, path
    # nor does its native code name them
    for path in glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        assert not re.search(r"\boracle\b", text), path


def test_oracle_and_generators_are_independent_of_the_cuda_path():
    for path in (os.path.join(ROOT, "oracle", "__init__.py"), os.path.join(ROOT, "workloads", "__init__.py")):
        mods = _imported_modules(path)
        assert not mods & {"quantized_kv_cache_tq_gb300", "torch", "ctypes", "bench"}, (path, mods)
    # the generators hold no method arithmetic, so they import nothing of the oracle either
    assert "oracle" not in _imported_modules(os.path.join(ROOT, "workloads", "__init__.py"))


def test_bench_reaches_the_oracle_only_in_its_cpu_legs():
    # bench.py imports the oracle lazily, inside the functions that time it on the host
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    top = {a.name.split(".")[0] for n in tree.body if isinstance(n, ast.Import) for a in n.names}
    top |= {n.module.split(".")[0] for n in tree.body if isinstance(n, ast.ImportFrom) and n.module}
    assert "oracle" not in top


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))))
def test_profile_commands_keep_the_clocks(path):
    text = open(path).read()
    joined = re.sub(r"\\\n\s*", " ", text)              # one line per command
    ncu = [ln for ln in joined.splitlines() if re.match(r"\s*ncu\s", ln)]
    assert ncu, f"{path}: no ncu command"
    for ln in ncu:
        assert "--clock-control none" in ln, ln
    assert "python bench.py" in text                    # the profiled program is committed


def test_decode_profile_record_parses():
    text = open(os.path.join(ROOT, "profiles", "decode_mma_32k_turbo3_ncu.md")).read()
    assert re.search(r"traffic_bytes_per_launch:\s*\d+", text)
    assert re.search(r"decode_sources_sha256_16:\s*[0-9a-f]{16}", text)
