"""The oracle and the CUDA path are independent: the product package never
imports, reads or runs anything under oracle/, the oracle imports nothing of
the product, and the two share no source file. No GPU needed."""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "rank_cache_attention_flash_b300")
ORACLE = os.path.join(ROOT, "oracle")


def _py_files(d):
    for base, _, files in os.walk(d):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(base, f)


def _imported_modules(path):
    tree = ast.parse(open(path).read(), filename=path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def test_product_package_never_imports_the_oracle_or_the_tests():
    for f in _py_files(PKG):
        mods = _imported_modules(f)
        assert "oracle" not in mods and "tests" not in mods, f
        assert "oracle/" not in open(f).read(), f


def test_oracle_never_imports_the_product():
    for f in _py_files(ORACLE):
        mods = _imported_modules(f)
        assert "rank_cache_attention_flash_b300" not in mods and "bench" not in mods, f


def test_cuda_sources_name_no_oracle_file():
    csrc = os.path.join(PKG, "csrc")
    for f in os.listdir(csrc):
        src = open(os.path.join(csrc, f), errors="replace").read()
        assert "oracle/" not in src and "#include \"../../oracle" not in src, f


def test_no_source_file_is_shared():
    oracle_files = {os.path.basename(f) for f in _py_files(ORACLE)} - {"__init__.py"}
    product_files = {os.path.basename(f) for f in _py_files(PKG)} - {"__init__.py"}
    assert not oracle_files & product_files
