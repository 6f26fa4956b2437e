"""The oracle and the CUDA path share no code: the oracle's C source includes
only standard headers, nothing of the library names the oracle, and the
scripts load the oracle only where they check against it or time it."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _read(*parts):
    with open(os.path.join(ROOT, *parts)) as f:
        return f.read()


def test_oracle_includes_only_standard_headers():
    src = _read("oracle", "dsv4_oracle.c")
    includes = re.findall(r'^\s*#\s*include\s*([<"][^>"]+[>"])', src, flags=re.M)
    assert includes, "no includes found"
    assert all(i.startswith("<") for i in includes), includes


def test_library_never_names_the_oracle():
    pkg = os.path.join(ROOT, "deepseek_v4_attention_gb300")
    files = [os.path.join(ROOT, "include", "dsv4.h"), os.path.join(ROOT, "dsv4_inputs.py")]
    for d, _, names in os.walk(pkg):
        if "__pycache__" in d:
            continue
        files += [os.path.join(d, n) for n in names if n.endswith((".py", ".cu", ".cuh", ".h"))]
    for path in files:
        with open(path) as f:
            text = f.read()
        code = re.sub(r'"""[\s\S]*?"""', "", text) if path.endswith(".py") else text
        assert not re.search(r"^\s*(import|from)\s+oracle\b", code, flags=re.M), path
        assert not re.search(r'#\s*include\s*["<][^">]*oracle', code), path


def _functions_importing_oracle(path):
    tree = ast.parse(_read(path))
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, (ast.FunctionDef, ast.AsyncFunctionDef)):
            for sub in ast.walk(node):
                if isinstance(sub, ast.Import) and any(a.name == "oracle" for a in sub.names):
                    out.add(node.name)
                if isinstance(sub, ast.ImportFrom) and sub.module == "oracle":
                    out.add(node.name)
    top = {a.name for n in tree.body if isinstance(n, ast.Import) for a in n.names}
    top |= {n.module for n in tree.body if isinstance(n, ast.ImportFrom)}
    return out, "oracle" in top


def test_scripts_load_the_oracle_only_to_check_or_time():
    funcs, at_top = _functions_importing_oracle("bench.py")
    assert not at_top and funcs == {"cpu_baseline", "run_reference"}, funcs
    funcs, at_top = _functions_importing_oracle("__graft_entry__.py")
    assert not at_top and funcs == {"build", "smoke"}, funcs
