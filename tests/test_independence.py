"""The oracle and the CUDA path share no code. Read from the sources (AST
and include lines): the product package never imports the oracle and the
oracle never imports the product; the seeded input generator in
`workloads`, the one module both sides use, imports neither; outside
`tests/`, only the CPU-baseline and reference-arm functions of bench.py and
`smoke()` import the oracle, inside their own bodies; no CUDA or C source
includes anything from `oracle/`. And the library reads no environment
variable, so what runs follows the config alone; `profiles/` holds short
text summaries whose ncu commands leave the clocks alone."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "mixture_experts_routed_gb300"


def _py_files(sub):
    base = os.path.join(ROOT, sub)
    for dirpath, _, files in os.walk(base):
        for fn in files:
            if fn.endswith(".py"):
                yield os.path.join(dirpath, fn)


def _imports(path):
    """(top-level package name, enclosing function name or None) per import."""
    tree = ast.parse(open(path).read())
    out = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(child, ast.Import):
                out.extend((a.name.split(".")[0], func) for a in child.names)
            elif isinstance(child, ast.ImportFrom) and child.level == 0 and child.module:
                out.append((child.module.split(".")[0], func))
            visit(child, f)

    visit(tree, None)
    return out


def test_product_never_imports_the_oracle():
    for path in _py_files(PKG):
        assert "oracle" not in [m for m, _ in _imports(path)], path


def test_oracle_never_imports_the_product():
    for path in _py_files("oracle"):
        mods = [m for m, _ in _imports(path)]
        assert PKG not in mods and "bench" not in mods, path


def test_input_generator_imports_neither_side():
    for path in _py_files("workloads"):
        mods = [m for m, _ in _imports(path)]
        assert "oracle" not in mods and PKG not in mods, path


def test_oracle_imported_only_by_the_baseline_arms_and_smoke():
    allowed = {"bench.py": {"cpu_oracle_run", "host_inputs"},
               "__graft_entry__.py": {"smoke"}}
    for name, funcs in allowed.items():
        for mod, func in _imports(os.path.join(ROOT, name)):
            if mod == "oracle":
                assert func in funcs, (name, func)


def test_no_native_source_includes_the_oracle():
    for sub in (os.path.join(PKG, "csrc"), "include"):
        for fn in os.listdir(os.path.join(ROOT, sub)):
            if fn.endswith((".cu", ".cuh", ".h", ".c", ".cpp")):
                text = open(os.path.join(ROOT, sub, fn)).read()
                for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', text):
                    assert "oracle" not in inc, (fn, inc)


def test_library_reads_no_environment_variable():
    # the kernel shapes the product runs follow the config alone: no source
    # of the library or its binding reads the environment (the build script
    # may look for nvcc there)
    for sub in (os.path.join(PKG, "csrc"), "include"):
        for fn in os.listdir(os.path.join(ROOT, sub)):
            text = open(os.path.join(ROOT, sub, fn)).read()
            assert "getenv" not in text and "environ" not in text, fn
    for path in _py_files(PKG):
        if os.path.basename(path) != "build.py":
            assert "environ" not in open(path).read(), path


def test_profiles_are_short_text_summaries():
    # ncu summaries only: text, a few KB each, every capture command with
    # --clock-control none and running committed files (bench.py)
    for fn in os.listdir(os.path.join(ROOT, "profiles")):
        path = os.path.join(ROOT, "profiles", fn)
        assert fn.endswith((".md", ".txt", ".json")), fn
        assert os.path.getsize(path) < 16 * 1024, fn
        if fn.endswith(".md") and fn != "INDEX.md":
            text = open(path).read()
            assert "ncu " in text and "--clock-control none" in text, fn
            assert "bench.py" in text, fn
