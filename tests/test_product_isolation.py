"""The oracle is test infrastructure and the product never routes through it
(CPU, static checks).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline and
reference legs may import the oracle; the library package never does, and
the oracle imports nothing of the CUDA path (the two share no code)."""
import ast
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _oracle_imports(path):
    """(enclosing function or None, line) of every import of the oracle package."""
    tree = ast.parse(open(path).read(), filename=path)
    found = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(child, ast.Import):
                if any(a.name == "oracle" or a.name.startswith("oracle.") for a in child.names):
                    found.append((func, child.lineno))
            elif isinstance(child, ast.ImportFrom):
                mod = child.module or ""
                if child.level == 0 and (mod == "oracle" or mod.startswith("oracle.")):
                    found.append((func, child.lineno))
            visit(child, f)

    visit(tree, None)
    return found


def _py_files(folder):
    for dirpath, _, files in os.walk(os.path.join(ROOT, folder)):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(dirpath, f)


def test_library_package_never_imports_the_oracle():
    for path in _py_files("rms_backward_gb300"):
        assert _oracle_imports(path) == [], path
    for dirpath, _, files in os.walk(os.path.join(ROOT, "rms_backward_gb300", "csrc")):
        for f in files:
            assert "oracle" not in open(os.path.join(dirpath, f), errors="replace").read().lower(), f


def test_oracle_imports_nothing_of_the_cuda_path():
    for path in _py_files("oracle"):
        tree = ast.parse(open(path).read())
        for node in ast.walk(tree):
            names = []
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom) and node.level == 0:
                names = [node.module or ""]
            for n in names:
                assert not n.startswith(("rms_backward_gb300", "bench", "__graft_entry__")), (path, n)


def test_entry_points_import_the_oracle_only_where_allowed():
    allowed = {
        "__graft_entry__.py": {"smoke"},
        # _oracle_impl: the oracle the CPU-baseline leg (its _cpu_worker child)
        # and the reference arm time
        "bench.py": {"_oracle_impl", "run_forward"},
    }
    for name, funcs in allowed.items():
        found = _oracle_imports(os.path.join(ROOT, name))
        assert found, name                                   # the checks do use it
        for func, line in found:
            assert func in funcs, (name, func, line)         # never at module level
    # in the forward bench the import sits in the CPU-baseline branch only
    src = open(os.path.join(ROOT, "bench.py")).read().splitlines()
    for func, line in _oracle_imports(os.path.join(ROOT, "bench.py")):
        if func == "run_forward":
            above = "\n".join(src[max(0, line - 4):line - 1])
            assert "no_cpu_baseline" in above, line
    # the CPU worker runs only from the CPU-baseline leg: main() starts it for
    # --cpu-worker, which only _cpu_baseline_protocol passes
    text = "\n".join(src)
    assert text.count('"--cpu-worker"') == 2   # the option and the one call that sets it


def test_importing_the_library_loads_no_oracle():
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import rms_backward_gb300, rms_backward_gb300.abi, rms_backward_gb300.workloads\n"
            "import rms_backward_gb300.build\n"
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == "False"
