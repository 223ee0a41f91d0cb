"""The oracle stays independent of the CUDA path, and the product path never reaches the
oracle: checked statically on the sources.

- The library (package + C/CUDA sources) neither imports nor includes anything of oracle/.
- The oracle includes only the C standard library and its own header: nothing of the
  library, its headers or the input generator.
- The library's sources include nothing of synth/ or oracle/ (the generator serves the tests
  and the benchmark, not the product).
- bench.py imports the oracle only inside functions (its CPU-baseline and reference legs),
  never at module level; __graft_entry__ only inside smoke() and build() (which compiles the
  oracle's C: building the checker is not using it).
- The input generator holds none of the method's arithmetic (no moments, bias correction or
  square root of a second moment)."""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "zero_partitioned_mixed_adam_gb300")


def _includes(path):
    return re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', open(path).read(), flags=re.M)


def _imports(tree):
    out = set()
    for n in ast.walk(tree):
        if isinstance(n, ast.Import):
            out |= {a.name.split(".")[0] for a in n.names}
        elif isinstance(n, ast.ImportFrom) and n.module:
            out.add(n.module.split(".")[0])
    return out


def test_library_never_reaches_the_oracle():
    for f in glob.glob(os.path.join(PKG, "*.py")):
        assert "oracle" not in _imports(ast.parse(open(f).read())), f
    for f in glob.glob(os.path.join(PKG, "csrc", "*")):
        for inc in _includes(f):
            assert "oracle" not in inc and "synth" not in inc, (f, inc)


def test_oracle_includes_only_the_c_library_and_itself():
    allowed = {"math.h", "stddef.h", "stdint.h", "stdlib.h", "string.h", "stdio.h",
               "zero_oracle.h"}
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.[ch]")):
        for inc in _includes(f):
            assert inc in allowed, (f, inc)
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        mods = _imports(ast.parse(open(f).read()))
        assert not mods & {"zero_partitioned_mixed_adam_gb300", "synth", "torch"}, (f, mods)


def test_oracle_imported_only_inside_functions():
    for name, funcs in (("bench.py", None),
                        ("__graft_entry__.py", {"smoke", "_smoke_step", "build"})):
        tree = ast.parse(open(os.path.join(ROOT, name)).read())
        for node in tree.body:   # module level
            if isinstance(node, (ast.Import, ast.ImportFrom)):
                assert "oracle" not in _imports(ast.Module(body=[node], type_ignores=[])), name
        if funcs:
            for fn in [n for n in tree.body if isinstance(n, ast.FunctionDef)]:
                if "oracle" in _imports(fn):
                    assert fn.name in funcs, (name, fn.name)


def test_generator_holds_none_of_the_method():
    code = ""
    for f in glob.glob(os.path.join(ROOT, "synth", "*.[ch]")) + \
            glob.glob(os.path.join(ROOT, "synth", "*.cu")):
        text = re.sub(r"/\*.*?\*/", "", open(f).read(), flags=re.S)
        code += "\n".join(line.split("//")[0] for line in text.splitlines())
    for word in ("beta1", "beta2", "b1", "b2", "m_hat", "v_hat", "bc1", "bc2", "lr", "eps",
                 "adam", "master_update", "world"):
        assert not re.search(r"\b%s\b" % word, code), word
