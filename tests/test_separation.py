"""The oracle and the product stay apart (checked on the sources, no GPU): the library and its
binding never import or include anything of the oracle, the oracle never reaches into the
library, the shared input module holds neither, and the benchmark loads the oracle only in its
CPU-baseline and reference legs."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "gated_delta_rule_prefill_gb300")


def _files(top, exts):
    for d, _, fs in os.walk(top):
        if "__pycache__" in d or "_build" in d:
            continue
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def _imports(path, tree=None):
    tree = tree or ast.parse(open(path).read(), filename=path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for n in node.names:
                yield n.name.split(".")[0], node
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            yield node.module.split(".")[0], node


def test_product_never_touches_the_oracle():
    for p in _files(PKG, (".py",)):
        assert all(mod != "oracle" for mod, _ in _imports(p)), p
    for p in list(_files(PKG, (".cu", ".cuh", ".h"))) + list(_files(os.path.join(ROOT, "include"), (".h",))):
        src = open(p).read()
        assert not re.search(r'#\s*include\s*[<"][^>"]*oracle', src), p
    build = open(os.path.join(PKG, "build.py")).read()
    assert "oracle" not in build  # the library's build compiles nothing of the oracle


def test_oracle_never_touches_the_product():
    odir = os.path.join(ROOT, "oracle")
    for p in _files(odir, (".py",)):
        mods = {mod for mod, _ in _imports(p)}
        assert "gated_delta_rule_prefill_gb300" not in mods, p
    for p in _files(odir, (".c", ".h")):
        src = open(p).read()
        assert not re.search(r'#\s*include\s*"[^"]*(csrc|gdr\.h|tc_common|umma)', src), p


def test_shared_inputs_module_is_neutral():
    mods = {mod for mod, _ in _imports(os.path.join(ROOT, "gdr_inputs.py"))}
    assert "oracle" not in mods and "gated_delta_rule_prefill_gb300" not in mods


def test_bench_loads_the_oracle_only_for_the_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    src = open(path).read()
    tree = ast.parse(src)
    parents = {}
    for node in ast.walk(tree):
        for ch in ast.iter_child_nodes(node):
            parents[ch] = node
    found = 0
    for mod, node in _imports(path, tree):
        if mod != "oracle":
            continue
        found += 1
        chain, n = [], node
        while n in parents:
            n = parents[n]
            chain.append(n)
        funcs = [c.name for c in chain if isinstance(c, ast.FunctionDef)]
        assert funcs, "module-level oracle import"
        if funcs[0] == "run_gpu":  # only under the CPU-baseline switch
            ifs = [c for c in chain if isinstance(c, ast.If)]
            assert any("no_cpu_baseline" in ast.get_source_segment(src, c.test) for c in ifs)
        else:
            assert funcs[0] in ("run_reference", "time_oracle"), funcs
    assert found >= 2
