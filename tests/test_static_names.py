"""Every name the Python sources read is bound somewhere in their module.

A coarse, module-wide check (a name bound in any scope counts), cheap enough
to run on every change.  It catches a function or import removed while a
caller remains, on paths that only a GPU run would otherwise reach: the
benchmark's roofline helpers were once lost that way.
"""
import ast
import builtins
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = ["bench.py", "__graft_entry__.py", "oracle/oracle.py", "oracle/build.py"] + [
    os.path.join("sparse_attention_26_b300", f)
    for f in sorted(os.listdir(os.path.join(ROOT, "sparse_attention_26_b300")))
    if f.endswith(".py")]


def unbound_names(source, name="<source>"):
    tree = ast.parse(source, name)
    bound = set(dir(builtins)) | {"__file__", "__name__", "__doc__"}
    for node in ast.walk(tree):
        if isinstance(node, (ast.FunctionDef, ast.AsyncFunctionDef, ast.ClassDef)):
            bound.add(node.name)
        elif isinstance(node, (ast.Import, ast.ImportFrom)):
            for a in node.names:
                if a.name == "*":
                    return set()  # star imports: nothing to check
                bound.add((a.asname or a.name).split(".")[0])
        elif isinstance(node, ast.Name) and isinstance(node.ctx, (ast.Store, ast.Del)):
            bound.add(node.id)
        elif isinstance(node, ast.arg):
            bound.add(node.arg)
        elif isinstance(node, ast.ExceptHandler) and node.name:
            bound.add(node.name)
        elif isinstance(node, (ast.Global, ast.Nonlocal)):
            bound.update(node.names)
    used = {n.id for n in ast.walk(tree) if isinstance(n, ast.Name) and isinstance(n.ctx, ast.Load)}
    return used - bound


@pytest.mark.parametrize("rel", SOURCES)
def test_every_name_read_is_bound(rel):
    path = os.path.join(ROOT, rel)
    assert unbound_names(open(path).read(), path) == set()


def test_the_check_sees_a_removed_function():
    assert unbound_names("def run():\n    return helper(1)\n") == {"helper"}
    assert unbound_names("def helper(x):\n    return x\n\ndef run():\n    return helper(1)\n") \
        == set()
