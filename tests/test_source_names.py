"""Every name that the host-side Python reads or deletes is bound somewhere it
can be seen from: a static scan of the benchmark, the entry points, the
binding and the workload generators (no GPU, nothing executed). A benchmark
leg that only runs on a GPU machine can otherwise carry an undefined name that no
CPU test reaches."""
import ast
import builtins
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ["bench.py", "__graft_entry__.py", "indexer_top_sparse_03_b300/binding.py",
         "indexer_top_sparse_03_b300/__init__.py", "indexer_top_sparse_03_b300/build.py",
         "workloads/__init__.py", "oracle/__init__.py"]
SCOPES = (ast.FunctionDef, ast.AsyncFunctionDef, ast.Lambda, ast.ClassDef, ast.ListComp, ast.SetComp,
          ast.DictComp, ast.GeneratorExp)


def _children(node):
    """Child nodes that belong to the same scope as `node`."""
    for c in ast.iter_child_nodes(node):
        yield c


def _bound(stmts):
    """Names bound in one scope by these statements (nested scopes contribute
    only the name of a def or class)."""
    out = set()
    stack = list(stmts)
    while stack:
        n = stack.pop()
        if isinstance(n, (ast.FunctionDef, ast.AsyncFunctionDef, ast.ClassDef)):
            out.add(n.name)
            stack.extend(n.decorator_list)
            continue
        if isinstance(n, SCOPES):
            continue
        if isinstance(n, ast.Name) and isinstance(n.ctx, ast.Store):
            out.add(n.id)
        elif isinstance(n, (ast.Import, ast.ImportFrom)):
            for a in n.names:
                out.add(a.asname or a.name.split(".")[0])
        elif isinstance(n, ast.ExceptHandler) and n.name:
            out.add(n.name)
        elif isinstance(n, (ast.Global, ast.Nonlocal)):
            out.update(n.names)
        stack.extend(_children(n))
    return out


def _args(a: ast.arguments):
    names = [x.arg for x in a.posonlyargs + a.args + a.kwonlyargs]
    names += [x.arg for x in (a.vararg, a.kwarg) if x is not None]
    return set(names)


def _check(node, visible, bad, fn):
    """Report every Name read or deleted under `node` that is not in `visible`
    (extended at each nested scope)."""
    for c in _children(node):
        if isinstance(c, (ast.FunctionDef, ast.AsyncFunctionDef)):
            for d in c.decorator_list + c.args.defaults + [x for x in c.args.kw_defaults if x is not None]:
                _check_expr(d, visible, bad, fn)
            inner = visible | _args(c.args) | _bound(c.body)
            for s in c.body:
                _check_stmt(s, inner, bad, fn)
        elif isinstance(c, ast.ClassDef):
            for d in c.decorator_list + c.bases:
                _check_expr(d, visible, bad, fn)
            cls = visible | _bound(c.body)
            for s in c.body:
                if isinstance(s, (ast.FunctionDef, ast.AsyncFunctionDef)):
                    _check(ast.Module(body=[s], type_ignores=[]), visible, bad, fn)
                else:
                    _check_stmt(s, cls, bad, fn)
        elif isinstance(c, ast.Lambda):
            inner = visible | _args(c.args)
            _check_expr(c.body, inner, bad, fn)
        elif isinstance(c, (ast.ListComp, ast.SetComp, ast.DictComp, ast.GeneratorExp)):
            inner = set(visible)
            for g in c.generators:
                _check_expr(g.iter, inner, bad, fn)
                inner |= {n.id for n in ast.walk(g.target) if isinstance(n, ast.Name)}
                for cond in g.ifs:
                    _check_expr(cond, inner, bad, fn)
            for part in ((c.key, c.value) if isinstance(c, ast.DictComp) else (c.elt,)):
                _check_expr(part, inner, bad, fn)
        else:
            if isinstance(c, ast.Name) and isinstance(c.ctx, (ast.Load, ast.Del)) and c.id not in visible:
                bad.append(f"{fn}:{c.lineno}: '{c.id}' is {'deleted' if isinstance(c.ctx, ast.Del) else 'read'}"
                           " but never bound in a visible scope")
            _check(c, visible, bad, fn)


def _check_stmt(s, visible, bad, fn):
    _check(ast.Module(body=[s], type_ignores=[]), visible, bad, fn)


def _check_expr(e, visible, bad, fn):
    _check(ast.Expression(body=e), visible, bad, fn)


def undefined_names(src: str, fn: str):
    tree = ast.parse(src, fn)
    visible = set(dir(builtins)) | {"__file__", "__name__", "__doc__", "__spec__"} | _bound(tree.body)
    bad = []
    _check(tree, visible, bad, fn)
    return bad


@pytest.mark.parametrize("rel", FILES)
def test_no_undefined_names(rel):
    path = os.path.join(ROOT, rel)
    assert undefined_names(open(path).read(), rel) == []


def test_checker_catches_a_delete_of_a_name_never_bound():
    src = ("def run():\n"
           "    inp = 1\n"
           "    del host, inp\n")
    bad = undefined_names(src, "x.py")
    assert len(bad) == 1 and "'host' is deleted" in bad[0]


def test_checker_sees_enclosing_scopes_and_comprehensions():
    src = ("import os\n"
           "def f(a, *b, c=os.sep, **d):\n"
           "    e = [x + a for x in b if x]\n"
           "    def g():\n"
           "        return e, c, d, lambda y: y + a\n"
           "    class K:\n"
           "        z = 1\n"
           "        def m(self):\n"
           "            return z\n"
           "    return g, K\n")
    bad = undefined_names(src, "x.py")
    assert len(bad) == 1 and "'z'" in bad[0]                 # class names are not seen by methods
