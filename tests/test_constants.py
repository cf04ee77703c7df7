"""The binding's constants equal the C header's: every `#define HS_<NAME> value`
in include/hs.h that the binding also names must have the same value there."""
import ast
import operator
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hs.h")


_OPS = {ast.Add: operator.add, ast.Sub: operator.sub, ast.Mult: operator.mul,
        ast.LShift: operator.lshift, ast.USub: operator.neg}


def _value(node, names):
    """An integer expression of the header: literals, earlier names, + - * << and negation."""
    if isinstance(node, ast.Expression):
        return _value(node.body, names)
    if isinstance(node, ast.Constant) and isinstance(node.value, int):
        return node.value
    if isinstance(node, ast.Name):
        return names[node.id]
    if isinstance(node, ast.UnaryOp) and type(node.op) in _OPS:
        return _OPS[type(node.op)](_value(node.operand, names))
    if isinstance(node, ast.BinOp) and type(node.op) in _OPS:
        return _OPS[type(node.op)](_value(node.left, names), _value(node.right, names))
    raise ValueError(ast.dump(node))


def header_defines():
    """NAME -> int for the header's integer defines (values may use earlier names)."""
    out = {}
    for line in open(HEADER):
        m = re.match(r"#define\s+(HS_\w+)\s+(.+?)\s*(/\*.*)?$", line)
        if not m or m.group(1) == "HS_H":
            continue
        expr = re.sub(r"\b(\d+)(?:ull|ul|ll|u|l)\b", r"\1", m.group(2), flags=re.I)  # C suffixes
        if not re.fullmatch(r"[\w\s()+*<>x-]+", expr):
            continue
        out[m.group(1)] = _value(ast.parse(expr, mode="eval"), out)
    return out


def test_header_constants_parse():
    d = header_defines()
    # the values every caller depends on
    assert d["HS_OK"] == 0 and d["HS_ERR_ARG"] < 0
    assert d["HS_FUSED_MAX_REQUEST_BYTES"] == 1 << 20
    assert d["HS_POOL_HUGE_MIN_BYTES"] == 16 << 30
    assert d["HS_NOALLOC_SCRATCH_BYTES"] == 8 * d["HS_NOALLOC_MAX_ENTRIES"] + 4 * d["HS_MAX_BATCH"]


def test_binding_constants_match_header():
    from hierarchical_kv_cache_hs_gb300 import hs
    d = header_defines()
    named = [k for k in d if hasattr(hs, k)]
    assert len(named) >= 25, named
    for k in named:
        assert getattr(hs, k) == d[k], k
