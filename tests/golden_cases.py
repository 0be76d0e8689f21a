"""Loader for the hand-derived worked examples in tests/golden/*.txt."""
import ast
import math
import os
import operator

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

_OPS = {ast.Add: operator.add, ast.Sub: operator.sub, ast.Mult: operator.mul,
        ast.Div: operator.truediv, ast.USub: operator.neg, ast.UAdd: operator.pos}
_FUNCS = {"log": math.log, "sqrt": math.sqrt}


def _eval(node):
    if isinstance(node, ast.Expression):
        return _eval(node.body)
    if isinstance(node, ast.Constant) and isinstance(node.value, (int, float)):
        return float(node.value)
    if isinstance(node, ast.BinOp) and type(node.op) in _OPS:
        return _OPS[type(node.op)](_eval(node.left), _eval(node.right))
    if isinstance(node, ast.UnaryOp) and type(node.op) in _OPS:
        return _OPS[type(node.op)](_eval(node.operand))
    if (isinstance(node, ast.Call) and isinstance(node.func, ast.Name)
            and node.func.id in _FUNCS and len(node.args) == 1):
        return _FUNCS[node.func.id](_eval(node.args[0]))
    raise ValueError(f"unsupported expression: {ast.dump(node)}")


def expr(text: str) -> float:
    return _eval(ast.parse(text.strip(), mode="eval"))


def _row(line):
    return [expr(t) for t in line.split()]


def load(path):
    header, blocks, cur = {}, {}, None
    with open(path) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                header[k.strip()] = v.strip()
                continue
            if line in ("Q", "K", "V", "O", "LSE"):
                cur = line
                blocks[cur] = []
                continue
            blocks[cur].append(_row(line))
    case = {
        "name": os.path.basename(path),
        "Nq": int(header["Nq"]), "Nk": int(header["Nk"]), "d": int(header["d"]),
        "scale": expr(header["scale"]), "tol": expr(header["tol"]),
    }
    for k, rows in blocks.items():
        case[k] = np.array(rows, dtype=np.float64)
    case["LSE"] = case["LSE"].reshape(-1)
    assert case["Q"].shape == (case["Nq"], case["d"]), path
    assert case["K"].shape == (case["Nk"], case["d"]) == case["V"].shape, path
    assert case["O"].shape == (case["Nq"], case["d"]), path
    assert case["LSE"].shape == (case["Nq"],), path
    return case


def all_cases():
    return [load(os.path.join(GOLDEN_DIR, f)) for f in sorted(os.listdir(GOLDEN_DIR)) if f.endswith(".txt")]
