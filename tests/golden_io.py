"""Reader for the small text fixtures under tests/golden/.

Each non-comment line is ``name = expression``; an expression is a number, a
list of numbers or arithmetic over ``exp`` and literals, exactly as the cited
page writes it.
"""
import math
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    env = {"__builtins__": {}, "exp": math.exp}
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, expr = (s.strip() for s in line.split("=", 1))
            out[key] = eval(expr, env, {})  # fixtures are committed text, no input
    return out
