"""Reader for the hand-derived fixtures in tests/golden/ (closed forms as
Python expressions over exp/log/sqrt/inf)."""
import math
import os
from fractions import Fraction  # noqa: F401  (allowed in expressions)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_ENV = {"exp": math.exp, "log": math.log, "sqrt": math.sqrt, "inf": math.inf, "__builtins__": {}}


def _val(tok: str):
    if tok == "none":
        return None
    return float(eval(tok, _ENV))  # fixture files are committed test data


def load(name: str):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key == "case":
                cur = {"name": rest[0]}
                cases.append(cur)
                continue
            vals = [_val(t) for t in rest]
            cur[key] = vals[0] if key in ("T", "dqk", "dv") else vals
    for c in cases:
        for key in ("T", "dqk", "dv"):
            if key in c:
                c[key] = int(c[key])
    return cases
