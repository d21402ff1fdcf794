"""Reader for the worked-example fixtures in tests/golden/ (plain text, cited)."""
from fractions import Fraction
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(tok):
    return Fraction(tok)


def load(fname="worked_examples.txt"):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, fname)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
                cases.append(cur)
            elif key == "cite":
                cur["cite"] = rest
            elif key in ("inc",):
                cur[key] = int(rest)
            else:
                cur[key] = [_num(t) for t in rest.split()]
    for c in cases:
        assert c.get("cite"), f"golden case {c['name']} has no citation"
    return cases
