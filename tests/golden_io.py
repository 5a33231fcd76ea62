"""Reader for the text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

UNITS = {"KB": 1e3, "MB": 1e6, "GB": 1e9}


def rows(name):
    out = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            out.append(line.split())
    return out


def quantity(s):
    """'57MB' -> (57.0, 1e6); '1.8GB' -> (1.8, 1e9)."""
    for u, f in UNITS.items():
        if s.endswith(u):
            return float(s[:-len(u)]), f
    return float(s), 1.0
