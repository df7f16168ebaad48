"""Readers for the small text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def kv(name):
    """'key = value' fixture -> dict of strings."""
    out = {}
    for line in _lines(name):
        key, val = line.split("=", 1)
        out[key.strip()] = val.strip()
    return out


def table(name):
    """Whitespace-separated numeric table -> list of tuples of floats."""
    return [tuple(float(x) for x in line.split()) for line in _lines(name)]
