"""Readers for the text fixtures under tests/golden/ (each file cites the page
and section its values come from)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def keyvals(name):
    """`key = value` lines -> dict of strings."""
    out = {}
    for line in _lines(name):
        k, v = line.split("=", 1)
        out[k.strip()] = v.strip()
    return out


def rows(name, sep=None):
    """Non-comment lines split on `sep` (whitespace by default)."""
    return [[c.strip() for c in line.split(sep)] for line in _lines(name)]


def floats(s):
    return [float(t) for t in s.split()]


def ints(s):
    return [int(t) for t in s.split()]


def hexbytes(s):
    return bytes.fromhex(s.replace(" ", ""))
