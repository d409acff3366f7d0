"""Readers for the small text fixtures under tests/golden/ (page facts only)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def kv(name):
    """`key = value` lines of a fixture, comments stripped, values as float."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = float(v)
    return out


def shapes(name="edge_shapes.txt"):
    """List of (M, N) pairs."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                m, n = line.split()
                out.append((int(m), int(n)))
    return out
