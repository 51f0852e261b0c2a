"""Readers for the cited fixtures under tests/golden/ (test-side, independent of the oracle)."""
import math
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def e2m1_table():
    """code -> value, from the OCP MX FP4 (E2M1) table."""
    t = {int(c): float(v) for c, v in _rows("e2m1_ocp_mx.txt")}
    assert sorted(t) == list(range(16))
    return t


def e4m3_specials():
    """byte -> value for the cited special encodings (NaN as float('nan'))."""
    return {int(b, 16): (math.nan if v == "nan" else float(v)) for b, v in _rows("e4m3_special.txt")}
