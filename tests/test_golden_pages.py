"""Pins against the values the pages print (tests/golden/pages_printed_values.txt,
each line cited there): the 12-bit grid and its 36-bit codes, and the coordinate
orders of the multi-curve variant, for the oracle and for the library's host-side
curve table."""
import os

import numpy as np

from order_retrieval_gb300 import binding as zb

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_printed_values.txt")


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, *vals = line.split()
            out[name] = vals
    return out


def _orders(vals):
    return [[int(a) for a in v.split(",")] for v in vals]


def test_twelve_bit_grid(oracle_mod):
    g = _golden()
    bits = int(g["bits_per_coordinate"][0])
    assert 2 ** bits == int(g["grid_size"][0])
    lo, hi = (int(v) for v in g["cell_range"])
    xs = np.linspace(-1, 1, 20001, endpoint=False, dtype=np.float32)
    cells = {oracle_mod.quantise(float(x), bits) for x in xs}
    assert min(cells) == lo and max(cells) == hi and len(cells) == hi - lo + 1


def test_thirty_six_bit_codes(oracle_mod):
    g = _golden()
    bits = int(g["bits_per_coordinate"][0])
    width = int(g["code_bits_d3"][0])
    top = np.full((1, 3), np.nextafter(np.float32(1), np.float32(0)), np.float32)
    code = int(oracle_mod.encode(top, bits)[0])
    assert code == 2 ** width - 1                      # every bit of the 36 set
    assert int(oracle_mod.encode(-np.ones((1, 3), np.float32), bits)[0]) == 0
    p = zb.problem(1, 1, 64, 3, 64, 8, 64, bits, "bf16")
    assert zb.code_dtype(p).itemsize == 8               # 36 bits need the 64-bit word


def test_curve_orders_in_printed_order(oracle_mod):
    g = _golden()
    for curves in (3, 6):
        want = _orders(g["curves%d" % curves])
        assert oracle_mod.curve_axes(3, curves) == want
        assert [list(a) for a in zb.curve_axes(3, curves)] == want

