"""Readers for the text fixtures under tests/golden/ (each cites its page)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


def mask_picture(name="txl_mask_M3_L4.txt"):
    """Bool [L, M+L] visibility read from the page's picture."""
    rows = []
    for ln in _lines(name):
        cells = ln.replace("|", "")
        rows.append([c in "mx" for c in cells])
    return np.array(rows, dtype=bool)


def worked_example(name="worked_example_L4_M8.txt"):
    return {k: int(v) for k, v in (ln.split() for ln in _lines(name))}


def rel_ids(name="rel_ids_L4_M3.txt"):
    return np.array([[int(x) for x in ln.split()] for ln in _lines(name)])
