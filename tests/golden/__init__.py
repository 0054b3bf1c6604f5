"""Readers for the small text fixtures in this folder."""
import os

_HERE = os.path.dirname(os.path.abspath(__file__))


def pins() -> dict:
    """key -> list of numbers (or list of rows for '/'-separated values)."""
    out = {}
    with open(os.path.join(_HERE, "pins.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            if "/" in val:
                out[key] = [[float(x) for x in row.split()] for row in val.split("/")]
            else:
                out[key] = [int(x, 16) if x.startswith("0x") else float(x) for x in val.split()]
    return out


def edge_counts() -> dict:
    """workload name -> dict(window_edges, window_plus_globals, total) (None where '-')."""
    out = {}
    with open(os.path.join(_HERE, "edge_counts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            p = line.split()
            conv = [None if x == "-" else int(x) for x in p[1:]]
            out[p[0]] = dict(n=conv[0], r=conv[1], g=conv[2], R=conv[3], window_edges=conv[4],
                             window_plus_globals=conv[5], total=conv[6])
    return out
