"""Readers for the hand-written fixtures in tests/golden."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def bitrev():
    out = {}
    for line in _lines("bitrev.txt"):
        v = [int(x) for x in line.split()]
        out[v[0]] = np.array(v[1:])
    return out


def hadamard():
    out = {}
    it = iter(_lines("hadamard_sylvester.txt"))
    for line in it:
        d = int(line)
        out[d] = np.array([[float(x) for x in next(it).split()] for _ in range(d)])
    return out


def percentiles():
    out = []
    for line in _lines("percentile_type7.txt"):
        p, e, vals = line.split("|")
        out.append((float(p), float(e), np.array([float(x) for x in vals.split()])))
    return out


def quant_groups():
    out = []
    for line in _lines("quant_groups.txt"):
        c, s, z, vals, codes = line.split("|")
        out.append((float(c), float(s), float(z), np.array([float(x) for x in vals.split()]),
                    np.array([int(x) for x in codes.split()])))
    return out
