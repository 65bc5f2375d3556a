"""Small test utilities: golden fixtures and tree arrays written out by hand."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def pointers_from_parents(parents):
    """First-child / next-sibling arrays of one tree given by its parent list
    (children in ascending node order)."""
    n = len(parents)
    nt = [-1] * n
    ns = [-1] * n
    for c in range(n):
        p = parents[c]
        if p < 0:
            continue
        if nt[p] == -1:
            nt[p] = c
        else:
            s = nt[p]
            while ns[s] != -1:
                s = ns[s]
            ns[s] = c
    return np.array(nt, np.int32), np.array(ns, np.int32)


def onehot_logits(rows_argmax, V, low=-5.0, high=5.0):
    """fp32 logits whose row r has its unique maximum at rows_argmax[r]."""
    x = np.full((len(rows_argmax), V), low, np.float32)
    for r, a in enumerate(rows_argmax):
        x[r, a] = high
    return x
