"""The bench's roofline arithmetic against its definition, by brute force.

The algorithmic bytes of one lora_apply call are the compulsory ones: every
distinct adapter slot named by an active row read once (its A and B' at the
slot rank), the x rows of the active rows read, their y slices read and
written, and the ids.  Here every byte address a call must touch is listed
one by one on small batches and counted, independently of the closed form
in bench.algorithmic_bytes.  Rows with id -1 touch nothing but their id.
"""
import numpy as np
import pytest

import bench
from lora_serving_gb300 import synth


def _brute_force_bytes(wl, group):
    touched = set()   # (buffer, byte offset); y counted once for the read, once for the write
    act = np.flatnonzero(wl.ids >= 0)
    for k in np.unique(wl.ids[act]):
        for p, (_, w) in enumerate(group.projs):
            for b in range(wl.r_slot * group.h_in * 2):
                touched.add(("A", p, int(k), b))
            for b in range(w * wl.r_slot * 2):
                touched.add(("B", p, int(k), b))
    for t in act:
        for b in range(group.h_in * 2):
            touched.add(("x", int(t), b))
        for off, (_, w) in zip(group.offsets, group.projs):
            for b in range(off * 2, (off + w) * 2):
                touched.add(("y_read", int(t), b))
                touched.add(("y_write", int(t), b))
    for t in range(wl.n_rows):
        for b in range(4):
            touched.add(("ids", t, b))
    return len(touched)


@pytest.mark.parametrize("ids", [
    [0, 1, -1, 0, 2, 2, -1, 1],      # three adapters, two base rows
    [-1, -1, -1],                    # base rows only: the ids alone
    [3, 3, 3, 3],                    # one adapter shared by every row
])
def test_algorithmic_bytes_equal_brute_force(ids):
    ids = np.array(ids, np.int32)
    n_slots = 4
    wl = synth.Workload("acct", 0, [synth.Group("g", 16, [("q", 16), ("k", 8), ("v", 8)])],
                        np.full(n_slots, 8), np.full(n_slots, 16.0), np.zeros(n_slots, bool), 8, ids, 0)
    g = wl.groups[0]
    assert bench.algorithmic_bytes(wl, g) == _brute_force_bytes(wl, g)


def test_merge_bytes_equal_brute_force():
    out, h_in, r = 24, 16, 8
    touched = set()
    for o in range(out):
        for k in range(h_in):
            for b in range(2):
                touched.add(("W_read", o, k, b))
                touched.add(("W_write", o, k, b))
    touched |= {("A", j, k, b) for j in range(r) for k in range(h_in) for b in range(2)}
    touched |= {("B", o, j, b) for o in range(out) for j in range(r) for b in range(2)}
    assert bench.merge_bytes(out, h_in, r) == len(touched)


def test_linear_flops_equal_counted_multiply_adds():
    """Base product for every row and output column, then the delta of each
    active row at its adapter's true rank: two flops per multiply-add."""
    ids = np.array([0, 1, -1, 1, 2], np.int32)
    ranks = np.array([8, 4, 16])
    wl = synth.Workload("acct", 0, [synth.Group("g", 16, [("q", 16), ("k", 8)])],
                        ranks, 2.0 * ranks, np.zeros(3, bool), 16, ids, 0)
    g = wl.groups[0]
    macs = 0
    for t in range(wl.n_rows):
        for _o in range(g.ld_y):
            for _k in range(g.h_in):
                macs += 1
        if ids[t] >= 0:
            r = int(ranks[ids[t]])
            for _, w in g.projs:
                macs += r * g.h_in      # shrink
                macs += w * r           # expand
    assert bench.linear_flops(wl, g) == 2 * macs
