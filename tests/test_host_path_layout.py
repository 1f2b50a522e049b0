"""The host-buffer path's head-group schedule, checked on the CPU.

vsa_forward_host runs every head group as three operations on three streams:
the copy-in of its q/k/v/gate slices, its forward, and the copy-out of its
output. Two groups' device buffers alternate. These tests take the layout the
library reports (vsa_plan_host_path_group, host only) and the ordering the
header states, build the happens-before graph of all operations, and check
that no two operations that may run at the same time touch overlapping bytes
where one of them writes. They cover every head count from 1 to 128 with and
without a gate, and plant two mistakes the check must catch: each group laid
out at its own width (a group's inputs then overlap the output of the group
two before it while that output is still being copied out), and a dropped
wait.
"""
import itertools

import pytest

import block_sparse_video_gb300 as bsv

ALIGN = 256


def _align(x):
    return (x + ALIGN - 1) // ALIGN * ALIGN


def _edges(n_groups, drop_fwd_wait=False):
    """Happens-before edges between ('in'|'fwd'|'out', group) operations."""
    e = set()
    for g in range(n_groups):
        e.add((("in", g), ("fwd", g)))
        e.add((("fwd", g), ("out", g)))
        if g >= 1:
            for kind in ("in", "fwd", "out"):  # each stream runs in order
                e.add(((kind, g - 1), (kind, g)))
        if g >= 2:
            if not drop_fwd_wait:
                e.add((("fwd", g - 2), ("in", g)))
            e.add((("out", g - 2), ("fwd", g)))
    return e


def _reach(nodes, edges):
    succ = {n: set() for n in nodes}
    for a, b in edges:
        succ[a].add(b)
    reach = {}
    for n in nodes:
        seen, stack = set(), [n]
        while stack:
            for m in succ[stack.pop()]:
                if m not in seen:
                    seen.add(m)
                    stack.append(m)
        reach[n] = seen
    return reach


def _footprints(layout, with_gate):
    """Per operation: (reads, writes) as lists of [lo, hi) byte ranges."""
    fp = {}
    n_in = 4 if with_gate else 3
    for g, L in enumerate(layout):
        tb = L["tensor_bytes"]
        ins = [(L["offsets"][i], L["offsets"][i] + tb) for i in range(n_in)]
        out = (L["offsets"][4], L["offsets"][4] + tb)
        ws = (L["workspace_offset"], L["workspace_offset"] + L["workspace_bytes"])
        fp[("in", g)] = ([], ins)
        fp[("fwd", g)] = (ins + [ws], [out, ws])
        fp[("out", g)] = ([out], [])
    return fp


def _overlap(a, b):
    return a[0] < b[1] and b[0] < a[1]


def schedule_conflicts(layout, with_gate=True, drop_fwd_wait=False):
    """Pairs of operations that may run concurrently and touch the same bytes
    with at least one write."""
    n = len(layout)
    nodes = [(k, g) for g in range(n) for k in ("in", "fwd", "out")]
    reach = _reach(nodes, _edges(n, drop_fwd_wait))
    fp = _footprints(layout, with_gate)
    bad = []
    for a, b in itertools.combinations(nodes, 2):
        if b in reach[a] or a in reach[b]:
            continue
        ra, wa = fp[a]
        rb, wb = fp[b]
        if any(_overlap(x, y) for x in wa for y in rb + wb) or any(_overlap(x, y) for x in wb for y in ra):
            bad.append((a, b))
    return bad


def library_layout(plan):
    first = bsv.vsa_plan_host_path_group(plan, 0)
    return [first] + [bsv.vsa_plan_host_path_group(plan, g) for g in range(1, first["n_groups"])]


SHAPE = (1, 100, 60, 700)  # batch, text, audio, video: small, ragged, so tensor sizes are not powers of two


@pytest.mark.parametrize("heads", range(1, 129))
@pytest.mark.parametrize("subblock", [False, True])
def test_host_path_schedule_has_no_conflicts(heads, subblock):
    b, lt, la, lv = SHAPE
    plan = (bsv.vsa_plan_create_subblock(b, heads, lt, la, lv, 0.5) if subblock
            else bsv.vsa_plan_create(b, heads, lt, la, lv, 0.2))
    try:
        layout = library_layout(plan)
        total = bsv.vsa_plan_host_path_bytes(plan)
        # the groups cover every head once, in order
        h0 = 0
        for L in layout:
            assert L["first_head"] == h0 and L["heads"] >= 1
            assert L["tensor_bytes"] == b * (lt + la + lv) * L["heads"] * 128 * 2
            h0 += L["heads"]
        assert h0 == heads
        # every region is 256-byte aligned and inside the buffer
        for L in layout:
            for o in L["offsets"]:
                assert o % ALIGN == 0 and o + L["tensor_bytes"] <= total
            assert L["workspace_offset"] % ALIGN == 0
            assert L["workspace_offset"] + L["workspace_bytes"] <= total
        assert schedule_conflicts(layout, with_gate=not subblock) == []
    finally:
        bsv.vsa_plan_destroy(plan)


def _own_width_layout(layout):
    """The planted mistake: each group's tensors at its own width's stride."""
    widest = max(L["tensor_bytes"] for L in layout)
    slot = 5 * _align(widest)
    out = []
    for g, L in enumerate(layout):
        t = _align(L["tensor_bytes"])
        out.append(dict(L, offsets=[(g & 1) * slot + i * t for i in range(5)]))
    return out


@pytest.mark.parametrize("heads", [24, 56])
def test_checker_catches_own_width_layout(heads):
    """Groups 4, 6, 8, ...: group 2 (8 heads) laid out at its own stride writes
    its gate over group 0's output while the copy-out may still read it."""
    b, lt, la, lv = SHAPE
    plan = bsv.vsa_plan_create(b, heads, lt, la, lv, 0.2)
    try:
        layout = library_layout(plan)
        bad = schedule_conflicts(_own_width_layout(layout))
        assert (("out", 0), ("in", 2)) in bad
    finally:
        bsv.vsa_plan_destroy(plan)


def test_checker_catches_a_dropped_wait():
    b, lt, la, lv = SHAPE
    plan = bsv.vsa_plan_create(b, 24, lt, la, lv, 0.2)
    try:
        bad = schedule_conflicts(library_layout(plan), drop_fwd_wait=True)
        assert (("fwd", 0), ("in", 2)) in bad
    finally:
        bsv.vsa_plan_destroy(plan)


def test_host_path_group_rejects_bad_arguments():
    plan = bsv.vsa_plan_create(1, 24, 100, 60, 700, 0.2)
    try:
        n = bsv.vsa_plan_host_path_group(plan, 0)["n_groups"]
        for bad in (-1, n):
            with pytest.raises(bsv.VsaError):
                bsv.vsa_plan_host_path_group(plan, bad)
    finally:
        bsv.vsa_plan_destroy(plan)
