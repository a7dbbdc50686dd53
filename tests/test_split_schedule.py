"""The split plan's schedule, modelled on the host from its shape query (no GPU).

For each shape the host logic cuts the rows into `lanes` groups of `parts`
blocks (softmax_rows_split_shape); the kernel's schedule is that group g takes
rows g, g + lanes, ... in turn, pass 1 of step t and pass 2 of step t - 2 in one
sweep, and the tagged pairs live in a ring of four slots. This model walks that
schedule and checks what the kernel relies on: every unit of every row is read
and written by exactly one block, every row a block touches exists, every
workspace slot lies inside the fixed workspace, and a slot is overwritten only
after every block of its group has merged the pairs it held.
"""
import pytest

import memory_bound_row_rows_gb300 as sr
from memory_bound_row_rows_gb300 import _build

ALIGNED_IN, ALIGNED_OUT = 0x7F0000000000, 0x7F0100000000
LAG, RING, MAX_BLOCKS_WS = 2, 4, 4096
L2 = 132644864


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sr.load()


def schedule(M, N, dtype, aligned, max_blocks):
    out = ALIGNED_OUT if aligned else ALIGNED_OUT + 2
    sh = sr.softmax_rows_split_shape(ALIGNED_IN, out, M, N, N, N, dtype, max_blocks, L2)
    lanes, parts, pu = sh["lanes"], sh["parts"], sh["part_units"]
    units = N // sh["unit_elems"]
    B = lanes * parts
    assert 1 <= B <= min(max_blocks, MAX_BLOCKS_WS)
    written = {}
    events = []  # (block, kind, step) in each block's program order
    for b in range(B):
        g, p = divmod(b, parts)
        u0, u1 = min(p * pu, units), min(p * pu + pu, units)
        assert u0 < u1, "an empty part"
        steps = (M - g + lanes - 1) // lanes
        for t in range(steps + LAG):
            stats, apply = t < steps, t >= LAG
            if apply:
                q = t - LAG
                r = g + q * lanes
                assert 0 <= r < M
                events.append((b, "merge", q))
                key = (r, u0)
                assert key not in written, "a part written twice"
                written[key] = u1
            if stats:
                r = g + t * lanes
                assert 0 <= r < M
                slot = (t % RING) * B + b
                assert 0 <= slot < RING * MAX_BLOCKS_WS
                events.append((b, "publish", t))
    # Every row covered exactly once, part by part.
    for r in range(M):
        spans = sorted((u0, u1) for (rr, u0), u1 in written.items() if rr == r)
        assert spans[0][0] == 0 and spans[-1][1] == units
        assert all(a[1] == c[0] for a, c in zip(spans, spans[1:]))
    return sh, B, lanes, parts, events


@pytest.mark.parametrize("M,N,dtype,aligned", [
    (32, 1 << 22, 0, True), (128, 1 << 19, 1, True), (512, 400008, 1, True),
    (64, 131072, 2, True), (4, 32769, 2, False), (130, 1 << 19, 2, True),
    (23, 1 << 20, 0, True), (9, 1 << 22, 0, True), (3, 1000, 0, True), (1, 1 << 20, 0, True),
])
@pytest.mark.parametrize("max_blocks", [304, 456, 608])
def test_schedule_covers_every_row_once(lib, M, N, dtype, aligned, max_blocks):
    schedule(M, N, dtype, aligned, max_blocks)


@pytest.mark.parametrize("M,N,dtype", [(130, 1 << 19, 1), (32, 1 << 22, 0), (23, 1 << 20, 0)])
def test_ring_slot_reuse_is_safe(lib, M, N, dtype):
    """Block Y stores its pair of step s in slot s mod 4 only after it merged step
    s - 2, which needed every block X of its group to have stored step s - 2, which
    X did only after it merged step s - 4: so X is done with the slot's old pair."""
    sh, B, lanes, parts, events = schedule(M, N, dtype, True, 456)
    order = {}  # per block: position of each event in its program order
    for b, kind, step in events:
        order.setdefault(b, []).append((kind, step))
    for b, seq in order.items():
        pos = {e: i for i, e in enumerate(seq)}
        for kind, s in seq:
            if kind == "publish" and s >= RING:
                # This block merged step s - LAG before publishing step s ...
                assert pos[("merge", s - LAG)] < pos[("publish", s)]
                # ... and it published step s - LAG only after merging step s - 2 LAG.
                assert pos[("merge", s - 2 * LAG)] < pos[("publish", s - LAG)]
