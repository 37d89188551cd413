"""Pins of the prefetch-plan oracle (DWDP §2 double-buffered prefetch; §4.3.2
fixed-size slices issued round-robin), checked exhaustively on small maps:
every byte of every non-resident expert is copied exactly once to its stage
slot, no slice exceeds the chunk size, only a region's last slice is short,
and the issue order is round-robin over the peers."""
import itertools

import numpy as np
import pytest

from oracle import plan_prefetch, stage_slots


def _check(E, H, I, ls, pid, ps, P, chunk):
    plan = plan_prefetch(E, H, I, ls, pid, ps, P, chunk)
    b = {0: 2 * I * H * 2, 1: H * I * 2}
    slot = stage_slots(E, ls)
    # byte coverage, built independently per expert
    want = set()
    for e in range(E):
        if ls[e] >= 0:
            continue
        for t in (0, 1):
            for byte in range(b[t]):
                want.add((pid[e], t, ps[e] * b[t] + byte, slot[e] * b[t] + byte))
    got = []
    for (p, t, s, d, n) in plan:
        assert 0 < n <= chunk
        for i in range(n):
            got.append((p, t, s + i, d + i))
    assert len(got) == len(set(got)), "a byte is copied twice"
    assert set(got) == want, "coverage mismatch"
    # round-robin: the peer sequence is c-th slices of all peers in turn
    per = {p: [x for x in plan if x[0] == p] for p in range(P)}
    order = []
    for c in range(max([len(v) for v in per.values()] + [0])):
        for p in range(P):
            if c < len(per[p]):
                order.append(per[p][c])
    assert order == plan
    return plan


def test_exhaustive_small_maps():
    H, I = 4, 2          # w13 = 32 B, w2 = 16 B per expert
    E = 4
    for P in (1, 2, 3):
        for assign in itertools.product(range(-1, P), repeat=E):
            ls = [e if a < 0 else -1 for e, a in enumerate(assign)]
            pid = [a for a in assign]
            ps = [0] * E
            used = {}
            for e in range(E):
                if pid[e] >= 0:
                    ps[e] = used.get(pid[e], 0)
                    used[pid[e]] = ps[e] + 1
            for chunk in (1, 7, 16, 48, 1000):
                _check(E, H, I, ls, pid, ps, P, chunk)


def test_contiguous_regions_merge():
    # 4 experts on one peer, in order: one w13 region and one w2 region
    plan = plan_prefetch(4, 4, 2, [-1] * 4, [0] * 4, [0, 1, 2, 3], 1, 10 ** 9)
    assert plan == [(0, 0, 0, 0, 4 * 32), (0, 1, 0, 0, 4 * 16)]


def test_last_slice_short_and_rr():
    plan = plan_prefetch(2, 4, 2, [-1, -1], [0, 1], [0, 0], 2, 20)
    # per peer: w13 32 B -> 20 + 12, w2 16 B -> 16; round robin p0, p1
    assert [x[4] for x in plan] == [20, 20, 12, 12, 16, 16]
    assert [x[0] for x in plan] == [0, 1, 0, 1, 0, 1]


def test_redundant_expert_not_copied():
    plan = plan_prefetch(3, 4, 2, [0, 1, -1], [0, 0, 0], [0, 1, 2], 1, 1000)
    assert all(x[2] in (2 * 32, 2 * 16) for x in plan)
    assert len(plan) == 2


def test_r1_split_counts():
    E, H, I = 256, 7168, 2048
    ls = [e if e < 64 else -1 for e in range(E)]
    pid = [-1 if e < 64 else (e - 64) // 64 for e in range(E)]
    ps = [-1 if e < 64 else (e - 64) % 64 for e in range(E)]
    plan = plan_prefetch(E, H, I, ls, pid, ps, 3, 16 << 20)
    total = sum(x[4] for x in plan)
    assert total == 192 * 3 * H * I * 2
    assert len(plan) == 3 * (-(-64 * 2 * I * H * 2 // (16 << 20)) + -(-64 * H * I * 2 // (16 << 20)))


def test_group_map_oracle_partitions_and_rotates():
    """The group-map oracle against what its reading fixes: every expert
    is hosted by exactly one rank, the blocks are contiguous and their sizes
    differ by at most one, a rank's own experts take slots 0, 1, ..., and
    peer p of rank r is rank (r + 1 + p) mod N."""
    from oracle import group_map
    for E in (5, 16, 256):
        for N in range(1, 9):
            if N > E:
                continue
            hosts = {}
            for r in range(N):
                ls, pid, ps = group_map(E, N, r)
                own = [e for e in range(E) if ls[e] >= 0]
                assert [ls[e] for e in own] == list(range(len(own)))
                assert own == list(range(own[0], own[0] + len(own))) if own else True
                for e in own:
                    hosts.setdefault(e, []).append(r)
                for e in range(E):
                    if ls[e] < 0:
                        q = (r + 1 + pid[e]) % N
                        assert q != r and 0 <= pid[e] < N - 1
                        lq, _, _ = group_map(E, N, q)
                        assert lq[e] == ps[e]                 # the slot the home rank keeps it in
            assert sorted(hosts) == list(range(E)) and all(len(v) == 1 for v in hosts.values())
            sizes = [sum(1 for e in range(E) if hosts[e] == [r]) for r in range(N)]
            assert max(sizes) - min(sizes) <= 1
