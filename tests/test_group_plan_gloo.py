"""A DWDP group's copy plans, rank by rank (DWDP §2: every rank keeps its
partition of the experts and pulls the rest from the other ranks; §4.3.1 and
§4.3.2: pulls of several destinations from one source contend, so the pulls
are cut into fixed-size slices issued round-robin).  Each of four gloo ranks
on CPU builds its own map (dwdp_group_map) and copy plan
(dwdp_plan_prefetch, R1 shapes, 16 MB slices) through the library's host
calls, then the ranks exchange, for every step of their plans, which rank
they pull from.  Checked: every rank stages exactly the experts it does not
host, each from its home rank, once; and at every step of the plan the
ranks pull from distinct sources (no source serves two destinations at
once) when the ranks host equal shares, with the contended steps of an
unequal split confined to its last expert's slices."""
import collections
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

E, H, I = 256, 7168, 2048


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q, chunk):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from moe_expert_grouped_split_gb300 import binding as B
        ls, pid, ps = B.dwdp_group_map(E, world, rank)
        plan = B.dwdp_plan_prefetch(E, H, I, ls, pid, ps, world - 1, chunk)
        # source rank of every slice, in plan order; peer p of rank r is rank (r + 1 + p) mod N
        src = torch.tensor([(rank + 1 + p) % world for (p, _, _, _, _) in plan], dtype=torch.int64)
        n = torch.tensor([src.numel()])
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, n)
        L = int(max(s.item() for s in sizes))
        pad = torch.full((L,), -1, dtype=torch.int64)
        pad[: src.numel()] = src
        gathered = [torch.zeros(L, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(gathered, pad)
        staged = sorted(int(e) for e in np.nonzero(ls < 0)[0])
        homes = {int(e): (rank + 1 + int(pid[e])) % world for e in staged}
        # the same experts with the peers numbered in absolute rank order
        # (peer p = the p-th other rank): every rank's plan then starts at
        # the lowest other rank
        others = [r for r in range(world) if r != rank]
        pid_abs = np.array([-1 if ls[e] >= 0 else others.index(homes[e]) for e in range(E)], dtype=np.int32)
        plan_abs = B.dwdp_plan_prefetch(E, H, I, ls, pid_abs, ps, world - 1, chunk)
        src_abs = torch.tensor([others[p] for (p, _, _, _, _) in plan_abs], dtype=torch.int64)
        pad_abs = torch.full((L,), -1, dtype=torch.int64)       # same slice count as the rotated plan
        pad_abs[: src_abs.numel()] = src_abs
        gathered_abs = [torch.zeros(L, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(gathered_abs, pad_abs)
        q.put((rank, [g.tolist() for g in gathered], staged, homes,
               sum(n_ for (*_, n_) in plan), [g.tolist() for g in gathered_abs]))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def _run(world, chunk):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, chunk)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def _home(e, world):
    return next(r for r in range(world) if r * E // world <= e < (r + 1) * E // world)


@pytest.mark.parametrize("world", [2, 4])
def test_group_plans_cover_and_do_not_contend(world):
    from moe_expert_grouped_split_gb300.build import build
    build()
    out = _run(world, 16 << 20)
    expert_bytes = 3 * H * I * 2
    for rank, gathered, staged, homes, nbytes, _ in out:
        assert staged == [e for e in range(E) if _home(e, world) != rank]
        assert all(homes[e] == _home(e, world) for e in staged)
        assert nbytes == len(staged) * expert_bytes
    seqs = out[0][1]
    L = len(seqs[0])
    assert all(len(s) == L and -1 not in s for s in seqs)        # equal shares: equal plan lengths
    for step in range(L):
        srcs = [seqs[r][step] for r in range(world)]
        assert len(set(srcs)) == world, f"step {step}: sources {srcs}"
        assert all(srcs[r] != r for r in range(world))
    # the contrast: numbered in absolute rank order, every rank's plan starts
    # at the lowest other rank, so one source serves up to N - 1 destinations
    abs_seqs = out[0][5]
    worst = max(max(collections.Counter(abs_seqs[r][step] for r in range(world)).values())
                for step in range(L))
    assert worst == world - 1


def test_unequal_split_contends_only_at_the_tail():
    """Three ranks over 256 experts (85, 85, 86): the plans differ in length
    by one expert's slices, so the steps where two ranks pull from one
    source are only the last ones."""
    from moe_expert_grouped_split_gb300.build import build
    build()
    world = 3
    out = _run(world, 16 << 20)
    seqs = out[0][1]
    L = len(seqs[0])
    bad = [s for s in range(L)
           if len({seqs[r][s] for r in range(world) if seqs[r][s] >= 0})
           < sum(1 for r in range(world) if seqs[r][s] >= 0)]
    per_expert = -(-3 * H * I * 2 // (16 << 20)) + 1                # slices of one expert (w13 and w2 regions)
    assert all(s >= L - 2 * (world - 1) * per_expert for s in bad), bad
