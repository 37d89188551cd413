"""Prefetch-plan oracle: TEST INFRASTRUCTURE ONLY (plain Python).

What it computes (DWDP: Distributed Weight Data Parallelism..., §2 and §4.3.2;
the news summary at thecoregrid.dev repeats it): before layer l runs, the
experts of layer l that are not resident are copied from the peers that host
them into one of two staging buffers; each copy is cut into fixed-size slices
and the slices of the different sources are issued round-robin, so no single
large pull holds the copy engine.

Readings taken where the pages are silent:
  * A staging buffer holds the non-resident experts of one layer in ascending
    expert id: the r-th non-resident expert goes to stage slot r.
  * The "queues" of the round-robin are the source peers (on one GPU the peers
    are separate device pools).  Each peer's work is its w13 copies in
    ascending expert id followed by its w2 copies in ascending expert id;
    copies that are contiguous in both source and destination are merged
    into one region; each region is cut into slices of ``chunk_bytes`` (the
    last one short).
  * Issue order: slice 0 of peer 0, slice 0 of peer 1, ..., slice 1 of
    peer 0, ...; a peer whose slices have run out drops out of the rotation.

Every entry is (peer, tensor, src_offset, dst_offset, nbytes), tensor 0 = w13
(``2*I*H`` bf16 per expert), 1 = w2 (``H*I`` bf16 per expert); offsets are in
bytes from the start of the peer pool and of the stage buffer respectively.
"""
from __future__ import annotations


def stage_slots(n_experts, local_slot):
    """Stage slot of each expert (-1 for a resident one)."""
    out, r = [], 0
    for e in range(n_experts):
        if local_slot[e] >= 0:
            out.append(-1)
        else:
            out.append(r)
            r += 1
    return out


def plan_prefetch(n_experts, hidden, inter, local_slot, peer_id, peer_slot,
                  n_peers, chunk_bytes, elem_bytes=2, tensor_bytes=None):
    """tensor_bytes = (bytes of one expert's w13, of its w2) overrides
    elem_bytes for formats that are not a whole number of bytes per element."""
    if chunk_bytes <= 0:
        raise ValueError("chunk_bytes must be positive")
    b13 = 2 * inter * hidden * elem_bytes
    b2 = hidden * inter * elem_bytes
    if tensor_bytes is not None:
        b13, b2 = tensor_bytes
    slot = stage_slots(n_experts, local_slot)
    per_peer = []
    for p in range(n_peers):
        copies = []
        for tensor, nb in ((0, b13), (1, b2)):
            for e in range(n_experts):
                if slot[e] < 0:
                    continue
                if peer_id[e] < 0 or peer_id[e] >= n_peers:
                    raise ValueError(f"expert {e} is neither resident nor on a peer")
                if peer_id[e] != p:
                    continue
                copies.append([tensor, peer_slot[e] * nb, slot[e] * nb, nb])
        regions = []
        for c in copies:
            if regions:
                last = regions[-1]
                if (last[0] == c[0] and last[1] + last[3] == c[1]
                        and last[2] + last[3] == c[2]):
                    last[3] += c[3]
                    continue
            regions.append(list(c))
        slices = []
        for tensor, src, dst, nb in regions:
            done = 0
            while done < nb:
                n = min(chunk_bytes, nb - done)
                slices.append((p, tensor, src + done, dst + done, n))
                done += n
        per_peer.append(slices)
    plan = []
    c = 0
    while True:
        emitted = False
        for p in range(n_peers):
            if c < len(per_peer[p]):
                plan.append(per_peer[p][c])
                emitted = True
        if not emitted:
            break
        c += 1
    return plan


def group_map(n_experts, n_ranks, rank):
    """Placement of rank `rank` in a DWDP group of n_ranks ranks (DWDP §2:
    the experts are partitioned over the ranks, each pulls the others'
    experts from their homes).  Readings: rank q hosts the contiguous block
    of experts [floor(q E / N), floor((q + 1) E / N)) in slots 0, 1, ...;
    a rank numbers its peers from the next rank on (peer p = rank
    (rank + 1 + p) mod N), so that the round-robin over peers of
    ``plan_prefetch`` starts every rank at a different source (DWDP §4.3.1:
    many destinations pulling from one source contend).  Returns
    (local_slot, peer_id, peer_slot) lists."""
    homes = []
    for q in range(n_ranks):
        lo, hi = q * n_experts // n_ranks, (q + 1) * n_experts // n_ranks
        homes += [(q, e - lo) for e in range(lo, hi)]
    local_slot, peer_id, peer_slot = [], [], []
    for e in range(n_experts):
        q, slot = homes[e]
        if q == rank:
            local_slot.append(slot)
            peer_id.append(-1)
            peer_slot.append(-1)
        else:
            local_slot.append(-1)
            peer_id.append((q - rank - 1) % n_ranks)
            peer_slot.append(slot)
    return local_slot, peer_id, peer_slot
