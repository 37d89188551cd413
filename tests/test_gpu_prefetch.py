"""dwdp_prefetch_layer (DWDP §2 double-buffered prefetch, §4.3.2 round-robin
slices): staged bytes equal their sources exactly, stage/layer bookkeeping
is enforced (device and pinned-host peer pools, two or three stages), and
the host-side bounded wait reports a timeout without faulting or hanging
anything (the copy stream is held back by a short GPU sleep, then
released)."""
import numpy as np
import pytest
import torch

from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu


def _setup(n_layers=2, n_stages=2):
    build()
    shape = I.LayerShape(T=64, H=256, I=128, E=12, k=2, S=1)
    pl = I.split_placement(12, 3, 3)
    lws = [I.make_layer(shape, pl, 5, l, device="cuda") for l in range(n_layers)]
    rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, n_layers, pl.n_remote(),
                   n_stages=n_stages)
    for l, lw in enumerate(lws):
        rt.set_layer(l, lw)
    return shape, pl, lws, rt


def _expected_stage(lw, pl):
    """Stage contents by definition: the r-th non-resident expert (ascending
    id) in slot r, copied from its peer slot."""
    w13, w2 = [], []
    for e in range(len(pl.local_slot)):
        if pl.local_slot[e] < 0:
            w13.append(lw.peer_w13[pl.peer_id[e]][pl.peer_slot[e]])
            w2.append(lw.peer_w2[pl.peer_id[e]][pl.peer_slot[e]])
    return torch.stack(w13), torch.stack(w2)


@pytest.mark.parametrize("chunk,n_streams", [(1 << 20, 1), (12_345, 1), (40_000, 3), (10 ** 9, 2)])
def test_stage_bytes_equal_sources(chunk, n_streams):
    shape, pl, lws, rt = _setup()
    try:
        streams = [torch.cuda.Stream() for _ in range(n_streams)]
        for layer, stage in ((0, 0), (1, 1), (1, 0), (0, 1)):
            rt.prefetch(layer, stage, chunk, streams)
            assert rt.wait_stage(stage, 20_000) == 0
            assert B.dwdp_stage_layer(rt.ctx, stage) == layer
            e13, e2 = _expected_stage(lws[layer], pl)
            n = e13.shape[0]
            # stage slots are raw bytes: compare byte for byte
            assert torch.equal(rt.stage_w13[stage][:n], e13.view(torch.uint8).reshape(n, -1))
            assert torch.equal(rt.stage_w2[stage][:n], e2.view(torch.uint8).reshape(n, -1))
    finally:
        rt.close()


def test_stage_from_pinned_host_pools():
    """Peer pools in pinned host memory: the slices cross the host link and
    the staged bytes still equal their sources; the layer output is the same
    as with device pools."""
    build()
    shape = I.LayerShape(T=64, H=256, I=128, E=12, k=2, S=1)
    pl = I.split_placement(12, 3, 3)
    lw = I.make_layer(shape, pl, 6, 0, device="cuda")
    x = I.make_tokens(shape.T, shape.H, 1).cuda()
    outs = []
    for where in ("device", "host"):
        if where == "host":
            for pools in (lw.peer_w13, lw.peer_w2):
                for i, t in enumerate(pools):
                    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    h.copy_(t)
                    pools[i] = h
        rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, 1, pl.n_remote())
        try:
            rt.set_layer(0, lw)
            rt.prefetch(0, 0, 40_000, [torch.cuda.Stream()])
            assert rt.wait_stage(0, 20_000) == 0
            e13, e2 = _expected_stage(lw, pl)
            n = e13.shape[0]
            assert torch.equal(rt.stage_w13[0][:n].cpu(), e13.cpu().view(torch.uint8).reshape(n, -1))
            assert torch.equal(rt.stage_w2[0][:n].cpu(), e2.cpu().view(torch.uint8).reshape(n, -1))
            rb = B.RouteBuffers(shape.T, shape.E, shape.k)
            out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
            rt.route(x, lw.wr, None, rb)
            rt.moe(0, 0, x, rb, out)
            torch.cuda.synchronize()
            assert rt.device_status() == 0
            outs.append(out.clone())
        finally:
            rt.close()
    assert torch.equal(outs[0], outs[1])


def test_stage_must_hold_the_layer():
    shape, pl, lws, rt = _setup()
    try:
        x = I.make_tokens(shape.T, shape.H, 0).cuda()
        rb = B.RouteBuffers(shape.T, shape.E, shape.k)
        out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
        rt.route(x, lws[0].wr, None, rb)
        with pytest.raises(B.DwdpError) as ei:        # nothing staged yet
            rt.moe(0, 0, x, rb, out)
        assert ei.value.code == -2
        rt.prefetch(1, 0, 1 << 20, [torch.cuda.Stream()])
        with pytest.raises(B.DwdpError) as ei:        # stage 0 holds layer 1
            rt.moe(0, 0, x, rb, out)
        assert ei.value.code == -2
        rt.prefetch(0, 1, 1 << 20, [torch.cuda.Stream()])
        rt.moe(0, 1, x, rb, out)                       # stage 1 holds layer 0
        torch.cuda.synchronize()
        assert rt.device_status() == 0
    finally:
        rt.close()


def test_stage_count():
    """A context has n_stages staging buffers (2 by default): stage indexes
    outside [0, n_stages) are rejected before anything is enqueued; with
    three, stage 2 holds a layer like the others."""
    shape, pl, lws, rt = _setup()
    try:
        s = torch.cuda.Stream()
        with pytest.raises(B.DwdpError) as ei:
            rt.prefetch(0, 2, 1 << 20, [s])
        assert ei.value.code == -1 and "stage 2" in str(ei.value)
        assert B.dwdp_stage_layer(rt.ctx, 2) == -1
    finally:
        rt.close()
    shape, pl, lws, rt = _setup(n_stages=3)
    try:
        x = I.make_tokens(shape.T, shape.H, 0).cuda()
        rb = B.RouteBuffers(shape.T, shape.E, shape.k)
        out2 = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
        out0 = torch.empty_like(out2)
        rt.prefetch(1, 2, 1 << 20, [torch.cuda.Stream()])
        rt.prefetch(1, 0, 1 << 20, [torch.cuda.Stream()])
        assert rt.wait_stage(2, 20_000) == 0 and B.dwdp_stage_layer(rt.ctx, 2) == 1
        e13, e2 = _expected_stage(lws[1], pl)
        n = e13.shape[0]
        assert torch.equal(rt.stage_w13[2][:n], e13.view(torch.uint8).reshape(n, -1))
        rt.route(x, lws[1].wr, None, rb)
        rt.moe(1, 2, x, rb, out2)
        rt.moe(1, 0, x, rb, out0)
        torch.cuda.synchronize()
        assert rt.device_status() == 0 and torch.equal(out2, out0)
        with pytest.raises(B.DwdpError) as ei:
            rt.moe(1, 3, x, rb, out2)
        assert ei.value.code == -1
    finally:
        rt.close()


def test_single_stage_serialises_layers():
    """n_stages = 1: layer 1's copy into the only stage waits for layer 0's
    down GEMM (the stage's free event), so the two layers run one after the
    other, and their outputs equal those of a two-stage context."""
    outs = {}
    for n_stages in (1, 2):
        shape, pl, lws, rt = _setup(n_stages=n_stages)
        try:
            copy = [torch.cuda.Stream()]
            compute = torch.cuda.Stream()
            res = []
            for layer in (0, 1):
                stage = 0 if n_stages == 1 else layer
                x = I.make_tokens(shape.T, shape.H, 7, step=layer).cuda()
                rb = B.RouteBuffers(shape.T, shape.E, shape.k)
                out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
                rt.prefetch(layer, stage, 50_000, copy)
                rt.route(x, lws[layer].wr, None, rb, compute)
                rt.moe(layer, stage, x, rb, out, compute)
                res.append(out)
            torch.cuda.synchronize()
            assert rt.device_status() == 0
            outs[n_stages] = [o.clone() for o in res]
        finally:
            rt.close()
    for a, b in zip(outs[1], outs[2]):
        assert torch.equal(a, b)


def test_unmapped_layer_and_bad_arguments():
    build()
    rt = B.Runtime(256, 128, 8, 2, 0, 64, 2, 4)
    try:
        s = torch.cuda.Stream()
        with pytest.raises(B.DwdpError) as ei:
            rt.prefetch(1, 0, 1 << 20, [s])
        assert ei.value.code == -2
        with pytest.raises(B.DwdpError) as ei:
            rt.prefetch(5, 0, 1 << 20, [s])
        assert ei.value.code == -1
        with pytest.raises(B.DwdpError) as ei:     # expert 7 has no copy
            ls = [0, 1, 2, 3, -1, -1, -1, -1]
            B.dwdp_set_expert_map(rt.ctx, 0, B.pool(rt.stage_w13[0], rt.stage_w2[0]), [B.pool(rt.stage_w13[1], rt.stage_w2[1])],
                                  ls, [-1, -1, -1, -1, 0, 0, 0, -1], [0, 0, 0, 0, 0, 1, 2, 0])
        assert ei.value.code == -1 and "expert 7" in str(ei.value)
    finally:
        rt.close()


def test_wait_stage_times_out_then_completes():
    shape, pl, lws, rt = _setup()
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            torch.cuda._sleep(int(2e8))          # ~0.1 s of GPU spinning on the copy stream
        rt.prefetch(0, 0, 1 << 20, [s])
        assert rt.wait_stage(0, 0) == -4       # TIMEOUT, reported on the host
        assert rt.wait_stage(0, 30_000) == 0
        assert rt.device_status() == 0
    finally:
        rt.close()
