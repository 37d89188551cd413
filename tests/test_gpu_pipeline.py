"""Several layers back to back with the double-buffered prefetch of DWDP
section 2: layer l+1's non-resident experts are copied into the other stage
while layer l computes, and a stage is refilled only after the last layer
that read it is done (the context's ready / freed events).

Every layer's output must be bit-identical to a fully serialised run
(prefetch, wait, compute, one layer at a time): a stage overwritten too
early, or read too soon, changes the bytes.  The overlapped outputs are also
checked against the oracle (bf16) on a token sample."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, host_layer, to_f64
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu

N_LAYERS = 4


def _layers(dtype, shape, pl):
    make = {B.DTYPE_BF16: I.make_layer, B.DTYPE_NVFP4: I.make_layer_nvfp4}[dtype]
    return [make(shape, pl, 11, l, device="cuda") for l in range(N_LAYERS)]


def _run(dtype, shape, pl, lws, xs, overlapped, chunk, n_stages=2):
    """Layer l reads stage l % S; after it is enqueued, layer l + S - 1 is
    prefetched into stage (l + S - 1) % S, which layer l - 1 read (S = 2:
    the next layer into the other stage)."""
    S = n_stages
    rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, N_LAYERS, pl.n_remote(),
                   weight_dtype=dtype, n_stages=S)
    try:
        for l, lw in enumerate(lws):
            rt.set_layer(l, lw)
        compute = torch.cuda.Stream()
        copy = [torch.cuda.Stream()]
        rbs = [B.RouteBuffers(x.shape[0], shape.E, shape.k) for x in xs]
        outs = [torch.empty((x.shape[0], shape.H), dtype=torch.bfloat16, device="cuda") for x in xs]
        for j in range(min(S - 1, N_LAYERS)):
            rt.prefetch(j, j, chunk, copy)
        for l in range(N_LAYERS):
            s = l % S
            if not overlapped:
                assert rt.wait_stage(s, 20_000) == 0
            rt.route(xs[l], lws[l].wr, None, rbs[l], compute)
            rt.moe(l, s, xs[l], rbs[l], outs[l], compute)
            if not overlapped:
                compute.synchronize()
            if l + S - 1 < N_LAYERS:
                # the context makes the copy wait for the down GEMM of the
                # last layer that read that stage
                rt.prefetch(l + S - 1, (l + S - 1) % S, chunk, copy)
        torch.cuda.synchronize()
        assert rt.device_status() == 0
        return [o.clone() for o in outs], rbs
    finally:
        rt.close()


@pytest.mark.parametrize("dtype", [B.DTYPE_BF16, B.DTYPE_NVFP4], ids=["bf16", "nvfp4"])
@pytest.mark.parametrize("ragged", [False, True], ids=["fixed_T", "ragged_T"])
def test_overlapped_layers_equal_serialised(dtype, ragged):
    """ragged: each layer gets its own token count (one workspace sized for
    the largest), as in the benchmark's 4-layer pipeline.  Two stages (the
    pages' double buffering) and three (copies two layers ahead)."""
    build()
    shape = I.LayerShape(T=300, H=512, I=256, E=12, k=2, S=1)
    pl = I.split_placement(12, 4, 2)
    lws = _layers(dtype, shape, pl)
    Ts = [300, 257, 129, 1] if ragged else [shape.T] * N_LAYERS
    xs = [I.make_tokens(Ts[l], shape.H, 3, step=l).cuda() for l in range(N_LAYERS)]
    ser, _ = _run(dtype, shape, pl, lws, xs, overlapped=False, chunk=1 << 20)
    for n_stages, chunk in ((2, 50_000), (2, 1 << 20), (3, 50_000), (4, 1 << 20)):
        ovl, _ = _run(dtype, shape, pl, lws, xs, overlapped=True, chunk=chunk, n_stages=n_stages)
        for l in range(N_LAYERS):
            assert torch.equal(ovl[l], ser[l]), \
                f"layer {l} differs from the serialised run ({n_stages} stages, chunk {chunk})"


def test_overlapped_layers_match_oracle():
    build()
    shape = I.LayerShape(T=300, H=512, I=256, E=12, k=2, S=1)
    pl = I.split_placement(12, 4, 2)
    lws = _layers(B.DTYPE_BF16, shape, pl)
    xs = [I.make_tokens(shape.T, shape.H, 3, step=l).cuda() for l in range(N_LAYERS)]
    outs, rbs = _run(B.DTYPE_BF16, shape, pl, lws, xs, overlapped=True, chunk=50_000)
    o = oracle.default()
    tok = np.arange(0, shape.T, 7)
    for l in range(N_LAYERS):
        xb = I.bf16_bits(xs[l])
        ref = o.route(xb[tok], I.bf16_bits(lws[l].wr), None, shape.k)
        same = (rbs[l].topk_ids.cpu().numpy()[tok] == ref["ids"]).all(axis=1)   # near-ties aside
        assert same.mean() > 0.9
        sub = np.nonzero(same)[0]
        w13s, w2s, sw13, sw2 = host_layer(lws[l])
        want = o.moe_tokens(xb[tok], sub, ref["ids"], ref["w"], w13s, w2s, sw13, sw2, mirrored=True)
        assert_close(to_f64(outs[l])[tok[sub]], want, what=f"layer {l}")
