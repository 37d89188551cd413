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


def test_full_size_pipeline_r1():
    """The 4-layer R1 pipeline in the benchmark's launch configuration: four
    distinct 8192-token-shaped layers (64 local + 192 staged experts, three
    peer pools, 16 MB slices), token counts drawn from [6554, 8192], an
    attention-sized GEMM stand-in (T x 7168 x 7168) after each layer while
    the next layer's copy runs.  Every layer's output must be bit-identical
    to the serialised run at full size, and a token sample of every layer
    within the bars of the oracle."""
    build()
    shape, pl = I.r1_layer(8192)
    lws = _layers(B.DTYPE_BF16, shape, pl)
    Ts = I.step_token_counts(N_LAYERS, 6554, 8192, 5)
    xs = [I.make_tokens(Ts[l], shape.H, 5, step=l).cuda() for l in range(N_LAYERS)]
    w_attn = I.randn_bf16((1, shape.H, shape.H), 0.02, I.seed_for(5, "W_attn"), "cuda")
    scratch = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")

    def run(overlapped):
        rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, N_LAYERS, pl.n_remote())
        try:
            for l, lw in enumerate(lws):
                rt.set_layer(l, lw)
            compute, copy = torch.cuda.Stream(), [torch.cuda.Stream()]
            rbs = [B.RouteBuffers(Ts[l], shape.E, shape.k) for l in range(N_LAYERS)]
            outs = [torch.empty((Ts[l], shape.H), dtype=torch.bfloat16, device="cuda") for l in range(N_LAYERS)]
            offs = [torch.tensor([0, Ts[l]], dtype=torch.int32, device="cuda") for l in range(N_LAYERS)]
            rt.prefetch(0, 0, 16 << 20, copy)
            for l in range(N_LAYERS):
                if not overlapped:
                    assert rt.wait_stage(l % 2, 30_000) == 0
                rt.route(xs[l], lws[l].wr, None, rbs[l], compute)
                rt.moe(l, l % 2, xs[l], rbs[l], outs[l], compute)
                if not overlapped:
                    compute.synchronize()
                if l + 1 < N_LAYERS:
                    rt.prefetch(l + 1, (l + 1) % 2, 16 << 20, copy)
                with torch.cuda.stream(compute):      # the attention stand-in, overlapping the copy
                    B.dwdp_grouped_gemm(rt.ctx, B.EPI_BF16, xs[l], Ts[l], shape.H, shape.H, offs[l], 1, [w_attn],
                                        [0, 0], scratch, compute)
            torch.cuda.synchronize()
            assert rt.device_status() == 0
            return outs, rbs
        finally:
            rt.close()

    ser, _ = run(False)
    ovl, rbs = run(True)
    for l in range(N_LAYERS):
        assert torch.equal(ovl[l], ser[l]), f"layer {l} (T={Ts[l]}) differs from the serialised run"
    del ser
    o = oracle.default()
    rng = np.random.default_rng(5)
    for l in range(N_LAYERS):
        tok = np.sort(rng.choice(Ts[l], 12, replace=False))
        xb = I.bf16_bits(xs[l])
        ref = o.route(xb[tok], I.bf16_bits(lws[l].wr), None, shape.k)
        same = (rbs[l].topk_ids.cpu().numpy()[tok] == ref["ids"]).all(axis=1)
        sub = np.nonzero(same)[0]
        assert sub.size >= 10
        used = np.unique(ref["ids"][sub])
        w13s, w2s = [None] * shape.E, [None] * shape.E
        for e in used:
            e = int(e)
            if pl.local_slot[e] >= 0:
                a, b = lws[l].local_w13[pl.local_slot[e]], lws[l].local_w2[pl.local_slot[e]]
            else:
                a, b = lws[l].peer_w13[pl.peer_id[e]][pl.peer_slot[e]], lws[l].peer_w2[pl.peer_id[e]][pl.peer_slot[e]]
            w13s[e], w2s[e] = I.bf16_bits(a), I.bf16_bits(b)
        want = o.moe_tokens(xb[tok], sub, ref["ids"], ref["w"], w13s, w2s, I.bf16_bits(lws[l].shared_w13),
                            I.bf16_bits(lws[l].shared_w2), mirrored=True)
        assert_close(to_f64(ovl[l])[tok[sub]], want, what=f"pipeline layer {l}")
