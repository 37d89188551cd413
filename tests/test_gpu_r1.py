"""Full-size R1-shaped layers in the launch configuration the benchmark
times (64 local experts, 192 staged from three peer pools in 32 MB
round-robin slices, one shared expert, H=7168, I=2048, E=256, top-8):

  * routing, every token: the oracle's top-k and grouping fed the GPU's own
    fp32 logits give the same expert ids, counts, offsets, perm and inv_perm
    bit for bit (and the same weights within fp32 rounding); independently,
    the GPU's logits match the oracle's fp64 logits and the oracle's own
    routing chooses the same experts for every token that is not a near-tie;
  * layer output: tokens chosen so that between them they own a row of every
    routed expert's last (ragged) 128-row m-tile and of the shared expert's
    last m-tile, against the oracle's mirrored layer (the graded comparison),
    and against its strict layer (fp64 throughout, no intermediate bf16
    rounding), where the GPU may be no further off than the mirrored rounding
    points themselves put the oracle.

Workloads: 8192 tokens (N(0,1) activations, N(0,0.02) router), 16384 tokens
with a Zipf(1.2) router bias over a seeded expert permutation and the 16
hottest experts replicated locally, 256 tokens with logits ~ N(0,1), and
32768 tokens (T (k + 1) = 294 912 expert rows) for the index arithmetic at
scale."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (GpuLayerRun, assert_close, assert_route_same_logits, check_choice_valid,
                         last_tile_tokens, near_tie_tokens, rel_metrics, to_f64)
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu


def _workload(name):
    if name == "r1_8k":
        shape, pl = I.r1_layer(8192)
        return shape, pl, 0.02, None
    if name == "r1_32k":
        shape, pl = I.r1_layer(32768)
        return shape, pl, 0.02, None
    if name == "r1_zipf_16k":
        shape, _ = I.r1_layer(16384)
        bias = I.zipf_bias(256, 1.2, I.seed_for(0, "zipf"))
        pl = I.split_placement(256, 64, 3, redundant=I.hottest_experts(bias, 16))
        return shape, pl, 0.02, bias
    if name == "r1_256":
        shape, pl = I.r1_layer(256)
        return shape, pl, 1.0 / np.sqrt(7168), None
    raise KeyError(name)


def expert_weights_host(lw, pl, experts, E, conv=I.bf16_bits):
    """Host copies of the given experts' weights, resolved through the
    placement (local slot, else its peer pool's slot)."""
    w13s, w2s = [None] * E, [None] * E
    for e in experts:
        e = int(e)
        if pl.local_slot[e] >= 0:
            a, b = lw.local_w13[pl.local_slot[e]], lw.local_w2[pl.local_slot[e]]
        else:
            a, b = lw.peer_w13[pl.peer_id[e]][pl.peer_slot[e]], lw.peer_w2[pl.peer_id[e]][pl.peer_slot[e]]
        w13s[e], w2s[e] = conv(a), conv(b)
    return w13s, w2s


@pytest.mark.parametrize("name", ["r1_8k", "r1_zipf_16k", "r1_256", "r1_32k"])
def test_full_size_layer(name):
    build()
    shape, pl, rstd, bias = _workload(name)
    lw = I.make_layer(shape, pl, 0, 0, device="cuda", router_std=rstd, bias=bias)
    x = I.make_tokens(shape.T, shape.H, 0).cuda()
    run = GpuLayerRun(shape, lw, stage_slots=pl.n_remote())
    try:
        rb, out = run.run(x, chunk_bytes=32 << 20)
        T, k, E = shape.T, shape.k, shape.E
        o = oracle.default()
        # routing of every token, bit for bit, on the GPU's own logits
        assert_route_same_logits(o, rb, T, k, E)
        ids = rb.topk_ids.cpu().numpy()[:T]
        counts = rb.counts.cpu().numpy()
        offsets = rb.offsets.cpu().numpy()
        perm = rb.perm.cpu().numpy()[: T * k]
        if bias is not None:
            # heavy skew really reaches the grouped GEMM
            assert counts.max() > 8 * counts.mean()

        # the oracle's own routing of every token, from its fp64 logits
        xs = I.bf16_bits(x)
        ref = o.route(xs, I.bf16_bits(lw.wr), bias, k)
        z_gpu = rb.logits.cpu().numpy()[:T].astype(np.float64)
        err = np.abs(z_gpu - ref["logits"]).max()
        assert err <= 1e-5 * max(1.0, np.abs(ref["logits"]).max()) + 1e-5, f"logit error {err}"
        tie = near_tie_tokens(ref["logits"], k)
        same = (ids == ref["ids"]).all(axis=1)
        assert same[~tie].all(), f"{(~same & ~tie).sum()} tokens differ without a near-tie"
        check_choice_valid(ref["logits"], ids, k)
        print(f"\n{name}: {tie.sum()} near-tie tokens, {(~same).sum()} chose differently from the oracle's "
              f"fp64 logits")

        # layer output on tokens that cover every expert's last m-tile
        sub, missed = last_tile_tokens(perm, offsets, k, T, same, n_shared=shape.S)
        assert not missed, f"experts {missed}: no token of their last m-tile routes like the oracle"
        w13s, w2s = expert_weights_host(lw, pl, np.unique(ref["ids"][sub]), E)
        sw13, sw2 = I.bf16_bits(lw.shared_w13), I.bf16_bits(lw.shared_w2)
        want = o.moe_tokens(xs, sub, ref["ids"], ref["w"], w13s, w2s, sw13, sw2, mirrored=True)
        got = to_f64(out[torch.from_numpy(sub).cuda()])
        r_m, mae_m = assert_close(got, want, what=f"{name} layer output")
        strict = o.moe_tokens(xs, sub, ref["ids"], ref["w"], w13s, w2s, sw13, sw2, mirrored=False)
        r_s, mae_s = rel_metrics(got, strict)
        r_o, mae_o = rel_metrics(want, strict)
        print(f"{name}: {sub.size} tokens covering {int((counts > 0).sum())} experts' last m-tiles: vs mirrored "
              f"max rel {r_m:.3e} MAE {mae_m:.3e}; vs strict max rel {r_s:.3e} MAE {mae_s:.3e}; oracle mirrored "
              f"vs strict max rel {r_o:.3e} MAE {mae_o:.3e}")
        assert mae_s <= 2.0 * mae_o + 1e-4, (mae_s, mae_o)
        assert r_s <= 2.0 * r_o + 2e-2, (r_s, r_o)
    finally:
        run.close()
