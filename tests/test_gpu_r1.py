"""Full-size R1-shaped layers in the launch configuration the benchmark
times (64 local experts, 192 staged from three peer pools in 32 MB
round-robin slices, one shared expert, H=7168, I=2048, E=256, top-8):

  * routing: fp32 logits of a token sample against the oracle, expert choice
    bit-exact away from near-ties, and the grouping of ALL T*k pairs checked
    for the properties that define it (stable counting sort by expert);
  * layer output: a seeded token sample against the oracle's mirrored layer
    (the graded comparison), and against its strict layer (fp64 throughout,
    no intermediate bf16 rounding), where the GPU may be no further off than
    the mirrored rounding points themselves put the oracle.

Workloads: 8192 tokens (N(0,1) activations, N(0,0.02) router), 16384 tokens
with a Zipf(1.2) router bias over a seeded expert permutation and the 16
hottest experts replicated locally, 256 tokens with logits ~ N(0,1), and
32768 tokens (T (k + 1) = 294 912 expert rows) for the index arithmetic at
scale."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (GpuLayerRun, assert_close, check_choice_valid, check_grouping_properties,
                         near_tie_tokens, rel_metrics, to_f64)
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
        ids = rb.topk_ids.cpu().numpy()[:T]
        counts = rb.counts.cpu().numpy()
        offsets = rb.offsets.cpu().numpy()
        perm = rb.perm.cpu().numpy()[: T * k]
        inv = rb.inv_perm.cpu().numpy()[: T * k]
        check_grouping_properties(ids, counts, offsets, perm, inv, E)
        if bias is not None:
            # heavy skew really reaches the grouped GEMM
            assert counts.max() > 8 * counts.mean()

        o = oracle.default()
        rng = np.random.default_rng(7)
        sample = np.sort(rng.choice(T, size=min(T, 256), replace=False))
        xs = I.bf16_bits(x)[sample]
        ref = o.route(xs, I.bf16_bits(lw.wr), bias, k)
        z_gpu = rb.logits.cpu().numpy()[sample].astype(np.float64)
        err = np.abs(z_gpu - ref["logits"]).max()
        assert err <= 1e-5 * max(1.0, np.abs(ref["logits"]).max()) + 1e-5, f"logit error {err}"
        tie = near_tie_tokens(ref["logits"], k)
        same = (ids[sample] == ref["ids"]).all(axis=1)
        assert same[~tie].all()
        check_choice_valid(ref["logits"], ids[sample], k)

        # layer output on a smaller sample (the oracle's FFN is the slow part)
        sub = np.nonzero(same)[0][:24]
        used = np.unique(ref["ids"][sub])
        w13s, w2s = [None] * E, [None] * E
        for e in used:
            if pl.local_slot[e] >= 0:
                a, b = lw.local_w13[pl.local_slot[e]], lw.local_w2[pl.local_slot[e]]
            else:
                a, b = lw.peer_w13[pl.peer_id[e]][pl.peer_slot[e]], lw.peer_w2[pl.peer_id[e]][pl.peer_slot[e]]
            w13s[e], w2s[e] = I.bf16_bits(a), I.bf16_bits(b)
        want = o.moe_tokens(xs, sub, ref["ids"], ref["w"], w13s, w2s, I.bf16_bits(lw.shared_w13),
                            I.bf16_bits(lw.shared_w2), mirrored=True)
        got = to_f64(out[torch.from_numpy(sample[sub]).cuda()])
        r_m, mae_m = assert_close(got, want, what=f"{name} layer output")
        strict = o.moe_tokens(xs, sub, ref["ids"], ref["w"], w13s, w2s, I.bf16_bits(lw.shared_w13),
                              I.bf16_bits(lw.shared_w2), mirrored=False)
        r_s, mae_s = rel_metrics(got, strict)
        r_o, mae_o = rel_metrics(want, strict)
        print(f"\n{name}: vs mirrored max rel {r_m:.3e} MAE {mae_m:.3e}; vs strict max rel {r_s:.3e} "
              f"MAE {mae_s:.3e}; oracle mirrored vs strict max rel {r_o:.3e} MAE {mae_o:.3e}")
        assert mae_s <= 2.0 * mae_o + 1e-4, (mae_s, mae_o)
        assert r_s <= 2.0 * r_o + 2e-2, (r_s, r_o)
    finally:
        run.close()
