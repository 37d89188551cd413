"""dwdp_route (router GEMM on tcgen05, warp top-k, stable grouping) against
the oracle: fp32 logits within accumulation error, chosen experts / counts /
offsets / permutations bit-exact (near-tie tokens checked for validity),
weights within fp32 error."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_choice_valid, check_grouping_properties, near_tie_tokens, to_f64
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu


def _route_case(T, H, E, k, seed, router_std=0.02, bias=None, zero_router=False):
    build()
    rt = B.Runtime(H, 128, E, k, 0, T, 1, 0)
    try:
        x = I.make_tokens(T, H, seed).cuda()
        wr = I.randn_bf16((E, H), router_std, I.seed_for(seed, "Wr"))
        if zero_router:
            wr.zero_()
        wr = wr.cuda()
        bt = torch.from_numpy(bias).cuda() if bias is not None else None
        rb = B.RouteBuffers(T, E, k, keep_logits=True)
        rt.route(x, wr, bt, rb)
        torch.cuda.synchronize()
        assert rt.device_status() == 0
        o = oracle.default()
        ref = o.route(I.bf16_bits(x), I.bf16_bits(wr), bias, k, decide_fp32=True)
        z_gpu = rb.logits.cpu().numpy().astype(np.float64)
        err = np.abs(z_gpu - ref["logits"]).max()
        assert err <= 1e-5 * max(1.0, np.abs(ref["logits"]).max()) + 1e-5, f"logit error {err}"
        ids = rb.topk_ids.cpu().numpy()
        tie = near_tie_tokens(ref["logits"], k)
        same = (ids == ref["ids"]).all(axis=1)
        assert same[~tie].all(), f"{(~same & ~tie).sum()} tokens differ without a near-tie"
        check_choice_valid(ref["logits"], ids, k)
        counts = rb.counts.cpu().numpy()
        offsets = rb.offsets.cpu().numpy()
        perm = rb.perm.cpu().numpy()[: T * k]
        inv = rb.inv_perm.cpu().numpy()[: T * k]
        if same.all():
            assert np.array_equal(counts, ref["counts"])
            assert np.array_equal(offsets, ref["offsets"])
            assert np.array_equal(perm, ref["perm"])
            assert np.array_equal(inv, ref["inv"])
        else:
            check_grouping_properties(ids, counts, offsets, perm, inv, E)
        w = rb.topk_w.cpu().numpy().astype(np.float64)
        # w_j = exp(z_j) / sum_i exp(z_i) over the chosen set, so
        # |dw_j| <= w_j * 2 max|dz| (+ fp32 rounding of the softmax itself)
        bound = 2.0 * err * w[same] + 2e-6
        assert (np.abs(w[same] - ref["w"][same]) <= bound).all()
        assert np.allclose(w.sum(1), 1.0, atol=2e-6)
        return ids, w
    finally:
        rt.close()


def test_tiny_layer_routing():
    _route_case(64, 256, 8, 2, seed=0)


def test_ragged_tokens_many_experts_with_bias():
    rng = np.random.default_rng(3)
    bias = rng.standard_normal(64).astype(np.float32)
    _route_case(1000, 512, 64, 6, seed=1, router_std=0.05, bias=bias)


def test_r1_router_shape_subset():
    # R1 router shapes (H=7168, E=256, top-8) on 300 tokens: 3 m-tiles, ragged
    _route_case(300, 7168, 256, 8, seed=2)


def test_k_equals_e_and_single_expert():
    ids, w = _route_case(77, 128, 4, 4, seed=4, router_std=0.2)
    assert (ids == np.arange(4)).all()
    ids, w = _route_case(5, 64, 1, 1, seed=5)
    assert (ids == 0).all() and np.allclose(w, 1.0)


def test_equal_logits_tie_to_lower_id():
    ids, w = _route_case(40, 128, 16, 3, seed=6, zero_router=True)
    assert (ids == np.arange(3)).all()
    assert np.allclose(w, 1.0 / 3.0, atol=1e-7)


def test_single_token():
    _route_case(1, 256, 8, 2, seed=7)


def test_non_finite_logit_is_reported_and_routing_stays_valid():
    """A NaN in one token's row makes every one of its logits NaN: that
    token still gets k distinct experts, every other token is routed as the
    oracle routes it, the grouping stays consistent, and the context's error
    word reports the non-finite logit (DEVICE_CHECK) once."""
    build()
    T, H, E, k = 200, 256, 16, 4
    rt = B.Runtime(H, 128, E, k, 0, T, 1, 0)
    try:
        x = I.make_tokens(T, H, 9).cuda()
        x[17, 3] = float("nan")
        wr = I.randn_bf16((E, H), 0.05, I.seed_for(9, "Wr")).cuda()
        rb = B.RouteBuffers(T, E, k)
        rt.route(x, wr, None, rb)
        torch.cuda.synchronize()
        assert rt.device_status() == -6                      # DEVICE_CHECK, read and cleared
        assert "0x80" in B.dwdp_last_error(rt.ctx)
        assert rt.device_status() == 0
        ids = rb.topk_ids.cpu().numpy()
        assert len(set(ids[17].tolist())) == k
        good = np.arange(T) != 17
        o = oracle.default()
        xs = I.bf16_bits(x)[good]
        ref = o.route(xs, I.bf16_bits(wr), None, k, decide_fp32=True)
        tie = near_tie_tokens(ref["logits"], k)
        same = (ids[good] == ref["ids"]).all(axis=1)
        assert same[~tie].all()
        check_grouping_properties(ids, rb.counts.cpu().numpy(), rb.offsets.cpu().numpy(),
                                  rb.perm.cpu().numpy()[: T * k], rb.inv_perm.cpu().numpy()[: T * k], E)
    finally:
        rt.close()


def test_tensor_mapped_inputs_must_be_this_devices_memory():
    """x and the router weight are read through TMA tensor maps: pinned host
    memory (which the GPU could reach) is refused on the host, before
    anything is enqueued."""
    build()
    T, H, E, k = 8, 256, 8, 2
    rt = B.Runtime(H, 128, E, k, 0, T, 1, 0)
    try:
        x_host = I.make_tokens(T, H, 1).pin_memory()
        wr = I.randn_bf16((E, H), 0.02, I.seed_for(1, "Wr")).cuda()
        rb = B.RouteBuffers(T, E, k)
        with pytest.raises(B.DwdpError) as ei:
            rt.route(x_host, wr, None, rb)
        assert ei.value.code == -1 and "device memory" in str(ei.value)
        with pytest.raises(B.DwdpError) as ei:
            B.dwdp_route_static(x_host, T, H, E, k, wr, None, rb.c)
        assert ei.value.code == -1 and "device memory" in str(ei.value)
        torch.cuda.synchronize()
        assert rt.device_status() == 0
    finally:
        rt.close()


@pytest.mark.parametrize("T, H, E, k", [(200, 256, 1024, 32), (300, 128, 300, 16), (129, 256, 512, 5)],
                         ids=["E1024_k32", "E300_k16", "E512_k5"])
def test_routing_at_the_limits(T, H, E, k):
    # the largest expert count and top-k the ABI accepts (32 logits per lane,
    # a four-n-tile router GEMM), E not a multiple of the warp, k beyond the
    # specialised widths
    _route_case(T, H, E, k, seed=8, router_std=0.05)
