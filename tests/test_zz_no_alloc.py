"""dwdp_route_static: routing for callers that cannot allocate device memory
(a framework whose caching allocator owns all device memory, a serving loop
that cannot afford cudaMalloc's possible synchronisation, a host with a
fixed memory budget).  It keeps its logits in a file-scope device array
instead of a context and workspace.  Checked through the C ABI against
dwdp_route on the same inputs, on two calls in a row (the second reuses the
array the first left behind), against the oracle's routing, plus its size
limit and its error word (dwdp_route_static_status: zero after clean calls,
the non-finite-logit bit after a token with a NaN, cleared once read).

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_choice_valid, near_tie_tokens
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu

H, E, K = 7168, 256, 8


def _inputs(T, seed, with_bias):
    x = I.make_tokens(T, H, seed, device="cuda")
    wr = I.randn_bf16((E, H), 0.02, I.seed_for(seed, "Wr"), "cuda")
    bias = None
    if with_bias:
        bias = torch.from_numpy(I.zipf_bias(E, 1.2, I.seed_for(seed, "zipf"))).cuda()
    return x, wr, bias


def _compare(a: B.RouteBuffers, b: B.RouteBuffers, T):
    for name in ("topk_ids", "counts", "offsets"):
        assert torch.equal(getattr(a, name)[: T if name == "topk_ids" else None],
                           getattr(b, name)[: T if name == "topk_ids" else None]), name
    assert torch.equal(a.perm[: T * K], b.perm[: T * K])
    assert torch.equal(a.inv_perm[: T * K], b.inv_perm[: T * K])
    dw = (a.topk_w[:T] - b.topk_w[:T]).abs().max().item()
    assert dw <= 2e-6, f"weights differ by {dw}"


def test_static_route_matches_route_twice():
    build()
    T_max = 8192
    rt = B.Runtime(H, 2048, E, K, 1, T_max, 1, 0)
    try:
        for call, (T, seed, with_bias) in enumerate([(300, 11, False), (8192, 12, True)]):
            x, wr, bias = _inputs(T, seed, with_bias)
            ref = B.RouteBuffers(T, E, K)
            rt.route(x, wr, bias, ref)
            got = B.RouteBuffers(T, E, K)
            # poison the outputs so stale values cannot pass
            for t in (got.topk_ids, got.counts, got.offsets, got.perm, got.inv_perm):
                t.fill_(-7)
            got.topk_w.fill_(float("nan"))
            B.dwdp_route_static(x, T, H, E, K, wr, bias, got.c)
            torch.cuda.synchronize()
            _compare(ref, got, T)
            assert int(got.counts.sum()) == T * K, f"call {call}"
            assert B.dwdp_route_static_status() == 0, f"call {call}: error word set"
    finally:
        rt.close()


def test_static_route_matches_the_oracle():
    """Expert choice bit-exact against the oracle's routing of the same
    tokens (fp32 decisions; a token whose k-th and (k+1)-th logits are a
    near-tie is checked for validity instead), and the grouping of the
    chosen ids identical to the oracle's grouping of them."""
    build()
    T = 1000
    x, wr, bias = _inputs(T, 21, True)
    got = B.RouteBuffers(T, E, K)
    B.dwdp_route_static(x, T, H, E, K, wr, bias, got.c)
    torch.cuda.synchronize()
    assert B.dwdp_route_static_status() == 0
    o = oracle.default()
    ref = o.route(I.bf16_bits(x), I.bf16_bits(wr), bias.cpu().numpy(), K, decide_fp32=True)
    ids = got.topk_ids.cpu().numpy()
    tie = near_tie_tokens(ref["logits"], K)
    same = (ids == ref["ids"]).all(axis=1)
    assert same[~tie].all(), f"{(~same & ~tie).sum()} tokens differ without a near-tie"
    check_choice_valid(ref["logits"], ids, K)
    counts, offsets, perm, inv = o.group(ids, E)
    assert np.array_equal(got.counts.cpu().numpy(), counts)
    assert np.array_equal(got.offsets.cpu().numpy(), offsets)
    assert np.array_equal(got.perm.cpu().numpy(), perm)
    assert np.array_equal(got.inv_perm.cpu().numpy(), inv)
    # w_j = exp(z_j) / sum over the chosen set: |dw_j| <= w_j * 2 max|dz|, with
    # |dz| within the logit tolerance of the routing tests (1e-5 relative)
    w = got.topk_w.cpu().numpy().astype(np.float64)
    dz = 1e-5 * max(1.0, np.abs(ref["logits"]).max()) + 1e-5
    assert (np.abs(w[same] - ref["w"][same]) <= 2.0 * dz * w[same] + 2e-6).all()


def test_static_route_reports_a_non_finite_logit_once():
    """A NaN in one token's row makes its logits NaN: the call still routes
    every token, sets the non-finite-logit bit, and the status call reads
    and clears it (the next read is zero)."""
    build()
    T = 64
    x, wr, _ = _inputs(T, 31, False)
    x[5, 100] = float("nan")
    rb = B.RouteBuffers(T, E, K)
    B.dwdp_route_static(x, T, H, E, K, wr, None, rb.c)
    with pytest.raises(B.DwdpError) as ei:
        B.dwdp_route_static_status()
    assert ei.value.code == -6 and ei.value.bits == 1 << 7 and "not finite" in str(ei.value)
    assert B.dwdp_route_static_status() == 0
    ids = rb.topk_ids.cpu().numpy()
    assert int(rb.counts.sum()) == T * K
    for t in range(T):                      # every token, the NaN one included, has k distinct experts
        assert len(set(ids[t].tolist())) == K
    # a clean call afterwards leaves the word at zero
    x[5, 100] = 0.0
    B.dwdp_route_static(x, T, H, E, K, wr, None, rb.c)
    assert B.dwdp_route_static_status() == 0


def test_static_route_rejects_sizes_beyond_its_array():
    build()
    T = (16 << 20) // (4 * E) + 1   # one token more than the array holds
    x, wr, _ = _inputs(16, 3, False)
    rb = B.RouteBuffers(16, E, K)
    with pytest.raises(B.DwdpError) as ei:
        B.dwdp_route_static(x, T, H, E, K, wr, None, rb.c)
    assert ei.value.code == -1 and "16 MiB" in str(ei.value)
