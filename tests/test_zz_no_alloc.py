"""dwdp_route_static: routing for callers that cannot allocate device memory
(a framework whose caching allocator owns all device memory, a serving loop
that cannot afford cudaMalloc's possible synchronisation, a host with a
fixed memory budget).  It keeps its logits in a file-scope device array
instead of a context and workspace.  Checked through the C ABI against
dwdp_route on the same inputs, on two calls in a row (the second reuses the
array the first left behind), plus its size limit.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import numpy as np
import pytest
import torch

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
    finally:
        rt.close()


def test_static_route_rejects_sizes_beyond_its_array():
    build()
    T = (16 << 20) // (4 * E) + 1   # one token more than the array holds
    x, wr, _ = _inputs(16, 3, False)
    rb = B.RouteBuffers(16, E, K)
    with pytest.raises(B.DwdpError) as ei:
        B.dwdp_route_static(x, T, H, E, K, wr, None, rb.c)
    assert ei.value.code == -1 and "16 MiB" in str(ei.value)
