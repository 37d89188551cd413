"""Seeded random small layers through the C ABI against the oracle: expert
counts 1..40 (not multiples of the warp), k = 1..min(E, 8) (the generic
combine path for k outside {2, 4, 8}), T = 1..300, with and without the shared
expert, random local / remote / redundant placements over 1..3 peer pools,
random slice sizes, and all three weight formats (NVFP4 with four and with
eight epilogue warps)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, assert_close_requantized, host_layer, to_f64
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu

DTYPES = {"bf16": B.DTYPE_BF16, "fp8": B.DTYPE_E4M3, "nvfp4": B.DTYPE_NVFP4}


def _u8(t):
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


def _config(seed):
    rng = np.random.default_rng(1000 + seed)
    dtype = ["bf16", "fp8", "nvfp4"][seed % 3]
    E = int(rng.integers(1, 41))
    k = int(rng.integers(1, min(E, 8) + 1))
    S = int(rng.integers(0, 2))
    if dtype == "nvfp4":
        H, I_ = int(rng.choice([256, 512])), int(rng.choice([256, 512]))
    elif dtype == "fp8":   # K at least one 128-byte slice
        H, I_ = int(rng.choice([128, 256, 448])), int(rng.choice([128, 192, 256]))
    else:
        H, I_ = int(rng.choice([128, 256, 448])), int(rng.choice([64, 128, 192]))
    T = int(rng.integers(1, 301))
    n_local = int(rng.integers(0, E + 1))
    n_peers = int(rng.integers(1, 4))
    remote = list(range(n_local, E))
    red = [int(e) for e in rng.choice(remote, size=min(len(remote), int(rng.integers(0, 3))), replace=False)] \
        if remote else []
    chunk = int(rng.choice([4096, 50_000, 1 << 20]))
    return dtype, I.LayerShape(T=T, H=H, I=I_, E=E, k=k, S=S), I.split_placement(E, n_local, n_peers, red), chunk


def _weights_for_oracle(dtype, lw, used):
    shape, pl = lw.shape, lw.placement

    def slot(e):
        if pl.local_slot[e] >= 0:
            return lw.local_w13[pl.local_slot[e]], lw.local_w2[pl.local_slot[e]]
        return lw.peer_w13[pl.peer_id[e]][pl.peer_slot[e]], lw.peer_w2[pl.peer_id[e]][pl.peer_slot[e]]

    if dtype == "bf16":
        return host_layer(lw)
    if dtype == "fp8":
        w13s, w2s = [None] * shape.E, [None] * shape.E
        for e in used:
            a, b = slot(int(e))
            w13s[e], w2s[e] = _u8(a), _u8(b)
        return w13s, w2s
    w = [[None] * shape.E for _ in range(4)]
    for e in used:
        a, b = slot(int(e))
        w[0][e], w[1][e] = I.unpack_nvfp4(a.cpu(), 2 * shape.I, shape.H)
        w[2][e], w[3][e] = I.unpack_nvfp4(b.cpu(), shape.H, shape.I)
    return w


@pytest.mark.parametrize("seed", range(48))
def test_random_layer(seed):
    build()
    dtype, shape, pl, chunk = _config(seed)
    make = {"bf16": I.make_layer, "fp8": I.make_layer_fp8, "nvfp4": I.make_layer_nvfp4}[dtype]
    lw = make(shape, pl, seed, 0, device="cuda", router_std=0.3)
    x = I.make_tokens(shape.T, shape.H, seed).cuda()
    # every other NVFP4 case drains the gate/up accumulator with eight warps
    flags = B.FLAG_WIDE_EPILOGUE if dtype == "nvfp4" and (seed // 3) % 2 else 0
    rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, 1, max(1, pl.n_remote()),
                   weight_dtype=DTYPES[dtype], flags=flags)
    try:
        rt.set_layer(0, lw)
        rb = B.RouteBuffers(shape.T, shape.E, shape.k)
        out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
        if pl.n_remote() > 0:
            rt.prefetch(0, 0, chunk, [torch.cuda.Stream()])
        rt.route(x, lw.wr, None, rb)
        rt.moe(0, 0, x, rb, out)
        torch.cuda.synchronize()
        assert rt.device_status() == 0
        ids = rb.topk_ids.cpu().numpy()
    finally:
        rt.close()
    o = oracle.default()
    xb = I.bf16_bits(x)
    ref = o.route(xb, I.bf16_bits(lw.wr), None, shape.k)
    same = (ids == ref["ids"]).all(axis=1)                 # near-ties aside
    assert same.mean() >= 0.9, f"{(~same).sum()} of {shape.T} tokens routed differently"
    sub = np.nonzero(same)[0]
    used = np.unique(ref["ids"][sub]) if sub.size else np.array([], dtype=np.int32)
    what = f"seed {seed}: {dtype} {shape} local {int((pl.local_slot >= 0).sum())} peers {pl.n_peers}"
    if dtype == "bf16":
        w13s, w2s, sw13, sw2 = _weights_for_oracle(dtype, lw, used)
        want = o.moe_tokens(xb, sub, ref["ids"], ref["w"], w13s, w2s, sw13, sw2, mirrored=True)
        assert_close(to_f64(out)[sub], want, what=what)
    elif dtype == "fp8":
        w13s, w2s = _weights_for_oracle(dtype, lw, used)
        kw = {}
        if shape.S:
            kw = dict(shared_w13=_u8(lw.shared_w13), shared_w2=_u8(lw.shared_w2), shared_s13=lw.shared_s13,
                      shared_s2=lw.shared_s2)
        want = o.moe_tokens_fp8(xb, sub, ref["ids"], ref["w"], w13s, w2s, lw.w13_scale, lw.w2_scale, mirrored=True,
                                **kw)
        assert_close(to_f64(out)[sub], want, what=what)
    else:
        w = _weights_for_oracle(dtype, lw, used)
        shared = None
        if shape.S:
            c13, f13 = I.unpack_nvfp4(lw.shared_w13.cpu(), 2 * shape.I, shape.H)
            c2, f2 = I.unpack_nvfp4(lw.shared_w2.cpu(), shape.H, shape.I)
            shared = (c13, f13, lw.shared_s13, c2, f2, lw.shared_s2)
        want = o.moe_tokens_nvfp4(xb, sub, ref["ids"], ref["w"], w[0], w[1], lw.w13_scale, w[2], w[3], lw.w2_scale,
                                  shared=shared, mirrored=True)
        assert_close_requantized(to_f64(out)[sub], want, what=what)


def _r1_width_config(seed):
    rng = np.random.default_rng(5000 + seed)
    dtype = ["bf16", "fp8", "nvfp4"][seed % 3]
    E = int(rng.integers(9, 65))
    k = int(rng.integers(1, 9))
    S = int(rng.integers(0, 2))
    T = int(rng.integers(1, 1500))
    n_local = int(rng.integers(0, E + 1))
    n_peers = int(rng.integers(1, 4))
    remote = list(range(n_local, E))
    red = [int(e) for e in rng.choice(remote, size=min(len(remote), int(rng.integers(0, 4))), replace=False)] \
        if remote else []
    return dtype, I.LayerShape(T=T, H=7168, I=2048, E=E, k=k, S=S), I.split_placement(E, n_local, n_peers, red)


@pytest.mark.parametrize("seed", range(6))
def test_random_r1_width_layer(seed):
    """Random layers at the R1 widths (H = 7168, I = 2048: 28 / 8 K slices and
    8 / 28 n-tiles per GEMM) with random expert counts, top-k, token counts,
    placements and the three weight formats, in 32 MB slices; the output of
    tokens that between them own a row of every expert's last m-tile (and the
    shared expert's) against the oracle."""
    from gpu_helpers import last_tile_tokens
    build()
    dtype, shape, pl = _r1_width_config(seed)
    make = {"bf16": I.make_layer, "fp8": I.make_layer_fp8, "nvfp4": I.make_layer_nvfp4}[dtype]
    # logits ~ N(0, 1), so every chosen expert carries weight
    lw = make(shape, pl, 50 + seed, 0, device="cuda", router_std=float(1.0 / np.sqrt(shape.H)))
    x = I.make_tokens(shape.T, shape.H, 50 + seed).cuda()
    rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, 1, max(1, pl.n_remote()),
                   weight_dtype=DTYPES[dtype])
    try:
        rt.set_layer(0, lw)
        rb = B.RouteBuffers(shape.T, shape.E, shape.k)
        out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
        if pl.n_remote() > 0:
            rt.prefetch(0, 0, 32 << 20, [torch.cuda.Stream()])
        rt.route(x, lw.wr, None, rb)
        rt.moe(0, 0, x, rb, out)
        torch.cuda.synchronize()
        assert rt.device_status() == 0
        ids = rb.topk_ids.cpu().numpy()[: shape.T]
        perm = rb.perm.cpu().numpy()[: shape.T * shape.k]
        offsets = rb.offsets.cpu().numpy()
    finally:
        rt.close()
    o = oracle.default()
    xb = I.bf16_bits(x)
    ref = o.route(xb, I.bf16_bits(lw.wr), None, shape.k)
    same = (ids == ref["ids"]).all(axis=1)
    assert same.mean() >= 0.9
    sub, missed = last_tile_tokens(perm, offsets, shape.k, shape.T, same, n_shared=shape.S)
    assert not missed
    used = np.unique(ref["ids"][sub])
    what = f"seed {seed}: {dtype} {shape} local {int((pl.local_slot >= 0).sum())} peers {pl.n_peers}"
    print(f"\n{what}: {sub.size} tokens")
    if dtype == "bf16":
        w13s, w2s, sw13, sw2 = _weights_for_oracle(dtype, lw, used)
        want = o.moe_tokens(xb, sub, ref["ids"], ref["w"], w13s, w2s, sw13, sw2, mirrored=True)
        assert_close(to_f64(out)[sub], want, what=what)
    elif dtype == "fp8":
        w13s, w2s = _weights_for_oracle(dtype, lw, used)
        kw = {}
        if shape.S:
            kw = dict(shared_w13=_u8(lw.shared_w13), shared_w2=_u8(lw.shared_w2), shared_s13=lw.shared_s13,
                      shared_s2=lw.shared_s2)
        want = o.moe_tokens_fp8(xb, sub, ref["ids"], ref["w"], w13s, w2s, lw.w13_scale, lw.w2_scale, mirrored=True,
                                **kw)
        assert_close(to_f64(out)[sub], want, what=what)
    else:
        w = _weights_for_oracle(dtype, lw, used)
        shared = None
        if shape.S:
            c13, f13 = I.unpack_nvfp4(lw.shared_w13.cpu(), 2 * shape.I, shape.H)
            c2, f2 = I.unpack_nvfp4(lw.shared_w2.cpu(), shape.H, shape.I)
            shared = (c13, f13, lw.shared_s13, c2, f2, lw.shared_s2)
        want = o.moe_tokens_nvfp4(xb, sub, ref["ids"], ref["w"], w[0], w[1], lw.w13_scale, w[2], w[3], lw.w2_scale,
                                  shared=shared, mirrored=True)
        assert_close_requantized(to_f64(out)[sub], want, what=what)
