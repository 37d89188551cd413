"""The E4M3 (FP8) layer through the C ABI against the oracle's FP8 layer
(mirrored mode): expert weights as E4M3 codes with one scale per expert
tensor, activations quantized per row to E4M3 (binary32 decisions on both
sides, so the codes of x are identical), FP8 tcgen05 GEMMs.  Also: the FP8
output does not depend on placement (DWDP §2), and the staged E4M3 bytes
equal their sources."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, last_tile_tokens, to_f64
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu


def _u8(t):
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


def _expert_codes(lw, e):
    pl = lw.placement
    if pl.local_slot[e] >= 0:
        return _u8(lw.local_w13[pl.local_slot[e]]), _u8(lw.local_w2[pl.local_slot[e]])
    return _u8(lw.peer_w13[pl.peer_id[e]][pl.peer_slot[e]]), _u8(lw.peer_w2[pl.peer_id[e]][pl.peer_slot[e]])


def _run(shape, placement, seed, tokens=None, router_std=0.02, chunk=1 << 20):
    build()
    lw = I.make_layer_fp8(shape, placement, seed, 0, device="cuda", router_std=router_std)
    x = I.make_tokens(shape.T, shape.H, seed).cuda()
    rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, 1, max(1, placement.n_remote()),
                   weight_dtype=B.DTYPE_E4M3)
    try:
        rt.set_layer(0, lw)
        rb = B.RouteBuffers(shape.T, shape.E, shape.k)
        out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
        if placement.n_remote() > 0:
            rt.prefetch(0, 0, chunk, [torch.cuda.Stream()])
        rt.route(x, lw.wr, None, rb)
        rt.moe(0, 0, x, rb, out)
        torch.cuda.synchronize()
        assert rt.device_status() == 0
        o = oracle.default()
        xs = I.bf16_bits(x)
        if isinstance(tokens, str) and tokens == "last_tiles":
            # tokens that own a row of every expert's last m-tile (and of the
            # shared expert's), among those the oracle routes the same way
            full = o.route(xs, I.bf16_bits(lw.wr), None, shape.k)
            agree = (rb.topk_ids.cpu().numpy()[: shape.T] == full["ids"]).all(axis=1)
            tokens, missed = last_tile_tokens(rb.perm.cpu().numpy()[: shape.T * shape.k], rb.offsets.cpu().numpy(),
                                              shape.k, shape.T, agree, n_shared=shape.S)
            assert not missed, f"experts {missed}: no token of their last m-tile routes like the oracle"
            print(f"\n{len(tokens)} tokens cover every expert's last m-tile")
        tok = np.arange(shape.T) if tokens is None else np.asarray(tokens)
        ref = o.route(xs[tok], I.bf16_bits(lw.wr), None, shape.k)
        ids = rb.topk_ids.cpu().numpy()[tok]
        same = (ids == ref["ids"]).all(axis=1)
        sub = np.nonzero(same)[0]
        used = np.unique(ref["ids"][sub])
        w13s, w2s = [None] * shape.E, [None] * shape.E
        for e in used:
            w13s[e], w2s[e] = _expert_codes(lw, int(e))
        kw = {}
        if shape.S:
            kw = dict(shared_w13=_u8(lw.shared_w13), shared_w2=_u8(lw.shared_w2), shared_s13=lw.shared_s13,
                      shared_s2=lw.shared_s2)
        want = o.moe_tokens_fp8(xs[tok], sub, ref["ids"], ref["w"], w13s, w2s, lw.w13_scale, lw.w2_scale,
                                mirrored=True, **kw)
        got = to_f64(out)[tok[sub]]
        assert_close(got, want, what="E4M3 layer output")
        return out.clone(), lw
    finally:
        rt.close()


def test_fp8_small_layer_with_shared_expert():
    _run(I.LayerShape(T=200, H=256, I=128, E=8, k=2, S=1), I.split_placement(8, 4, 1), seed=0)


@pytest.mark.parametrize("H, I_", [(64, 64), (64, 192), (192, 64)])
def test_fp8_rows_narrower_than_a_slice(H, I_):
    # E4M3 rows of 64 bytes (H or I = 64) are narrower than the GEMMs'
    # 128-byte K slice, and 192 bytes end half-way into the second one: the
    # slice's tail past the row end must contribute nothing
    _run(I.LayerShape(T=97, H=H, I=I_, E=6, k=2, S=1), I.split_placement(6, 2, 2), seed=5)


def test_fp8_ragged_many_experts():
    _run(I.LayerShape(T=333, H=512, I=256, E=16, k=4, S=0), I.split_placement(16, 5, 3), seed=1)


def test_fp8_output_independent_of_placement():
    shape = I.LayerShape(T=130, H=256, I=128, E=8, k=2, S=1)
    a, _ = _run(shape, I.split_placement(8, 8, 0), seed=2)
    b, _ = _run(shape, I.split_placement(8, 0, 2), seed=2)
    c, _ = _run(shape, I.split_placement(8, 3, 2, redundant=[4, 6]), seed=2)
    assert torch.equal(a, b) and torch.equal(a, c)


def test_fp8_r1_layer_sample():
    # full R1 shapes in the benchmark's launch configuration; the output of
    # tokens covering every expert's last m-tile
    shape, pl = I.r1_layer(8192)
    _run(shape, pl, seed=3, tokens="last_tiles", chunk=32 << 20)


@pytest.mark.parametrize("shape", [I.LayerShape(T=300, H=512, I=256, E=12, k=2, S=1),
                                   I.LayerShape(T=2048, H=7168, I=2048, E=32, k=4, S=1)],
                         ids=["small", "r1_widths"])
def test_fp8_layer_stages(shape):
    """The E4M3 layer split at its quantized intermediates (workspace
    regions): every routed row of xp holds its token's E4M3 codes and row
    scale as the oracle quantizes x, bit for bit; a against the oracle's
    SiLU(gate) * up of those codes with the row's expert weights; every row
    of the GPU's a quantized by the oracle gives the codes and row scale the
    down GEMM read, bit for bit; y against the oracle's product of those
    codes with the expert's w2.  (Rows: all for the small layer, the first
    and last row of every group at R1 widths.)"""
    build()
    pl = I.split_placement(shape.E, shape.E // 3, 2)
    lw = I.make_layer_fp8(shape, pl, 23, 0, device="cuda")
    x = I.make_tokens(shape.T, shape.H, 23).cuda()
    rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, 1, pl.n_remote(), weight_dtype=B.DTYPE_E4M3)
    try:
        rt.set_layer(0, lw)
        rb = B.RouteBuffers(shape.T, shape.E, shape.k)
        out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
        rt.prefetch(0, 0, 1 << 20, [torch.cuda.Stream()])
        rt.route(x, lw.wr, None, rb)
        rt.moe(0, 0, x, rb, out)
        torch.cuda.synchronize()
        assert rt.device_status() == 0
        T, k, H, I_, E = shape.T, shape.k, shape.H, shape.I, shape.E
        rows_r, rows_all = T * k, T * (k + shape.S)
        xp = _u8(rt.ws_region(T, "xp")).reshape(rows_r, H)
        sxp = rt.ws_region(T, "sxp").view(torch.float32).cpu().numpy()
        a_gpu = rt.ws_region(T, "a").view(torch.bfloat16).reshape(rows_all, I_).float().cpu().numpy()
        aq = _u8(rt.ws_region(T, "aq")).reshape(rows_all, I_)
        sa = rt.ws_region(T, "sa").view(torch.float32).cpu().numpy()
        y_gpu = rt.ws_region(T, "y").view(torch.bfloat16).reshape(rows_all, H).float().cpu().numpy()
        perm = rb.perm.cpu().numpy()[:rows_r]
        offsets = rb.offsets.cpu().numpy()
    finally:
        rt.close()
    o = oracle.default()
    xf = x.float().cpu().numpy()
    xq = [o.quantize_row_e4m3(xf[t]) for t in range(T)]
    for r in range(rows_r):
        c, s_ = xq[perm[r] // k]
        assert np.array_equal(xp[r], c) and np.float32(s_) == sxp[r], f"xp row {r}"
    for r in range(rows_all):
        c, s_ = o.quantize_row_e4m3(a_gpu[r])
        assert np.array_equal(aq[r], c) and np.float32(s_) == sa[r], f"a row {r}: codes or scale differ"
    bounds = list(offsets) + [rows_all]
    a_want, a_got, y_want, y_got = [], [], [], []
    for g in range(E + shape.S):
        lo, hi = int(bounds[g]), int(bounds[g + 1])
        rows = list(range(lo, hi)) if H <= 512 else sorted({lo, hi - 1} if hi > lo else set())
        if not rows:
            continue
        if g < E:
            w13, w2 = _expert_codes(lw, g)
            s13, s2 = lw.w13_scale[g], lw.w2_scale[g]
        else:
            w13, w2, s13, s2 = _u8(lw.shared_w13), _u8(lw.shared_w2), lw.shared_s13, lw.shared_s2
        w13, w2 = w13.reshape(2 * I_, H), w2.reshape(H, I_)
        toks = [perm[r] // k if r < rows_r else r - rows_r for r in rows]
        a_want.append(o.e4m3_linear(np.stack([xq[t][0] for t in toks]),
                                    np.array([xq[t][1] for t in toks], np.float32), w13, s13, epilogue=1))
        a_got.append(a_gpu[rows])
        y_want.append(o.e4m3_linear(aq[rows], sa[rows], w2, s2))
        y_got.append(y_gpu[rows])
    assert_close(np.concatenate(a_got), np.concatenate(a_want), what="E4M3 gate/up output a")
    assert_close(np.concatenate(y_got), np.concatenate(y_want), what="E4M3 down output y")


def test_fp8_layer_at_the_limits():
    # 1024 experts, top-32, shared expert (1025 groups)
    _run(I.LayerShape(T=48, H=128, I=128, E=1024, k=32, S=1), I.split_placement(1024, 512, 2), seed=45)
