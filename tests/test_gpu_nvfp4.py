"""The NVFP4 path through the C ABI against the oracle.

* Activation quantization (dwdp_quantize_rows, the kernels the layer uses):
  codes, E4M3 block scales and row scales bit-exact against the oracle's row
  quantizer, which takes every decision in binary32 as the kernels do (E4M3
  rows too).
* The NVFP4 layer (mirrored mode): expert weights as E2M1 codes with E4M3
  scales per 16-element block and a tensor scale per expert tensor,
  activations quantized per row, block-scaled FP4 tcgen05 GEMMs.  x's codes
  are the same on both sides; a's can differ where a one-ulp difference of
  bf16 a (fp32 vs fp64 sums) straddles an E2M1 rounding boundary, so the
  bar admits rare flips (gpu_helpers.assert_close_requantized).
* The output does not depend on placement (DWDP section 2).

Pool slots are read back into math layout here by plain index arithmetic
from the layout dwdp.h states for DWDP_DTYPE_NVFP4."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, assert_close_requantized, last_tile_tokens, to_f64
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu


def _u8(t):
    return t.detach().contiguous().cpu().numpy().view(np.uint8).ravel()


def _sf_offsets(rows, K):
    """Byte of the block scale of (row, 16-element block) in the chunk layout:
    chunk (row // 128, block // 4) at (rb * K / 64 + ks) * 512, then
    16 * (row % 32) + 4 * ((row % 128) // 32) + block % 4."""
    r = np.arange(rows)[:, None]
    b = np.arange(K // 16)[None, :]
    return ((r // 128) * (K // 64) + b // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + b % 4


def _unpack_codes(packed, rows, K):
    p = np.asarray(packed, dtype=np.uint8).reshape(rows, K // 2)
    c = np.empty((rows, K), dtype=np.uint8)
    c[:, 0::2] = p & 15
    c[:, 1::2] = p >> 4
    return c


def _unpack_slot(blob, rows, K):
    """(codes [rows][K], block scales [rows][K/16]) of one NVFP4 pool slot."""
    blob = np.asarray(blob, dtype=np.uint8)
    n = rows * K // 2
    return _unpack_codes(blob[:n], rows, K), blob[n:][_sf_offsets(rows, K)]


def _expert(lw, e):
    pl, H, I_ = lw.placement, lw.shape.H, lw.shape.I
    if pl.local_slot[e] >= 0:
        b13, b2 = lw.local_w13[pl.local_slot[e]], lw.local_w2[pl.local_slot[e]]
    else:
        b13, b2 = lw.peer_w13[pl.peer_id[e]][pl.peer_slot[e]], lw.peer_w2[pl.peer_id[e]][pl.peer_slot[e]]
    return _unpack_slot(_u8(b13), 2 * I_, H) + _unpack_slot(_u8(b2), H, I_)


def _rows(rng, n, K):
    v = rng.standard_normal((n, K)).astype(np.float32) * rng.uniform(0.01, 30, size=(n, 1)).astype(np.float32)
    v[rng.random((n, K)) < 0.01] *= 40                        # outliers
    v[3] = 0                                                  # an all-zero row
    v[5, 16:48] = 0                                           # two zero blocks
    v[7, :16] = -1e-30                                        # a block of negative near-zeros
    return torch.from_numpy(v).to(torch.bfloat16)


def test_quantize_rows_nvfp4_bit_exact():
    build()
    rng = np.random.default_rng(21)
    rows, K = 300, 512
    x = _rows(rng, rows, K)
    pad = (rows + 127) // 128 * 128
    codes = torch.empty(rows * K // 2, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(pad * K // 16, dtype=torch.uint8, device="cuda")
    rs = torch.empty(rows, dtype=torch.float32, device="cuda")
    B.dwdp_quantize_rows(B.DTYPE_NVFP4, x.cuda(), rows, K, codes, sf, rs)
    torch.cuda.synchronize()
    got_c = _unpack_codes(_u8(codes), rows, K)
    got_sf = _u8(sf)[_sf_offsets(rows, K)]
    got_s = rs.cpu().numpy()
    o = oracle.default()
    xf = x.float().numpy()
    for r in range(rows):
        c, f, s = o.quantize_row_nvfp4(xf[r])
        assert np.float32(s) == got_s[r], f"row {r}: scale {got_s[r]} != {s}"
        assert np.array_equal(f, got_sf[r]), f"row {r}: block scales differ"
        assert np.array_equal(c, got_c[r]), f"row {r}: codes differ at {np.nonzero(c != got_c[r])[0][:8]}"


def _bf16_step(v, up):
    """The bf16 neighbour of float32 v (exactly representable in bf16)."""
    b = np.array([v], dtype=np.float32).view(np.uint32)[0] >> 16
    b = b + 1 if (up == (v >= 0)) else b - 1
    return np.array([b << 16], dtype=np.uint32).view(np.float32)[0]


def test_quantize_rows_nvfp4_rounding_boundaries():
    """Rows whose quotients v / eff land exactly on the E2M1 rounding
    thresholds (0.25, 0.75, ..., 5: ties to even) and one bf16 step either
    side.  The row amax is 2688 * 2^j, so s = 2^j and each block's scale
    (block amax 6 * e * 2^j) is the E4M3 value e exactly; every value is
    bf16-representable.  Codes, scales and row scales must match the oracle
    (binary32 division) bit for bit."""
    build()
    rng = np.random.default_rng(24)
    rows, K = 256, 512
    thresholds = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    mant = np.array([1, 1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875], dtype=np.float32)
    x = np.zeros((rows, K), dtype=np.float32)
    for r in range(rows):
        s = np.float32(2.0 ** int(rng.integers(-30, 30)))
        x[r, 0] = np.float32(2688.0) * s                              # the row amax: s = 2^j
        for b in range(1, K // 16):
            e = mant[rng.integers(0, 8)] * np.float32(2.0 ** int(rng.integers(-6, 6)))
            blk = np.empty(16, dtype=np.float32)
            blk[0] = np.float32(6.0) * e * s                          # the block amax: scale code = e
            for i in range(1, 16):
                v = thresholds[rng.integers(0, 7)] * e * s
                step = rng.integers(0, 3)                             # on the threshold, or one bf16 step off
                if step:
                    v = _bf16_step(v, step == 1)
                blk[i] = v if rng.random() < 0.5 else -v
            x[r, 16 * b:16 * b + 16] = blk
    xt = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(xt.float(), torch.from_numpy(x)), "test rows must be bf16-representable"
    pad = (rows + 127) // 128 * 128
    codes = torch.empty(rows * K // 2, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(pad * K // 16, dtype=torch.uint8, device="cuda")
    rs = torch.empty(rows, dtype=torch.float32, device="cuda")
    B.dwdp_quantize_rows(B.DTYPE_NVFP4, xt.cuda(), rows, K, codes, sf, rs)
    torch.cuda.synchronize()
    got_c = _unpack_codes(_u8(codes), rows, K)
    got_sf = _u8(sf)[_sf_offsets(rows, K)]
    o = oracle.default()
    for r in range(rows):
        c, f, sc = o.quantize_row_nvfp4(x[r])
        assert np.float32(sc) == rs.cpu().numpy()[r], f"row {r}: scale"
        assert np.array_equal(f, got_sf[r]), f"row {r}: block scales differ"
        assert np.array_equal(c, got_c[r]), f"row {r}: codes differ at {np.nonzero(c != got_c[r])[0][:8]}"


def test_quantize_rows_e4m3_bit_exact():
    build()
    rng = np.random.default_rng(22)
    rows, K = 130, 256
    x = _rows(rng, rows, K)
    codes = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    rs = torch.empty(rows, dtype=torch.float32, device="cuda")
    B.dwdp_quantize_rows(B.DTYPE_E4M3, x.cuda(), rows, K, codes, None, rs)
    torch.cuda.synchronize()
    o = oracle.default()
    xf = x.float().numpy()
    got_c, got_s = codes.cpu().numpy(), rs.cpu().numpy()
    for r in range(rows):
        c, s = o.quantize_row_e4m3(xf[r])
        assert np.float32(s) == got_s[r] and np.array_equal(c, got_c[r]), f"row {r}"


def test_quantize_rows_rejects_bad_arguments():
    build()
    x = torch.zeros((4, 96), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(4 * 96, dtype=torch.uint8, device="cuda")
    rs = torch.zeros(4, dtype=torch.float32, device="cuda")
    with pytest.raises(B.DwdpError):    # K not a multiple of 64
        B.dwdp_quantize_rows(B.DTYPE_NVFP4, x, 4, 96, c, c, rs)
    with pytest.raises(B.DwdpError):    # bf16 is not a quantized type
        B.dwdp_quantize_rows(B.DTYPE_BF16, x, 4, 64, c, c, rs)
    with pytest.raises(B.DwdpError):    # NVFP4 needs block scales
        B.dwdp_quantize_rows(B.DTYPE_NVFP4, x, 4, 64, c, None, rs)


def _run(shape, placement, seed, tokens=None, router_std=0.02, chunk=1 << 20):
    build()
    lw = I.make_layer_nvfp4(shape, placement, seed, 0, device="cuda", router_std=router_std)
    x = I.make_tokens(shape.T, shape.H, seed).cuda()
    rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, 1, max(1, placement.n_remote()),
                   weight_dtype=B.DTYPE_NVFP4)
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
        w = [[None] * shape.E for _ in range(4)]
        for e in used:
            for i, a in enumerate(_expert(lw, int(e))):
                w[i][e] = a
        shared = None
        if shape.S:
            c13, f13 = _unpack_slot(_u8(lw.shared_w13), 2 * shape.I, shape.H)
            c2, f2 = _unpack_slot(_u8(lw.shared_w2), shape.H, shape.I)
            shared = (c13, f13, lw.shared_s13, c2, f2, lw.shared_s2)
        want = o.moe_tokens_nvfp4(xs[tok], sub, ref["ids"], ref["w"], w[0], w[1], lw.w13_scale, w[2], w[3],
                                  lw.w2_scale, shared=shared, mirrored=True)
        got = to_f64(out)[tok[sub]]
        assert_close_requantized(got, want, what=f"NVFP4 layer output T={shape.T} H={shape.H} I={shape.I}")
        return out.clone(), lw
    finally:
        rt.close()


def test_nvfp4_small_layer_with_shared_expert():
    _run(I.LayerShape(T=200, H=256, I=256, E=8, k=2, S=1), I.split_placement(8, 4, 1), seed=0)


def test_nvfp4_ragged_several_k_blocks_and_n_tiles():
    # K = 512 (two 256-element slices), G1 4 n-tiles, G2 2 n-tiles, 16 experts top-4
    _run(I.LayerShape(T=333, H=512, I=512, E=16, k=4, S=0), I.split_placement(16, 5, 3), seed=1)


def test_nvfp4_single_token_and_k_equals_e():
    _run(I.LayerShape(T=1, H=256, I=256, E=4, k=2, S=1), I.split_placement(4, 2, 1), seed=5)
    _run(I.LayerShape(T=70, H=256, I=256, E=4, k=4, S=0), I.split_placement(4, 1, 2), seed=6)


def test_nvfp4_all_local_and_all_remote():
    shape = I.LayerShape(T=129, H=256, I=512, E=8, k=2, S=1)
    a, _ = _run(shape, I.split_placement(8, 8, 0), seed=7)
    b, _ = _run(shape, I.split_placement(8, 0, 3), seed=7)
    assert torch.equal(a, b)


def test_nvfp4_output_independent_of_placement():
    shape = I.LayerShape(T=130, H=256, I=256, E=8, k=2, S=1)
    a, _ = _run(shape, I.split_placement(8, 8, 0), seed=2)
    b, _ = _run(shape, I.split_placement(8, 0, 2), seed=2)
    c, _ = _run(shape, I.split_placement(8, 3, 2, redundant=[4, 6]), seed=2)
    assert torch.equal(a, b) and torch.equal(a, c)


def _a_tiles(offsets, rows_r, rows_all):
    """A tile and row-in-tile of every row of the down GEMM's A operand:
    expert by expert, ceil(rows / 128) tiles each, then the shared rows."""
    E = offsets.size - 1
    tile = np.empty(rows_all, dtype=np.int64)
    base = 0
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        r = np.arange(lo, hi)
        tile[lo:hi] = base + (r - lo) // 128
        base += (hi - lo + 127) // 128
    r = np.arange(rows_r, rows_all)
    tile[rows_r:] = base + (r - rows_r) // 128
    within = np.empty(rows_all, dtype=np.int64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        within[lo:hi] = (np.arange(lo, hi) - lo) % 128
    within[rows_r:] = (np.arange(rows_r, rows_all) - rows_r) % 128
    return tile, within


def _down_path_case(shape, placement, seed, n_gate_rows, chunk):
    """The NVFP4 layer split at its quantized intermediate, each stage held
    to the plain bars (no allowance for requantization flips):
      0. x: every row the gate/up GEMM reads (each routed row in expert order
         and the shared expert's copy) holds the token's codes, block scales
         and row scale as the oracle's row quantizer gives them, bit for bit;
      1. gate/up: the GPU's bf16 a of sampled rows against the oracle's
         SiLU(gate) * up of the same token's x codes (the oracle quantizes x
         itself) and the row's expert weights;
      2. a's codes: every row of the GPU's bf16 a quantized by the oracle's
         row quantizer gives, bit for bit, the codes, E4M3 block scales (at
         their A-tile chunk positions) and row scale the down GEMM read;
      3. down: the GPU's y of sampled rows (the last row of every expert's
         group, in its last m-tile, and of the shared rows) against the
         oracle's product of those codes with the expert's w2.
    The layer output itself keeps the end-to-end check of _run."""
    build()
    sh = shape
    lw = I.make_layer_nvfp4(sh, placement, seed, 0, device="cuda")
    x = I.make_tokens(sh.T, sh.H, seed).cuda()
    rt = B.Runtime(sh.H, sh.I, sh.E, sh.k, sh.S, sh.T, 1, max(1, placement.n_remote()), weight_dtype=B.DTYPE_NVFP4)
    try:
        rt.set_layer(0, lw)
        rb = B.RouteBuffers(sh.T, sh.E, sh.k)
        out = torch.empty((sh.T, sh.H), dtype=torch.bfloat16, device="cuda")
        if placement.n_remote() > 0:
            rt.prefetch(0, 0, chunk, [torch.cuda.Stream()])
        rt.route(x, lw.wr, None, rb)
        rt.moe(0, 0, x, rb, out)
        torch.cuda.synchronize()
        assert rt.device_status() == 0
        T, k, H, I_, E = sh.T, sh.k, sh.H, sh.I, sh.E
        rows_r, rows_all = T * k, T * (k + sh.S)
        a_gpu = rt.ws_region(T, "a").view(torch.bfloat16).reshape(rows_all, I_).float().cpu().numpy()
        aq = _unpack_codes(_u8(rt.ws_region(T, "aq")), rows_all, I_)
        sa = rt.ws_region(T, "sa").view(torch.float32).cpu().numpy()
        sfa = _u8(rt.ws_region(T, "sfa"))
        y_gpu = rt.ws_region(T, "y").view(torch.bfloat16).reshape(rows_all, H).float().cpu().numpy()
        xp = _unpack_codes(_u8(rt.ws_region(T, "xp")), rows_r, H)
        sxp = rt.ws_region(T, "sxp").view(torch.float32).cpu().numpy()
        xq_sh = _unpack_codes(_u8(rt.ws_region(T, "xq")), T, H)
        sx = rt.ws_region(T, "sx").view(torch.float32).cpu().numpy()
        sfx = _u8(rt.ws_region(T, "sfx"))
        offsets = rb.offsets.cpu().numpy()
        perm = rb.perm.cpu().numpy()[:rows_r]
        o = oracle.default()
        tile, within = _a_tiles(offsets, rows_r, rows_all)

        # 0. x's codes, block scales and row scales in every row the gate/up
        # GEMM reads (each routed row and the shared expert's copy), bit for bit
        xf = x.float().cpu().numpy()
        qx = [o.quantize_row_nvfp4(xf[t]) for t in range(T)]
        cx = np.stack([q[0] for q in qx])
        fx = np.stack([q[1] for q in qx])
        s_x = np.array([q[2] for q in qx], dtype=np.float32)
        tok = perm // k
        assert np.array_equal(xp, cx[tok]), "x codes in expert order differ from the oracle's"
        assert np.array_equal(sxp[:rows_r], s_x[tok]), "x row scales in expert order differ"
        # block scales at their A-tile chunk positions (the gate/up GEMM's A
        # tiles are numbered like the down GEMM's: expert by expert, then the
        # shared rows)
        xblk = np.arange(H // 16)
        r_all = np.arange(rows_all)
        m_all = within[r_all]
        at_x = ((tile[r_all, None] * (H // 64) + xblk[None, :] // 4) * 512 + 16 * (m_all[:, None] % 32)
                + 4 * (m_all[:, None] // 32) + xblk[None, :] % 4)
        want_fx = np.concatenate([fx[tok], fx]) if sh.S else fx[tok]
        assert np.array_equal(sfx[at_x[: want_fx.shape[0]]], want_fx), "x block scales differ"
        if sh.S:
            assert np.array_equal(xq_sh, cx) and np.array_equal(sx, s_x), "the shared expert's x codes differ"

        # 2. a's codes, every row
        blk = np.arange(I_ // 16)
        for r in range(rows_all):
            c, f, s_ = o.quantize_row_nvfp4(a_gpu[r])
            assert np.float32(s_) == sa[r], f"row {r}: row scale {sa[r]} != {s_}"
            assert np.array_equal(c, aq[r]), f"row {r}: codes differ at {np.nonzero(c != aq[r])[0][:8]}"
            m = within[r]
            at = (tile[r] * (I_ // 64) + blk // 4) * 512 + 16 * (m % 32) + 4 * (m // 32) + blk % 4
            assert np.array_equal(f, sfa[at]), f"row {r}: block scales differ"

        def weights(g):
            """(w13 codes, sf, scale, w2 codes, sf, scale) of group g (E: shared)."""
            if g == E:
                c13, f13 = _unpack_slot(_u8(lw.shared_w13), 2 * I_, H)
                c2, f2 = _unpack_slot(_u8(lw.shared_w2), H, I_)
                return c13, f13, lw.shared_s13, c2, f2, lw.shared_s2
            c13, f13, c2, f2 = _expert(lw, g)
            return c13, f13, lw.w13_scale[g], c2, f2, lw.w2_scale[g]

        groups = [(e, int(offsets[e + 1]) - 1) for e in range(E) if offsets[e + 1] > offsets[e]]
        if sh.S:
            groups.append((E, rows_all - 1))
        xb = x.float().cpu().numpy()
        rng = np.random.default_rng(seed)
        gate_rows = set(rng.choice(len(groups), size=min(n_gate_rows, len(groups)), replace=False).tolist())
        a_want, a_got, y_want, y_got = [], [], [], []
        for i, (g, r) in enumerate(groups):
            c13, f13, s13, c2, f2, s2 = weights(g)
            if i in gate_rows:
                # 1. gate/up from the token's own x codes
                t = (int(perm[r]) // k) if r < rows_r else r - rows_r
                xc, xf, xs = o.quantize_row_nvfp4(xb[t])
                a_want.append(o.nvfp4_linear(xc[None], xf[None], np.array([xs], np.float32), c13, f13, s13,
                                             epilogue=1)[0])
                a_got.append(a_gpu[r])
            # 3. down from the codes the GPU's a quantized to
            at = (tile[r] * (I_ // 64) + blk // 4) * 512 + 16 * (within[r] % 32) + 4 * (within[r] // 32) + blk % 4
            y_want.append(o.nvfp4_linear(aq[r][None], sfa[at][None], sa[r:r + 1], c2, f2, s2)[0])
            y_got.append(y_gpu[r])
        ra, ma = assert_close(np.array(a_got), np.array(a_want), what="NVFP4 gate/up output a")
        ry, my = assert_close(np.array(y_got), np.array(y_want), what="NVFP4 down output y")
        print(f"\nNVFP4 T={T}: {rows_all} a rows requantized bit-exact; a vs oracle max rel {ra:.2e} MAE {ma:.2e} "
              f"({len(a_got)} rows); y vs oracle max rel {ry:.2e} MAE {my:.2e} ({len(y_got)} rows)")
    finally:
        rt.close()


def test_nvfp4_down_path_exact_a_codes_small():
    # ragged groups, two K slices for both GEMMs, the shared expert
    _down_path_case(I.LayerShape(T=333, H=512, I=512, E=16, k=4, S=1), I.split_placement(16, 5, 3), seed=8,
                    n_gate_rows=17, chunk=1 << 20)


def test_nvfp4_down_path_exact_a_codes_r1():
    # the 8192-token R1 layer: all 73 728 a rows' codes, down output of every
    # expert's last row, gate/up output of 64 of them
    shape, pl = I.r1_layer(8192)
    _down_path_case(shape, pl, seed=4, n_gate_rows=64, chunk=32 << 20)


def test_nvfp4_r1_layer_sample():
    # full R1 shapes in the benchmark's launch configuration; the output of
    # tokens covering every expert's last m-tile
    shape, pl = I.r1_layer(8192)
    _run(shape, pl, seed=4, tokens="last_tiles", chunk=32 << 20)


@pytest.mark.parametrize("shape", [I.LayerShape(T=333, H=512, I=512, E=16, k=4, S=1),
                                   I.LayerShape(T=2048, H=7168, I=2048, E=32, k=4, S=1)],
                         ids=["small", "r1_widths"])
def test_nvfp4_wide_epilogue_bit_identical(shape):
    """DWDP_FLAG_WIDE_EPILOGUE drains the gate/up accumulator with eight warps
    instead of four: the same arithmetic per element, so the layer's output
    (and a, in the workspace) must not change by a single bit."""
    build()
    pl = I.split_placement(shape.E, shape.E // 4, 3)
    lw = I.make_layer_nvfp4(shape, pl, 11, 0, device="cuda")
    x = I.make_tokens(shape.T, shape.H, 11).cuda()
    outs = []
    for flags in (0, B.FLAG_WIDE_EPILOGUE):
        rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, 1, pl.n_remote(),
                       weight_dtype=B.DTYPE_NVFP4, flags=flags)
        try:
            rt.set_layer(0, lw)
            rb = B.RouteBuffers(shape.T, shape.E, shape.k)
            out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
            rt.prefetch(0, 0, 1 << 20, [torch.cuda.Stream()])
            rt.route(x, lw.wr, None, rb)
            rt.moe(0, 0, x, rb, out)
            torch.cuda.synchronize()
            assert rt.device_status() == 0
            outs.append((out.clone(), rt.ws_region(shape.T, "a").clone()))
        finally:
            rt.close()
    assert torch.equal(outs[0][1], outs[1][1]), "a differs between four and eight epilogue warps"
    assert torch.equal(outs[0][0], outs[1][0]), "output differs between four and eight epilogue warps"


def test_nvfp4_layer_at_the_limits():
    # 1024 experts, top-32, shared expert: 1025 groups, the largest tile
    # table beside the NVFP4 GEMM's shared-memory ring
    _run(I.LayerShape(T=48, H=256, I=256, E=1024, k=32, S=1), I.split_placement(1024, 512, 2), seed=46)
