"""The merge-copy baseline (the design DWDP §4.2 removes: the grouped GEMM
reads one contiguous weight buffer per layer, so the resident experts are
merged into it by a device-to-device copy after the staged ones arrive),
as the benchmark times it (bench.MergeCopyLayer, public ABI only):

  * the merged buffer holds, slot for slot, exactly the layer's experts:
    the staged ones in slots 0..R-1 (ascending id), the resident ones after
    them, byte for byte equal to their source pools;
  * the layer computed on the merged buffer is bit-identical to the
    split-pointer layer on the same inputs (the merge changes where the
    weights are read from, not the result), and within the bars of the
    oracle;
  * two layers alternate over the two merged buffers, as in the benchmark."""
import numpy as np
import pytest
import torch

import bench
import oracle
from gpu_helpers import assert_close, host_layer, to_f64
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu


def _expert_bytes(lw, e):
    pl = lw.placement
    if pl.local_slot[e] >= 0:
        a, b = lw.local_w13[pl.local_slot[e]], lw.local_w2[pl.local_slot[e]]
    else:
        a, b = lw.peer_w13[pl.peer_id[e]][pl.peer_slot[e]], lw.peer_w2[pl.peer_id[e]][pl.peer_slot[e]]
    return a.contiguous().view(torch.uint8).reshape(-1), b.contiguous().view(torch.uint8).reshape(-1)


@pytest.mark.parametrize("wdtype", ["bf16", "nvfp4"])
def test_merged_buffer_and_output(wdtype):
    build()
    shape = I.LayerShape(T=300, H=512, I=256, E=16, k=4, S=1)
    pl = I.split_placement(16, 5, 3)
    make = {"bf16": I.make_layer, "nvfp4": I.make_layer_nvfp4}[wdtype]
    code = {"bf16": B.DTYPE_BF16, "nvfp4": B.DTYPE_NVFP4}[wdtype]
    layers = [make(shape, pl, 3, l, device="cuda") for l in range(2)]
    xs = [I.make_tokens(shape.T, shape.H, 3, step=l, device="cuda") for l in range(2)]
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()

    # split pointers: the library's own path
    rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, 2, pl.n_remote(), weight_dtype=code)
    split = []
    try:
        for l, lw in enumerate(layers):
            rt.set_layer(l, lw)
        for l in range(2):
            rb = B.RouteBuffers(shape.T, shape.E, shape.k)
            out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
            rt.prefetch(l, l, 64 << 10, [copy])
            with torch.cuda.stream(compute):
                rt.route(xs[l], layers[l].wr, None, rb, compute)
                rt.moe(l, l, xs[l], rb, out, compute)
            torch.cuda.synchronize()
            assert rt.device_status() == 0
            split.append((out.clone(), rb))
    finally:
        rt.close()

    mc = bench.MergeCopyLayer(B, torch, shape, pl, layers, wdtype)
    try:
        assert mc.R == pl.n_remote() and mc.n_local == 5
        for step in range(4):                   # layers 0, 1, 0, 1 over buffers 0, 1, 0, 1
            l = s = step % 2
            rb = B.RouteBuffers(shape.T, shape.E, shape.k)
            out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
            mc.prefetch(l, s, 64 << 10, [copy])
            mc.layer(l, s, xs[l], rb, out, compute)
            torch.cuda.synchronize()
            assert mc.rt.device_status() == 0
            # the merged buffer: expert e in slot merged_slot[e], byte for byte
            w13 = mc.rt.stage_w13[s]
            w2 = mc.rt.stage_w2[s]
            for e in range(shape.E):
                a, b = _expert_bytes(layers[l], e)
                slot = mc.merged_slot[e]
                assert torch.equal(w13[slot], a), f"step {step}: w13 of expert {e} in slot {slot}"
                assert torch.equal(w2[slot], b), f"step {step}: w2 of expert {e} in slot {slot}"
            assert sorted(mc.merged_slot) == list(range(shape.E))
            # the same layer, bit for bit
            ref_out, ref_rb = split[l]
            assert torch.equal(rb.topk_ids, ref_rb.topk_ids) and torch.equal(rb.perm, ref_rb.perm)
            assert torch.equal(out, ref_out), f"step {step}: merged layer differs from the split-pointer layer"
    finally:
        mc.close()

    # and within the bars of the oracle (bf16; the NVFP4 layer has its own tests)
    if wdtype == "bf16":
        o = oracle.default()
        for l in range(2):
            w13s, w2s, sw13, sw2 = host_layer(layers[l])
            xb = I.bf16_bits(xs[l])
            r = o.route(xb, I.bf16_bits(layers[l].wr), None, shape.k)
            ids = split[l][1].topk_ids.cpu().numpy()
            same = np.nonzero((ids == r["ids"]).all(axis=1))[0]
            want = o.moe_tokens(xb, same, r["ids"], r["w"], w13s, w2s, sw13, sw2, mirrored=True)
            assert_close(to_f64(split[l][0])[same], want, what=f"merge-copy layer {l}")
