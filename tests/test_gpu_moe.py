"""The whole MoE layer through the C ABI (route -> prefetch -> gather ->
G1 -> G2 -> combine) against the oracle's mirrored layer, plus the DWDP
invariant that the output does not depend on where experts live (DWDP §2):
bit-identical GPU outputs under different local/remote/redundant maps."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import GpuLayerRun, assert_close, host_layer, to_f64
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu


def _run_and_check(shape, placement, seed, chunk=1 << 20, n_copy_streams=1, tokens=None):
    build()
    lw = I.make_layer(shape, placement, seed, 0, device="cuda")
    x = I.make_tokens(shape.T, shape.H, seed).cuda()
    run = GpuLayerRun(shape, lw)
    try:
        rb, out = run.run(x, chunk_bytes=chunk, n_copy_streams=n_copy_streams)
        o = oracle.default()
        ref = o.route(I.bf16_bits(x), I.bf16_bits(lw.wr), None if lw.bias is None else lw.bias.cpu().numpy(),
                      shape.k)
        ids = rb.topk_ids.cpu().numpy()[: shape.T]
        same = (ids == ref["ids"]).all(axis=1)
        tok = np.arange(shape.T) if tokens is None else np.asarray(tokens)
        tok = tok[same[tok]]
        w13s, w2s, sw13, sw2 = host_layer(lw)
        want = o.moe_tokens(I.bf16_bits(x), tok, ref["ids"], ref["w"], w13s, w2s, sw13, sw2, mirrored=True)
        got = to_f64(out)[tok]
        assert_close(got, want, what="layer output")
        return out
    finally:
        run.close()


def test_tiny_layer():
    shape, placement = I.tiny_layer()
    _run_and_check(shape, placement, seed=0)


def test_shared_expert_ragged_tokens():
    shape = I.LayerShape(T=300, H=256, I=128, E=16, k=4, S=1)
    _run_and_check(shape, I.split_placement(16, 5, 3), seed=1)


def test_all_local_and_all_remote():
    shape = I.LayerShape(T=130, H=128, I=64, E=8, k=2, S=1)
    _run_and_check(shape, I.split_placement(8, 8, 0), seed=2)
    _run_and_check(shape, I.split_placement(8, 0, 2), seed=2)


def test_single_token_and_k_equals_e():
    _run_and_check(I.LayerShape(T=1, H=128, I=64, E=4, k=2, S=1), I.split_placement(4, 2, 1), seed=3)
    _run_and_check(I.LayerShape(T=70, H=128, I=64, E=4, k=4, S=0), I.split_placement(4, 1, 2), seed=4)


def test_wide_hidden_multi_tile():
    # H spans several n-tiles of the down GEMM and k-blocks of the gate/up GEMM
    shape = I.LayerShape(T=200, H=1024, I=256, E=8, k=2, S=1)
    _run_and_check(shape, I.split_placement(8, 3, 2), seed=5, chunk=100_000, n_copy_streams=2)


def test_output_independent_of_placement():
    """DWDP §2: any split or redundant placement gives the same bytes."""
    build()
    shape = I.LayerShape(T=257, H=256, I=128, E=12, k=3, S=1)
    x = I.make_tokens(shape.T, shape.H, 9).cuda()
    outs = []
    for placement in (I.split_placement(12, 12, 0), I.split_placement(12, 4, 2),
                      I.split_placement(12, 0, 3), I.split_placement(12, 4, 2, redundant=[5, 9, 11])):
        lw = I.make_layer(shape, placement, 9, 0, device="cuda")
        run = GpuLayerRun(shape, lw)
        try:
            _, out = run.run(x, chunk_bytes=50_000)
            outs.append(out.clone())
        finally:
            run.close()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_empty_batch():
    build()
    shape = I.LayerShape(T=0, H=128, I=64, E=4, k=2, S=0)
    lw = I.make_layer(shape, I.split_placement(4, 2, 1), 0, 0, device="cuda")
    run = GpuLayerRun(I.LayerShape(T=8, H=128, I=64, E=4, k=2, S=0), lw)
    try:
        x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
        rb, out = run.run(x)
        assert out.shape[0] == 0
        assert (rb.counts.cpu() == 0).all() and (rb.offsets.cpu() == 0).all()
    finally:
        run.close()


def test_bad_inverse_permutation_is_flagged():
    """inv_perm comes from the caller, so the scatter and the combine check
    every row it names: rows outside [0, T k) are not written or read, the
    context's device error word reports DEVICE_CHECK (no fault), tokens that
    do not use a bad row are unchanged, and the context stays usable."""
    build()
    shape, placement = I.tiny_layer()
    lw = I.make_layer(shape, placement, 0, 0, device="cuda")
    x = I.make_tokens(shape.T, shape.H, 0).cuda()
    run = GpuLayerRun(shape, lw)
    try:
        rb, clean = run.run(x)
        clean = clean.clone()
        bad = rb.inv_perm.clone()
        bad[5] = shape.T * shape.k + 100          # token 2's second slot
        bad[7] = -3                               # token 3's second slot
        rb.inv_perm.copy_(bad)
        out = torch.empty_like(clean)
        run.rt.moe(0, 0, x, rb, out)
        torch.cuda.synchronize()
        assert run.rt.device_status() == -6
        keep = [t for t in range(shape.T) if t not in (2, 3)]
        assert torch.equal(out[keep], clean[keep])
        _, again = run.run(x)                     # clean inputs: no flag, same bytes
        assert torch.equal(again, clean)
    finally:
        run.close()


@pytest.mark.parametrize("shape", [I.LayerShape(T=300, H=512, I=256, E=12, k=2, S=1),
                                   I.LayerShape(T=2048, H=7168, I=2048, E=32, k=4, S=1)],
                         ids=["small", "r1_widths"])
def test_layer_stages_bf16(shape):
    """The bf16 layer split at its intermediates (read from the workspace with
    dwdp_workspace_region): xp holds x's rows in grouped order, bit for bit;
    a = SiLU(gate) * up of those rows (and of x for the shared expert) against
    the oracle's grouped GEMM with each group's own w13; y = a W_down against
    the oracle's grouped GEMM on the GPU's own a with each group's w2; both
    at the layer's bars."""
    build()
    pl = I.split_placement(shape.E, shape.E // 3, 2)
    lw = I.make_layer(shape, pl, 21, 0, device="cuda")
    x = I.make_tokens(shape.T, shape.H, 21).cuda()
    run = GpuLayerRun(shape, lw)
    try:
        rb, out = run.run(x)
        T, k, H, I_ = shape.T, shape.k, shape.H, shape.I
        rows_r, rows_all = T * k, T * (k + shape.S)
        rt = run.rt
        xp = rt.ws_region(T, "xp").view(torch.bfloat16).reshape(rows_r, H)
        a = rt.ws_region(T, "a").view(torch.bfloat16).reshape(rows_all, I_)
        y = rt.ws_region(T, "y").view(torch.bfloat16).reshape(rows_all, H)
        perm = rb.perm[:rows_r].long()
        assert torch.equal(xp, x[perm // k]), "xp is not x in grouped order"
        offsets = rb.offsets.cpu().numpy().astype(np.int64)
        bounds = np.concatenate([offsets, [rows_all]])                    # the shared expert is the last group
        # rows checked: all of them for the small layer; at R1 widths the
        # first and last row of every group (the last one in its ragged last
        # m-tile)
        sel = []
        for g in range(shape.E + shape.S):
            lo, hi = int(bounds[g]), int(bounds[g + 1])
            rows = range(lo, hi) if shape.H <= 512 else sorted({lo, hi - 1} if hi > lo else set())
            sel.append(list(rows))
        offs_sel = np.concatenate([[0], np.cumsum([len(r) for r in sel])]).astype(np.int32)
        flat = np.array([r for rows in sel for r in rows], dtype=np.int64)
        w13s, w2s, sw13, sw2 = host_layer(lw)
        o = oracle.default()
        a_in = np.concatenate([I.bf16_bits(xp), I.bf16_bits(x)])          # routed rows, then the shared rows
        # the oracle's sums rounded once to bf16, the layer's declared rounding points
        as_bf16 = lambda v: (o.round_bf16_array(v).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        a_want = as_bf16(o.grouped_gemm(np.ascontiguousarray(a_in[flat]), offs_sel,
                                        [w13s[e] for e in range(shape.E)] + [sw13], I_, 1))
        assert_close(to_f64(a)[flat], a_want, what="gate/up output a")
        y_want = as_bf16(o.grouped_gemm(np.ascontiguousarray(I.bf16_bits(a)[flat]), offs_sel,
                                        [w2s[e] for e in range(shape.E)] + [sw2], H, 0))
        assert_close(to_f64(y)[flat], y_want, what="down output y")
    finally:
        run.close()


def test_phase_events_in_order_and_kept_on_a_rejected_call():
    """dwdp_set_phase_events: the seven events of a layer step come in the
    documented order (route start, route end, x in expert order, stage
    waited for, gate/up, down, combine), and a call with a NULL event is
    rejected without touching the events in effect."""
    import ctypes

    build()
    shape = I.LayerShape(T=300, H=512, I=256, E=12, k=2, S=1)
    pl = I.split_placement(shape.E, shape.E // 3, 2)
    lw = I.make_layer(shape, pl, 41, 0, device="cuda")
    x = I.make_tokens(shape.T, shape.H, 41).cuda()
    run = GpuLayerRun(shape, lw)
    try:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(B.DWDP_PHASE_EVENTS)]
        for e in evs:
            e.record()                    # torch creates the CUDA event on its first record
        B.dwdp_set_phase_events(run.rt.ctx, evs)
        run.run(x)
        gaps = [evs[i].elapsed_time(evs[i + 1]) for i in range(B.DWDP_PHASE_EVENTS - 1)]
        assert all(g >= 0.0 for g in gaps), gaps
        bad = (ctypes.c_void_p * B.DWDP_PHASE_EVENTS)(*[e.cuda_event for e in evs])
        bad[3] = None
        assert B.lib().dwdp_set_phase_events(run.rt.ctx, bad, B.DWDP_PHASE_EVENTS) == -1   # INVALID_ARG
        mark = torch.cuda.Event(enable_timing=True)
        mark.record()
        run.run(x)                        # the first set is still in effect: re-recorded after `mark`
        assert mark.elapsed_time(evs[0]) >= 0.0 and evs[0].elapsed_time(evs[6]) >= 0.0
        B.dwdp_set_phase_events(run.rt.ctx, None)
    finally:
        run.close()


def test_bounded_wait_gives_up_and_reports():
    """The bounded mbarrier wait every grouped-GEMM role uses, made to run out
    (dwdp_selftest_bounded_wait: a barrier phase that nothing completes):
    the kernel returns after about the limit, the host reads DEVICE_CHECK
    with bit 8, the error word is cleared, and the context then runs a layer
    as before."""
    build()
    shape = I.LayerShape(T=64, H=256, I=128, E=8, k=2, S=1)
    pl = I.split_placement(8, 4, 1)
    lw = I.make_layer(shape, pl, 43, 0, device="cuda")
    x = I.make_tokens(shape.T, shape.H, 43).cuda()
    run = GpuLayerRun(shape, lw)
    try:
        _, before = run.run(x)
        before = before.clone()
        with pytest.raises(B.DwdpError):
            B.dwdp_selftest_bounded_wait(run.rt.ctx, 0)            # limit outside [1, 1e6] us
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream = torch.cuda.current_stream()
        start.record(stream)
        B.dwdp_selftest_bounded_wait(run.rt.ctx, 20_000, stream)  # 20 ms
        end.record(stream)
        torch.cuda.synchronize()
        ms = start.elapsed_time(end)
        assert 19.0 <= ms < 1000.0, f"the wait took {ms} ms"
        assert run.rt.device_status() == -6                         # DEVICE_CHECK
        assert "0x100" in B.dwdp_last_error(run.rt.ctx)
        assert run.rt.device_status() == 0                          # cleared by the read
        _, after = run.run(x)
        assert torch.equal(after, before)
    finally:
        run.close()


def test_layer_at_the_limits():
    """1024 experts (the ABI's maximum) with top-32 (its maximum k) and the
    shared expert: 1025 groups in the GEMMs' tile tables, the generic
    scatter and combine paths, half the experts staged from two pools."""
    _run_and_check(I.LayerShape(T=48, H=128, I=64, E=1024, k=32, S=1), I.split_placement(1024, 512, 2), seed=44)
