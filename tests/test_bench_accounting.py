"""The benchmark's algorithmic work per layer, against the figures the
hot-path scope states for the 8192-token R1 layer (T = 8192, H = 7168,
I = 2048, E = 256 routed experts all active, top-8, one shared expert,
192 experts staged): 6.49 TFLOP of expert FLOPs plus 3.0e10 for the
router, 4.33e12 FLOPs and 16.45 GB for the gate/up GEMM (w13 of 257
experts, 58.72 MB each, plus the rows in and a out), 22.64 GB of expert
weights read once (88.08 MB per expert), and the prefetch moving 16.91 GB
read plus 16.91 GB written.  The roofline fractions the bench prints
divide these by measured times, so a wrong term would misstate them."""
import pytest

import bench

T, H, I, E, K, S, R = 8192, 7168, 2048, 256, 8, 1, 192
MB = 1e6


def test_layer_and_gate_up_flops():
    router = 2 * T * H * E
    assert router == pytest.approx(3.0e10, rel=0.01)
    assert bench.layer_flops(T, H, I, E, K, S) - router == pytest.approx(6.49e12, rel=1e-3)
    assert bench.g1_flops(T, H, I, K, S) == pytest.approx(4.33e12, rel=1e-3)


def test_gate_up_bytes():
    w13 = 2 * I * H * 2                      # one expert's gate/up weights, bf16
    assert w13 / MB == pytest.approx(58.72, rel=1e-3)
    assert bench.g1_bytes(T, H, I, E, K, S) / 1e9 == pytest.approx(16.45, rel=2e-3)
    # E4M3 weights and rows: one byte per element, a still written in bf16
    assert bench.g1_bytes(T, H, I, E, K, S, wb=1) == (E + S) * w13 // 2 + T * (K + S) * H + T * (K + S) * I * 2


def test_step_bytes_terms():
    expert = 3 * H * I * 2
    assert expert / MB == pytest.approx(88.08, rel=1e-3)
    weights = (E + S) * expert
    assert weights / 1e9 == pytest.approx(22.64, rel=1e-3)
    prefetch = 2 * R * expert                # read + written on this GPU's memory
    assert prefetch / 2 / 1e9 == pytest.approx(16.91, rel=1e-3)
    xp, a, y, x_out = 2 * T * K * H * 2, 2 * T * (K + S) * I * 2, 2 * T * (K + S) * H * 2, 2 * T * H * 2
    assert bench.step_bytes(T, H, I, E, K, S, R) == weights + xp + a + y + x_out + prefetch
    # with no staged experts the copy term vanishes
    assert bench.step_bytes(T, H, I, E, K, S, 0) == weights + xp + a + y + x_out


def test_kernels_per_step_match_the_launch_lists():
    # the ncu launch lists of one step show 9 (bf16), 10 (E4M3) and 10 (NVFP4)
    # of this library's kernels
    assert bench.kernels_per_layer("bf16") == 9
    assert bench.kernels_per_layer("fp8") == 10
    assert bench.kernels_per_layer("nvfp4") == 10


PEAKS = {"hbm_gbs": 6792.7, "bf16_tflops": 1928.3, "bf16_tflops_sustained": 1712.7}


def test_roofline_bound_follows_the_ridge():
    """The gate/up GEMM at 8192 tokens does 4.33e12 FLOP over 16.45 GB of
    algorithmic bytes: 263 FLOP/B, below the burst ridge 1928.3 TFLOP/s /
    6792.7 GB/s = 284 FLOP/B, so it is HBM-bound and its fraction is
    bytes / time / HBM peak."""
    tc, hbm, note = bench.roofline_peaks(PEAKS, "measured", "bf16")
    assert tc == 1928.3 and hbm == 6792.7 and "burst" in note
    g1, g1b = bench.g1_flops(T, H, I, K, S), bench.g1_bytes(T, H, I, E, K, S)
    r = bench.roofline_entry("g1", g1, g1b, 5.8134e-3, tc, hbm, note, "hbm")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["ridge"] == pytest.approx(283.9, abs=0.1)
    assert r["achieved"] == pytest.approx(g1b / 5.8134e-3 / 1e9, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / 6792.7, abs=1e-4)
    assert 0.41 < r["frac"] < 0.43
    # twice the FLOPs per byte crosses the ridge: tensor-bound, FLOP/s against the tensor peak
    r2 = bench.roofline_entry("g1", 2 * g1, g1b, 5.8134e-3, tc, hbm, note, "hbm")
    assert r2["bound"] == "tensor" and r2["frac"] == pytest.approx(2 * g1 / 5.8134e-3 / 1e12 / tc, abs=1e-4)


def test_low_precision_peaks_scale_the_measured_bf16_burst():
    assert bench.roofline_peaks(PEAKS, "measured", "fp8")[0] == pytest.approx(2 * 1928.3)
    assert bench.roofline_peaks(PEAKS, "measured", "nvfp4")[0] == pytest.approx(6 * 1928.3)


def test_variant_names():
    assert bench.parse_variant("r1_moe_layer_8k", "nvfp4") == ("r1_moe_layer_8k", "nvfp4", False)
    assert bench.parse_variant("r1_moe_layer_8k", "nvfp4_wide") == ("r1_moe_layer_8k", "nvfp4", True)
    assert bench.parse_variant("r1_moe_layer_8k", "r1_zipf_16k") == ("r1_zipf_16k", "bf16", False)
    assert bench.parse_variant("r1_moe_layer_8k", "r1_pipeline_4layer:nvfp4") == ("r1_pipeline_4layer", "nvfp4", False)
    with pytest.raises(ValueError):
        bench.parse_variant("r1_moe_layer_8k", "int3")
    args = bench.parse([])
    for v in args.variants.split(","):
        bench.parse_variant(args.workload, v)       # every default variant parses


def test_traffic_record_is_the_full_size_capture():
    """The committed DRAM record of the gate/up GEMM is a capture of the
    8192-token launch itself: scaled to that launch's algorithmic bytes it
    gives back the captured read + write bytes, and it is keyed to the
    kernel source it was taken on (otherwise the bench reports no traffic)."""
    import json
    import os
    path = os.path.join(bench.ROOT, "profiles", "gate_up_gemm_traffic_r1_moe_layer_8k.json")
    rec = json.load(open(path))
    g1b = bench.g1_bytes(T, H, I, E, K, S)
    assert rec["algorithmic_bytes"] == g1b
    got = bench.measured_traffic(os.path.join(bench.ROOT, "moe_expert_grouped_split_gb300", "csrc", "gemm.cu"), g1b)
    assert got is not None, "gemm.cu changed since the capture"
    assert got == pytest.approx(rec["dram_bytes_read"] + rec["dram_bytes_write"], rel=1e-4)
    assert 1.0 <= got / g1b < 1.1


def test_both_arms_report_the_same_workload_config():
    """The reference arm (the oracle) and the GPU arm build their config from
    one function, so the two lines name the same workload, shapes,
    placement and prefetch settings."""
    args = bench.parse([])
    spec = bench.WORKLOADS[args.workload](group=args.group)
    cfg = bench.workload_config(args, spec.shape, spec.placement, 2)
    assert cfg["workload"] == "r1_moe_layer_8k" and cfg["T"] == T and cfg["E"] == E and cfg["k"] == K
    assert (cfg["local_experts"], cfg["remote_experts"], cfg["peer_pools"]) == (64, 192, 3)
    assert cfg["chunk_mb"] == 64.0 and cfg["expert_weights"] == "bf16" and cfg["layers"] == 2
    assert bench.default_chunk_mb("r1_moe_layer_8k", "nvfp4") == 32.0
    assert bench.default_chunk_mb("r1_pipeline_4layer", "bf16") == 16.0
    assert bench.default_copy_streams("r1_moe_layer_8k", "bf16") == 1
    assert bench.default_copy_streams("r1_moe_layer_8k", "nvfp4") == 2
    assert bench.default_copy_streams("r1_moe_layer_256", "bf16") == 2
    assert bench.default_copy_streams("r1_pipeline_4layer", "bf16") == 2
    src = open(bench.__file__).read()
    assert src.count("\"config\": workload_config(args,") == 2     # the GPU arm's line and the reference arm's
