"""The timing model of DWDP section 3 (and the news summary): with the next
layer's prefetch overlapped, a layer takes about max(T_compute, T_prefetch)
rather than T_compute + T_prefetch.  Checked on the benchmark's machinery
(R1 widths, 2048 tokens, 32 experts top-4 + shared, 8 resident, 24 staged
from three peer pools, 32 MB slices): the overlapped step is never faster
than the larger of the compute-only step and the copy alone (it cannot beat
either), and is faster than running them one after the other.  On one GPU
the copy's reads and writes share HBM with the GEMMs, so the overlapped
step sits between the two bounds rather than on the lower one."""
import pytest

import bench
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wdtype", ["bf16", "nvfp4"])
def test_overlapped_step_between_max_and_sum(wdtype):
    build()
    shape = I.LayerShape(T=2048, H=7168, I=2048, E=32, k=4, S=1)
    spec = bench.Spec(shape, I.split_placement(32, 8, 3), 0.02, None)
    wl = bench.Workload(spec, 32 << 20, 1, wdtype=wdtype)
    try:
        K, W = 10, 3
        ms_total, _ = bench.run_overlapped(wl, K, W, None)
        over = ms_total / K
        comp = bench.run_compute_only(wl, K)
        copy = bench.run_copy_only(wl, K)
        print(f"\n{wdtype}: overlapped {over:.3f} ms, compute-only {comp:.3f} ms, copy-only {copy:.3f} ms, "
              f"max {max(comp, copy):.3f}, sum {comp + copy:.3f}")
        assert over >= 0.97 * max(comp, copy), "faster than the compute or the copy alone: a step was skipped"
        assert over < comp + copy, "no overlap: the copy and the compute ran one after the other"
    finally:
        wl.rt.close()
