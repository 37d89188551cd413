"""Benchmark of the DWDP single-rank hot path on synthetic DeepSeek-R1-shaped
MoE layers.

One step = one MoE layer for one batch of T tokens, the way a DWDP rank runs
it (DWDP §2): route + gather + gate/up GEMM + down GEMM + combine on the
compute stream, while the next layer's 192 non-resident experts are copied
from three emulated peer pools into the other stage buffer in fixed-size
slices issued round-robin (DWDP §4.3.2) on a copy stream.  Two distinct
layers alternate, so every step's weights (22.6 GB read by the GEMMs) and
copies (16.9 GB) are far larger than L2: no flush is needed between steps.

Prints one JSON line.  ``value`` = tokens/s over the timed steps with inputs
resident in HBM; ``e2e`` = the same with each step's tokens copied in from
pinned host memory and the layer output copied back, inside the timed
region.  ``roofline`` describes the dominant kernel (the gate/up grouped GEMM)
timed with CUDA events the library records around it on its own stream;
``step_hbm`` relates the step's algorithmic HBM bytes to the measured HBM
peak.  ``cpu_baseline`` times the CPU oracle on a bounded token sample.

Workloads (--workload): r1_moe_layer_8k (default), r1_zipf_16k (Zipf-skewed
routing, 16 hottest experts replicated), r1_moe_layer_256 (decode-like;
--chunk-sweep reports exposed copy time per chunk size), r1_pipeline_4layer
(4 layers per step with attention-sized GEMM stand-ins, T per step uniform in
[6554, 8192], 16 steps) and r1_small_profile (for profiler captures).

--impl reference runs the same metric with the CPU oracle on host cores.

One GPU only: the DWDP rank's hot path runs on one GPU (its peers are
emulated by device pools), and its grouped GEMM shares weight tiles between
the two CTAs of a cluster with multicast loads, which are kept to one-GPU
runs.  With --gpus > 1 or WORLD_SIZE > 1 the benchmark prints one JSON line
saying so ("unavailable") and exits before building or loading the library.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time
from collections import namedtuple

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s & TFLOP/s at 8K tokens, prefetch overlapped; % of TC peak"
UNIT = "tokens/s"

Spec = namedtuple("Spec", "shape placement router_std bias")


def _r1(T, zipf=False, router_std=0.02):
    def make(group=4):
        """group: DWDP group size N: E / N experts resident, the rest spread
        over the N - 1 peers (N = 4: 64 local + 3 x 64, the default)."""
        from moe_expert_grouped_split_gb300 import inputs as I
        shape, _ = I.r1_layer(T)
        n_local = shape.E // group
        bias = None
        redundant = ()
        if zipf:
            bias = I.zipf_bias(shape.E, 1.2, I.seed_for(0, "zipf"))
            redundant = I.hottest_experts(bias, 16)
        placement = I.split_placement(shape.E, n_local, group - 1, redundant=redundant)
        return Spec(shape, placement, router_std, bias)
    return make


def _r1_small(group=4):
    """R1 layer widths (H=7168, I=2048) with 16 routed experts, top-4, one
    shared expert and 1024 tokens (256 rows per expert, as at 8K tokens with
    256 experts and top-8): a few GB, for profiler captures."""
    from moe_expert_grouped_split_gb300 import inputs as I
    return Spec(I.LayerShape(T=1024, H=7168, I=2048, E=16, k=4, S=1), I.split_placement(16, 4, 3), 0.02, None)


WORKLOADS = {
    "r1_moe_layer_8k": _r1(8192),
    "r1_zipf_16k": _r1(16384, zipf=True),
    "r1_moe_layer_256": _r1(256, router_std=1.0 / math.sqrt(7168)),
    "r1_pipeline_4layer": _r1(8192),
    "r1_small_profile": _r1_small,
}


def default_chunk_mb(workload: str, wdtype: str) -> float:
    """Prefetch slice size: 16 MB for the 4-layer pipeline (its workload's
    own figure); otherwise the fastest measured on one GB300 (same-box A/B,
    two to three runs each): 64 MB for bf16 and E4M3 (against 32 MB: C1
    bf16 -1.5%, E4M3 -2%, the 256-token layer -4.8%; 128 MB no better), 32
    MB for NVFP4 (0.3% ahead of 64 MB, with two copy chains)."""
    if workload == "r1_pipeline_4layer":
        return 16.0
    return 32.0 if wdtype == "nvfp4" else 64.0


def default_copy_streams(workload: str, wdtype: str) -> int:
    """Copy chains of the prefetch graph: two for NVFP4 layers, for the
    copy-bound 256-token layer and for the 4-layer pipeline, whose 16 MB
    slices make the copy the longer side (same-box A/B: NVFP4 C1 -1.5%, 256
    tokens bf16 -1.7%, pipeline bf16 -5%), one otherwise (two slow the GEMMs
    beside them more than they speed the copy: C1 bf16 +0.8%, E4M3 +0.6%)."""
    if wdtype == "nvfp4" or workload in ("r1_moe_layer_256", "r1_pipeline_4layer"):
        return 2
    return 1


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="r1_moe_layer_8k", choices=sorted(WORKLOADS))
    p.add_argument("--chunk-mb", type=float, default=None,
                   help="prefetch slice size in MB (default 16 for the 4-layer pipeline, as that workload "
                        "specifies; else the fastest measured: 64 for bf16 and E4M3, 32 for NVFP4)")
    p.add_argument("--copy-streams", type=int, default=None,
                   help="copy chains the prefetch graph is split into, one per peer pool modulo this count "
                        "(default 2 for NVFP4, the 256-token layer and the 4-layer pipeline, else 1: the "
                        "fastest measured)")
    p.add_argument("--stages", type=int, default=2,
                   help="staging buffers (2: the pages' double buffering; 3: the copy of layer l+2 may start "
                        "while layer l computes)")
    p.add_argument("--prefetch-start", choices=["layer", "route", "gate_up"], default="route",
                   help="when a layer's copy may start, besides its stage being free: with the current layer, "
                        "once its routing is done, or once its gate/up GEMM is done (best with --stages 3)")
    p.add_argument("--group", type=int, default=4,
                   help="DWDP group size N: E/N experts resident, the rest staged from N-1 peer pools")
    p.add_argument("--dtype", default="bf16", choices=["bf16", "fp8", "nvfp4"],
                   help="expert weight type (fp8: E4M3 weights and activations; nvfp4: E2M1 codes with E4M3 "
                        "scales per 16-element block; next-row variants)")
    p.add_argument("--chunk-sweep", default="", help="comma-separated chunk sizes in MB (exposed copy per size)")
    p.add_argument("--merge-copy", action="store_true",
                   help="also time the merge-copy baseline (one contiguous weight buffer per layer); on by "
                        "default for the 8K-token layer")
    p.add_argument("--no-merge-copy", action="store_true", help="skip the merge-copy baseline")
    p.add_argument("--variants", default=None,
                   help="comma-separated further measurements after the main line, each summarised under "
                        "'variants': a weight type for the same workload (fp8, nvfp4, nvfp4_wide = nvfp4 with "
                        "--wide-epilogue) or another workload, optionally with a weight type "
                        "(r1_zipf_16k:nvfp4).  Default for the 8K-token bf16 layer: fp8, nvfp4, nvfp4_wide, the "
                        "Zipf 16K layer and the 256-token layer (bf16 with its chunk sweep, fp8, nvfp4) and the "
                        "4-layer pipeline (bf16, nvfp4)")
    p.add_argument("--peer-pools", default="device", choices=["device", "host"],
                   help="where the emulated peers' pools live (host: pinned host memory, copies over the "
                        "host link, so only their writes use this GPU's HBM)")
    p.add_argument("--wide-epilogue", action="store_true",
                   help="NVFP4: the gate/up GEMM drains its accumulator with eight warps (faster alone, but it "
                        "starves the overlapped copy on one GPU)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extras", action="store_true", help="skip compute-only / copy-only / e2e legs")
    p.add_argument("--duration-study", type=float, default=0.0,
                   help="also run the compute-only and the overlapped step back to back for this many seconds "
                        "each, sampling SM clock and power (long-duration overlap, the analogue of the pages' "
                        "appendix A.2)")
    args = p.parse_args(argv)
    if args.chunk_mb is None:
        args.chunk_mb = default_chunk_mb(args.workload, args.dtype)
    args.copy_streams_given = args.copy_streams is not None
    if args.copy_streams is None:
        args.copy_streams = default_copy_streams(args.workload, args.dtype)
    if args.workload == "r1_moe_layer_8k" and not args.no_extras and args.group == 4:
        args.merge_copy = True
    if args.no_merge_copy:
        args.merge_copy = False
    if args.variants is None:
        default = args.workload == "r1_moe_layer_8k" and args.dtype == "bf16" and not args.no_extras
        args.variants = ("fp8,nvfp4,nvfp4_wide,r1_zipf_16k,r1_zipf_16k:fp8,r1_zipf_16k:nvfp4,"
                         "r1_zipf_16k:nvfp4_wide,r1_moe_layer_256,"
                         "r1_moe_layer_256:fp8,r1_moe_layer_256:nvfp4,r1_pipeline_4layer,r1_pipeline_4layer:nvfp4"
                         ) if default and args.group == 4 else ""
    return args


# ------------------------------------------------------------- helpers ----
def layer_flops(T, H, I, E, k, S):
    """Algorithmic FLOPs of one layer: router 2*T*H*E, experts T*(k+S)*6*H*I."""
    return 2 * T * H * E + T * (k + S) * 6 * H * I


def g1_flops(T, H, I, k, S):
    """Gate/up grouped GEMM: 2 * (rows) * H * 2I with rows = T*(k+S)."""
    return 4 * T * (k + S) * H * I


def g1_bytes(T, H, I, E_active, k, S, wb=2):
    """Gate/up grouped GEMM, algorithmic HBM bytes: every active expert's
    w13 once (2I*H elements of wb bytes), the gathered rows and x once (same
    element size), a written once (bf16)."""
    return int((E_active + S) * 2 * I * H * wb + T * (k + S) * H * wb + T * (k + S) * I * 2)


def step_bytes(T, H, I, E_active, k, S, R, wb=2):
    """Algorithmic HBM bytes of one overlapped step: weights once
    ((E_active+S)*3*H*I elements of wb bytes), xp / a / y written and read
    once, x read and out written, and the prefetch of R experts (read +
    write, both on this GPU's HBM under the one-GPU emulation).  With E4M3
    weights (wb = 1) the GEMM operands xp and a are E4M3 too, plus x's and
    a's quantization passes (codes written and read once)."""
    b = ((E_active + S) * 3 * H * I * wb + 2 * T * k * H * wb + 2 * T * (k + S) * I * 2
         + 2 * T * (k + S) * H * 2 + 2 * T * H * 2 + 2 * R * 3 * H * I * wb)
    if wb < 2:   # quantized: x's codes (shared expert) and a's codes, each written and read once
        b += 2 * T * H * wb + 2 * T * (k + S) * I * wb
    return int(b)


def kernels_per_layer(wdtype: str) -> int:
    """This library's kernel launches per layer step: route = router GEMM,
    top-k and the three grouping kernels; the layer = (quantizers,) scatter
    into expert order (fused into the E4M3 and NVFP4 x quantizers), the two
    GEMMs and the combine.  (The ncu launch lists in profiles/ show the same
    counts.)"""
    layer = {"bf16": 4, "fp8": 5, "nvfp4": 5}[wdtype]
    return 5 + layer


# Bytes per weight (and quantized activation) element: NVFP4 is half a byte
# of E2M1 code plus one E4M3 scale per 16 elements.
WEIGHT_BYTES = {"bf16": 2, "fp8": 1, "nvfp4": 9 / 16}


def measured_traffic(kernel_file: str, algorithmic_bytes: int):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch of the gate/up
    GEMM: the committed ncu record's measured-to-algorithmic ratio (a 1-pass
    capture of the 8192-token launch) times this launch's algorithmic bytes,
    i.e. the captured bytes; None when the kernel source has changed since
    the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "gate_up_gemm_traffic_r1_moe_layer_8k.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    with open(kernel_file, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    if rec.get("gemm_cu_sha256") != sha:
        return None
    return int(round(rec["traffic_over_algorithmic"] * algorithmic_bytes))


class ClockSampler:
    """nvidia-smi clocks sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.25)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        power_sorted = sorted(power)
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None,
                "power_w_median": power_sorted[len(power_sorted) // 2] if power_sorted else None}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# nominal dense tensor-core throughput of each operand type relative to bf16
# (2.25 / 4.5 / 13.5 PFLOP/s for bf16 / FP8 / FP4 on GB300)
TC_RATIO = {"bf16": 1.0, "fp8": 2.0, "nvfp4": 6.0}


def roofline_peaks(peaks: dict, src: str, wdtype: str):
    """(tensor peak TFLOP/s, HBM peak GB/s, note) for the benchmark's GEMMs.
    The burst bf16 figure applies: every timed kernel runs inside a timed
    region of well under a second at full SM clock, while the sustained
    figure was taken over seconds under the power cap at a lower clock.
    FP8 / FP4 take the measured bf16 burst peak times the nominal ratio."""
    r = TC_RATIO[wdtype]
    tc = peaks["bf16_tflops"] * r
    note = f"{src} bf16_tflops (burst)" + (f" x {r:g} (nominal dense {wdtype} / bf16 ratio)" if r != 1 else "")
    return tc, peaks["hbm_gbs"], note


def roofline_entry(kernel: str, flops: float, nbytes: float, seconds: float, tc_peak: float, hbm_peak: float,
                   tc_note: str, hbm_note: str) -> dict:
    """The kernel against the roof its arithmetic intensity puts it under:
    intensity (FLOP per algorithmic HBM byte) at or above the ridge
    tc_peak / hbm_peak -> tensor-bound, achieved TFLOP/s against tc_peak;
    below it -> HBM-bound, achieved algorithmic GB/s against hbm_peak."""
    ai = flops / nbytes
    ridge = tc_peak * 1e12 / (hbm_peak * 1e9)
    if ai >= ridge:
        ach = flops / seconds / 1e12
        return {"kernel": kernel, "bound": "tensor", "achieved": round(ach, 1), "peak": tc_peak, "unit": "TFLOP/s",
                "frac": round(ach / tc_peak, 4), "peak_source": tc_note, "arithmetic_intensity": round(ai, 1),
                "ridge": round(ridge, 1)}
    ach = nbytes / seconds / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(ach / hbm_peak, 4), "peak_source": hbm_note, "arithmetic_intensity": round(ai, 1),
            "ridge": round(ridge, 1)}


def whole_job_rate(units_per_step: int, steps: int, ms_total: float) -> float:
    """Units processed per second over the timed steps."""
    return steps * units_per_step / (ms_total / 1e3)


def single_gpu_refusal(args, world: int):
    """The JSON line printed instead of a measurement when more than one GPU
    is asked for, or None for a one-GPU run."""
    if world <= 1 and args.gpus <= 1:
        return None
    return {"metric": METRIC, "unit": UNIT, "n_gpus": max(world, args.gpus), "higher_is_better": True,
            "unavailable": "single-GPU path: one DWDP rank on one GPU (peers emulated by device pools); its "
                           "grouped GEMM's cluster-multicast loads are kept to one-GPU runs"}


PHASES = ["route", "gather", "wait_stage", "gate_up_gemm", "down_gemm", "combine"]


# -------------------------------------------------------- our arm ----------
class Workload:
    """n_layers R1-shaped layers with their pools, a Runtime, route buffers
    and per-layer token batches, all resident in HBM."""

    def __init__(self, spec: Spec, chunk_bytes, n_copy_streams, n_layers=2, base_seed=0, wdtype="bf16",
                 peer_pools="device", prefetch_start="route", n_stages=2, flags=0):
        import torch

        from moe_expert_grouped_split_gb300 import binding as B
        from moe_expert_grouped_split_gb300 import inputs as I

        self.B, self.I, self.torch = B, I, torch
        self.spec = spec
        self.wdtype = wdtype
        self.shape, self.placement = spec.shape, spec.placement
        sh = self.shape
        self.n_layers = n_layers
        make = {"bf16": I.make_layer, "fp8": I.make_layer_fp8, "nvfp4": I.make_layer_nvfp4}[wdtype]
        self.layers = [make(sh, self.placement, base_seed, l, device="cuda", router_std=spec.router_std,
                            bias=spec.bias) for l in range(n_layers)]
        self.peer_pools = peer_pools
        if peer_pools == "host":
            # generated on the GPU, then moved to pinned host memory
            for lw in self.layers:
                for pools in (lw.peer_w13, lw.peer_w2):
                    for i, t in enumerate(pools):
                        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                        h.copy_(t)
                        pools[i] = h
            torch.cuda.empty_cache()
        if n_stages < 2:
            raise ValueError("the benchmark overlaps the copy: it needs at least 2 stages")
        self.n_stages = n_stages
        self.rt = B.Runtime(sh.H, sh.I, sh.E, sh.k, sh.S, sh.T, n_layers, self.placement.n_remote(),
                            weight_dtype={"bf16": B.DTYPE_BF16, "fp8": B.DTYPE_E4M3, "nvfp4": B.DTYPE_NVFP4}[wdtype],
                            n_stages=n_stages, flags=flags)
        for l, lw in enumerate(self.layers):
            self.rt.set_layer(l, lw)
        self.x = [I.make_tokens(sh.T, sh.H, base_seed, step=s, device="cuda") for s in range(n_layers)]
        self.rb = B.RouteBuffers(sh.T, sh.E, sh.k)
        self.out = torch.empty((sh.T, sh.H), dtype=torch.bfloat16, device="cuda")
        self.compute = torch.cuda.Stream()
        self.copies = [torch.cuda.Stream() for _ in range(n_copy_streams)]
        self.chunk = int(chunk_bytes)
        self.issue_s = []
        # "route": the copy streams wait for the current layer's routing, so
        # the small latency-bound routing kernels run without the copy;
        # "gate_up": for its gate/up GEMM (the library's phase event 4), so
        # the copy overlaps the down GEMM, the combine and the next layer's
        # routing first
        self.prefetch_start = prefetch_start
        self.routed = torch.cuda.Event()
        self.gate_ev = [torch.cuda.Event() for _ in range(B.DWDP_PHASE_EVENTS)]
        for e in self.gate_ev:       # torch creates the CUDA event on its first record
            e.record()
        self.gated_by = None      # the phase events of the last layer step
        self._phases_set = False

    def layer_step(self, layer, stage, T=None, x=None, out=None):
        T = self.shape.T if T is None else T
        x = (self.x[layer] if x is None else x)[:T]
        out = (self.out if out is None else out)[:T]
        with self.torch.cuda.stream(self.compute):
            self.rt.route(x, self.layers[layer].wr, self.layers[layer].bias, self.rb, self.compute)
            self.routed.record(self.compute)
            self.rt.moe(layer, stage, x, self.rb, out, self.compute)

    def set_phases(self, events):
        """Phase events for the following layer steps (None: none)."""
        if events is not None or self._phases_set:
            self.B.dwdp_set_phase_events(self.rt.ctx, events)
        self._phases_set = events is not None

    def prefetch(self, layer, stage):
        t0 = time.perf_counter()
        if self.prefetch_start == "route":
            for c in self.copies:
                c.wait_event(self.routed)
        elif self.prefetch_start == "gate_up" and self.gated_by is not None:
            for c in self.copies:
                c.wait_event(self.gated_by[4])
        self.rt.prefetch(layer, stage, self.chunk, self.copies)
        self.issue_s.append(time.perf_counter() - t0)

    def step(self, i, prefetch_next=True, x=None, out=None, phases=None):
        """Step i of the layer alternation: layer i % n_layers from stage
        i % S, then the prefetch of step i + S - 1's layer into its stage
        (S = 2: the next layer into the other stage).  Without prefetch_next
        every layer is already staged at stage = layer.  phases: the timing
        events of this step, or None."""
        l = i % self.n_layers
        gate = self.prefetch_start == "gate_up" and prefetch_next
        ev = phases if phases is not None else (self.gate_ev if gate else None)
        self.set_phases(ev)
        self.gated_by = ev
        if not prefetch_next:
            self.layer_step(l, l, x=x, out=out)
            return
        S = self.n_stages
        self.layer_step(l, i % S, x=x, out=out)
        j = i + S - 1
        self.prefetch(j % self.n_layers, j % S)

    def prologue(self):
        """The copies of steps 0 .. S-2, before step 0."""
        for j in range(self.n_stages - 1):
            self.prefetch(j % self.n_layers, j)

    def sync(self):
        self.torch.cuda.synchronize()


def _events(torch, n):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:          # create the underlying CUDA events now
        e.record()
    torch.cuda.synchronize()
    return evs


def _phase_avg(phases, K):
    ph = [[phases[i][j].elapsed_time(phases[i][j + 1]) for j in range(6)] for i in range(K)]
    return {n_: round(sum(p[j] for p in ph) / K, 4) for j, n_ in enumerate(PHASES)}


def run_overlapped(wl, K, W, phases, clocks_index=0):
    """K timed steps (after W warm-up steps) of the two-layer alternation with
    the next layer's prefetch overlapped."""
    torch, B = wl.torch, wl.B
    wl.prologue()
    n = 0
    for i in range(W):
        wl.step(n)
        n += 1
    wl.sync()
    start, stop = _events(torch, 2)
    with ClockSampler(clocks_index) as clk:
        start.record(wl.compute)
        for c in wl.copies:
            c.wait_stream(wl.compute)
        for i in range(K):
            wl.step(n, phases=phases[i] if phases is not None else None)
            n += 1
        wl.set_phases(None)
        for c in wl.copies:
            wl.compute.wait_stream(c)
        stop.record(wl.compute)
        stop.synchronize()
    assert wl.rt.device_status() == 0
    ms_total = start.elapsed_time(stop)
    return ms_total, clk.summary()


def run_compute_only(wl, K, phases=None):
    """K steps with every expert already staged and no copies (the
    all-resident reference for the exposed-prefetch figure)."""
    torch, B = wl.torch, wl.B
    wl.sync()
    for l in (0, 1):
        wl.prefetch(l, l)
    wl.sync()
    for i in range(2):
        wl.step(i, prefetch_next=False)
    a, b = _events(torch, 2)
    a.record(wl.compute)
    for i in range(K):
        wl.step(i, prefetch_next=False, phases=phases[i] if phases is not None else None)
    wl.set_phases(None)
    b.record(wl.compute)
    b.synchronize()
    return a.elapsed_time(b) / K


def run_duration(wl, seconds: float, overlapped: bool, K: int = 20):
    """Steps back to back for about `seconds` (batches of 50), the last K of
    them with phase events; clocks and power sampled throughout."""
    torch = wl.torch
    wl.sync()
    if overlapped:
        wl.prologue()
    else:
        for l in (0, 1):
            wl.prefetch(l, l)
    wl.sync()
    phases = [_events(torch, 7) for _ in range(K)]
    n, t0 = 0, time.perf_counter()
    a, b = _events(torch, 2)
    with ClockSampler(0) as clk:
        a.record(wl.compute)
        for c in wl.copies:
            c.wait_stream(wl.compute)
        while time.perf_counter() - t0 < seconds:
            for _ in range(50):
                wl.step(n, prefetch_next=overlapped)
                n += 1
            wl.compute.synchronize()
        for i in range(K):
            wl.step(n, prefetch_next=overlapped, phases=phases[i])
            n += 1
        wl.set_phases(None)
        for c in wl.copies:
            wl.compute.wait_stream(c)
        b.record(wl.compute)
        b.synchronize()
    assert wl.rt.device_status() == 0
    return {"steps": n, "seconds": round(a.elapsed_time(b) / 1e3, 2), "ms_per_step": round(a.elapsed_time(b) / n, 4),
            "last_steps_phase_ms": _phase_avg(phases, K), "clocks": clk.summary()}


def run_copy_only(wl, K):
    torch = wl.torch
    wl.sync()
    a, b = _events(torch, 2)
    a.record(wl.copies[0])
    for c in wl.copies[1:]:
        c.wait_stream(wl.copies[0])
    for i in range(K):
        wl.prefetch(i % 2, i % 2)
    b.record(wl.copies[0])
    b.synchronize()
    return a.elapsed_time(b) / K


def run_e2e(wl, K):
    """The metric through the public API with host buffers: each step copies
    its tokens in from pinned host memory and its output back to pinned host
    memory, inside the timed region.  The copies run on their own streams,
    double-buffered, so step i+1's tokens arrive and step i-1's output
    leaves while step i computes."""
    torch = wl.torch
    sh = wl.shape
    T = sh.T
    xh = [x.cpu().pin_memory() for x in wl.x]
    oh = [torch.empty((T, sh.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(wl.x[0]) for _ in range(2)]
    od = [torch.empty_like(wl.out) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    x_ready, x_free, o_ready, o_free = ([torch.cuda.Event() for _ in range(2)] for _ in range(4))

    def step(i):
        b = i % 2
        h2d.wait_event(x_free[b])                 # step i-2 has finished reading xd[b]
        with torch.cuda.stream(h2d):
            xd[b].copy_(xh[i % 2], non_blocking=True)
        x_ready[b].record(h2d)
        wl.compute.wait_event(x_ready[b])
        wl.compute.wait_event(o_free[b])          # step i-2's output has left od[b]
        wl.step(i, x=xd[b], out=od[b])
        x_free[b].record(wl.compute)
        o_ready[b].record(wl.compute)
        d2h.wait_event(o_ready[b])
        with torch.cuda.stream(d2h):
            oh[b].copy_(od[b], non_blocking=True)
        o_free[b].record(d2h)

    wl.sync()
    wl.prologue()
    for i in range(2):
        step(i)
    wl.sync()
    a, b = _events(torch, 2)
    a.record(wl.compute)
    for s_ in wl.copies + [h2d, d2h]:
        s_.wait_stream(wl.compute)
    for i in range(2, 2 + K):
        step(i)
    for s_ in wl.copies + [h2d, d2h]:
        wl.compute.wait_stream(s_)
    b.record(wl.compute)
    b.synchronize()
    assert wl.rt.device_status() == 0
    e2e_ms = a.elapsed_time(b)
    return {"value": round(whole_job_rate(T, K, e2e_ms), 1), "unit": UNIT,
            "h2d_bytes_per_step": T * sh.H * 2, "d2h_bytes_per_step": T * sh.H * 2}


def workload_config(args, sh, placement, n_layers) -> dict:
    """The JSON line's config: the workload, its shapes and placement and
    the prefetch settings (the reference arm reports the same keys)."""
    wbytes = WEIGHT_BYTES[args.dtype]
    return {"workload": args.workload, "T": sh.T, "H": sh.H, "I": sh.I, "E": sh.E, "k": sh.k,
            "shared": sh.S, "local_experts": int((placement.local_slot >= 0).sum()),
            "remote_experts": placement.n_remote(), "peer_pools": placement.n_peers,
            "chunk_mb": args.chunk_mb, "copy_streams": args.copy_streams, "expert_weights": args.dtype,
            "prefetch_start": args.prefetch_start, "stages": args.stages,
            "wide_epilogue": bool(args.wide_epilogue),
            "peer_pool_memory": args.peer_pools,
            "layers": n_layers,
            "dwdp_group": args.group,
            "l2": "inputs larger than L2 ({:.1f} GB of expert weights + {:.1f} GB of copies per layer)".format(
                (sh.E + sh.S) * 3 * sh.H * sh.I * wbytes / 1e9, placement.n_remote() * 3 * sh.H * sh.I * wbytes / 1e9),
            "parallelism": "single rank"}


def wl_flags(args) -> int:
    """dwdp_config.flags for the benchmark's options."""
    from moe_expert_grouped_split_gb300 import binding as B
    return B.FLAG_WIDE_EPILOGUE if getattr(args, "wide_epilogue", False) else 0


def run_layer_bench(args):
    """The single-layer workloads (8K default, Zipf 16K, 256 tokens)."""
    import torch
    torch.cuda.set_device(0)
    spec = WORKLOADS[args.workload](group=args.group)
    wl = Workload(spec, args.chunk_mb * (1 << 20), args.copy_streams, wdtype=args.dtype, peer_pools=args.peer_pools,
                  prefetch_start=args.prefetch_start, n_stages=args.stages,
                  flags=wl_flags(args))
    sh = wl.shape
    K, W = args.steps, args.warmup
    phases = [_events(torch, 7) for _ in range(K)]
    ms_total, clocks = run_overlapped(wl, K, W, phases)
    res = {"ms_step": ms_total / K, "value": whole_job_rate(sh.T, K, ms_total),
           "phase_ms": _phase_avg(phases, K), "clocks": clocks,
           "issue_ms": round(1e3 * sum(wl.issue_s) / max(1, len(wl.issue_s)), 3)}
    e_active = int((wl.rb.counts[: sh.E] > 0).sum().item())
    res["e_active"] = e_active
    if not args.no_extras:
        res["compute_only_ms"] = run_compute_only(wl, K, phases)
        res["compute_only_phase_ms"] = _phase_avg(phases, K)
        res["copy_only_ms"] = run_copy_only(wl, K)
        res["e2e"] = run_e2e(wl, K)
    if args.chunk_sweep:
        sweep = []
        comp = res.get("compute_only_ms") or run_compute_only(wl, K)
        for mb in [float(v) for v in args.chunk_sweep.split(",") if v]:
            wl.chunk = int(mb * (1 << 20))
            wl.issue_s = []
            ms, _ = run_overlapped(wl, K, W, None)
            issue = 1e3 * sum(wl.issue_s) / max(1, len(wl.issue_s))
            copy = run_copy_only(wl, K)
            over = ms / K
            exposed = max(0.0, over - comp)
            sweep.append({"chunk_mb": mb, "overlapped_ms": round(over, 4), "copy_only_ms": round(copy, 4),
                          "compute_only_ms": round(comp, 4), "exposed_ms": round(exposed, 4),
                          "hidden_frac": round(max(0.0, 1 - exposed / copy), 4) if copy > 0 else None,
                          "host_issue_ms_per_prefetch": round(issue, 3),
                          "slices_per_prefetch": len(wl.B.dwdp_plan_prefetch(
                              sh.E, sh.H, sh.I, wl.placement.local_slot, wl.placement.peer_id,
                              wl.placement.peer_slot, wl.placement.n_peers, wl.chunk))})
        res["chunk_sweep"] = sweep
    if args.duration_study > 0:
        comp = run_duration(wl, args.duration_study, overlapped=False)
        over = run_duration(wl, args.duration_study, overlapped=True)
        res["duration_study"] = {
            "compute_only": comp, "overlapped": over,
            "step_ratio": round(over["ms_per_step"] / comp["ms_per_step"], 3),
            "gate_up_ratio": round(over["last_steps_phase_ms"]["gate_up_gemm"]
                                   / comp["last_steps_phase_ms"]["gate_up_gemm"], 3),
            "sm_clock_ratio": (round(over["clocks"]["sm_mhz"] / comp["clocks"]["sm_mhz"], 3)
                               if over["clocks"]["sm_mhz"] and comp["clocks"]["sm_mhz"] else None)}
    if args.merge_copy:
        res["merge_copy"] = run_merge_baseline(wl, K, W)
    res["wl"] = wl
    return res


class MergeCopyLayer:
    """The pages' baseline before split-weight management (DWDP §4.2): the
    grouped GEMM reads ONE contiguous [E] weight buffer per layer, so after
    the non-resident experts arrive the resident ones are merged into it
    with a device-to-device copy on the critical path.  Built from the
    public ABI only, in the variant most favourable to the baseline: the
    prefetch lands directly in the merged buffer (its slots 0..R-1, the
    stage slots of the non-resident experts in ascending id) and only the
    resident experts are copied (to slots R..E-1), then the same kernels run
    on a map in which every expert is resident in that buffer.  Merged
    buffer s (a staging buffer of a context with E stage slots) serves
    layer l of `layers` at step parity s: maps 2 + 2 l + s."""

    def __init__(self, B, torch, shape, placement, layers, wdtype: str, max_tokens=None):
        sh, pl = shape, placement
        if (pl.local_slot >= 0).sum() != pl.n_local_slots or pl.n_remote() + pl.n_local_slots != sh.E:
            raise ValueError("a redundant placement has no single merged layout")
        self.B, self.torch, self.shape, self.pl, self.layers = B, torch, sh, pl, layers
        wd = {"bf16": B.DTYPE_BF16, "fp8": B.DTYPE_E4M3, "nvfp4": B.DTYPE_NVFP4}[wdtype]
        self.rt = B.Runtime(sh.H, sh.I, sh.E, sh.k, sh.S, max_tokens or sh.T, 2 + 2 * len(layers), sh.E,
                            weight_dtype=wd)
        stage_slot = [-1] * sh.E
        r = 0
        for e in range(sh.E):
            if pl.local_slot[e] < 0:
                stage_slot[e] = r
                r += 1
        self.R = r
        self.merged_slot = [stage_slot[e] if pl.local_slot[e] < 0 else r + int(pl.local_slot[e]) for e in range(sh.E)]
        for l, lw in enumerate(layers):
            self.rt.set_layer(l, lw)                          # layers 0, 1: where the prefetch reads from
            for s in (0, 1):                                  # maps 2+2l+s: everything resident in merged[s]
                local = B.pool(self.rt.stage_w13[s], self.rt.stage_w2[s])
                B.dwdp_set_expert_map(self.rt.ctx, 2 + 2 * l + s, local, [], self.merged_slot, [-1] * sh.E,
                                      [-1] * sh.E, lw.shared_w13, lw.shared_w2)
                if getattr(lw, "w13_scale", None) is not None:
                    B.dwdp_set_expert_scales(self.rt.ctx, 2 + 2 * l + s, lw.w13_scale, lw.w2_scale, lw.shared_s13,
                                             lw.shared_s2)
        self.w13_bytes = B.weight_slot_bytes(2 * sh.I, sh.H, wd)
        self.w2_bytes = B.weight_slot_bytes(sh.H, sh.I, wd)
        self.n_local = pl.n_local_slots
        self.merge_bytes = self.n_local * (self.w13_bytes + self.w2_bytes)
        self.arrived = [torch.cuda.Event(), torch.cuda.Event()]
        self.freed = [torch.cuda.Event(), torch.cuda.Event()]

    def prefetch(self, l, s, chunk, copies):
        """Layer l's non-resident experts into merged buffer s (slots 0..R-1)."""
        copies[0].wait_event(self.freed[s])
        self.rt.prefetch(l, s, chunk, copies)
        self.arrived[s].record(copies[0])

    def merge(self, l, s, stream):
        """The D2D merge: layer l's resident experts into slots R.. of buffer s."""
        lw, n = self.layers[l], self.n_local
        with self.torch.cuda.stream(stream):
            stream.wait_event(self.arrived[s])
            self.rt.stage_w13[s][self.R:self.R + n].copy_(lw.local_w13[:n].view(self.torch.uint8).reshape(n, -1),
                                                          non_blocking=True)
            self.rt.stage_w2[s][self.R:self.R + n].copy_(lw.local_w2[:n].view(self.torch.uint8).reshape(n, -1),
                                                         non_blocking=True)

    def layer(self, l, s, x, rb, out, stream):
        """Merge, route and the MoE layer on the merged buffer."""
        self.merge(l, s, stream)
        lw = self.layers[l]
        with self.torch.cuda.stream(stream):
            self.rt.route(x, lw.wr, lw.bias, rb, stream)
            self.rt.moe(2 + 2 * l + s, s, x, rb, out, stream)
            self.freed[s].record(stream)

    def close(self):
        self.rt.close()


def run_merge_baseline(wl, K, W):
    """The merge-copy baseline (MergeCopyLayer) timed like the split-pointer
    step: ms per step overlapped with the next layer's prefetch, and with
    every expert already staged (merge + compute only), plus the merge bytes."""
    torch = wl.torch
    try:
        mc = MergeCopyLayer(wl.B, torch, wl.shape, wl.placement, wl.layers, wl.wdtype)
    except ValueError:
        return None

    def step(i, prefetch_next=True):
        l = s = i % 2
        mc.layer(l, s, wl.x[l], wl.rb, wl.out, wl.compute)
        if prefetch_next:
            mc.prefetch((i + 1) % 2, (i + 1) % 2, wl.chunk, wl.copies)

    wl.sync()
    mc.prefetch(0, 0, wl.chunk, wl.copies)
    for i in range(W):
        step(i)
    wl.sync()
    a, b = _events(torch, 2)
    a.record(wl.compute)
    for c in wl.copies:
        c.wait_stream(wl.compute)
    for i in range(W, W + K):
        step(i)
    for c in wl.copies:
        wl.compute.wait_stream(c)
    b.record(wl.compute)
    b.synchronize()
    over = a.elapsed_time(b) / K
    # every expert already staged: merge + compute only
    wl.sync()
    for l in (0, 1):
        mc.prefetch(l, l, wl.chunk, wl.copies)
    wl.sync()
    for i in range(2):
        step(i, prefetch_next=False)
    a, b = _events(torch, 2)
    a.record(wl.compute)
    for i in range(K):
        step(i, prefetch_next=False)
    b.record(wl.compute)
    b.synchronize()
    comp = a.elapsed_time(b) / K
    assert mc.rt.device_status() == 0
    merge_bytes, n_local = mc.merge_bytes, mc.n_local
    mc.close()
    return {"overlapped_ms": round(over, 4), "compute_only_ms": round(comp, 4),
            "merge_bytes_per_layer": merge_bytes, "merged_experts_copied": n_local}


def run_pipeline_bench(args):
    """Four distinct R1 layers per step with an attention-sized GEMM
    stand-in (x . W_attn, T x 7168 x 7168, on this library's grouped GEMM)
    after each MoE layer; the copy of the next layer's experts overlaps the
    current MoE layer and the stand-in that follows it (DWDP §2).  T per step is
    uniform in [6554, 8192] (0.8x-1.0x of 8K), 16 steps by default."""
    import numpy as np
    import torch

    from moe_expert_grouped_split_gb300 import binding as B
    from moe_expert_grouped_split_gb300 import inputs as I

    torch.cuda.set_device(0)
    spec = WORKLOADS[args.workload](group=args.group)
    wl = Workload(spec, args.chunk_mb * (1 << 20), args.copy_streams, n_layers=4, wdtype=args.dtype,
                  prefetch_start=args.prefetch_start, n_stages=args.stages, flags=wl_flags(args))
    S = wl.n_stages
    sh = wl.shape
    steps = args.steps
    Ts = I.step_token_counts(steps + args.warmup, 6554, 8192, 0)
    w_attn = I.randn_bf16((1, sh.H, sh.H), 0.02, I.seed_for(0, "W_attn"), "cuda")
    scratch = torch.empty((sh.T, sh.H), dtype=torch.bfloat16, device="cuda")
    offs = torch.zeros((len(Ts), 4), dtype=torch.int32)
    offs[:, 1] = torch.tensor(Ts, dtype=torch.int32)
    offs = offs.cuda()

    def attn_standin(l, s):
        x = wl.x[l][: Ts[s]]
        with torch.cuda.stream(wl.compute):
            B.dwdp_grouped_gemm(wl.rt.ctx, B.EPI_BF16, x, Ts[s], sh.H, sh.H, offs[s], 1, [w_attn], [0, 0],
                                scratch, wl.compute)

    def run(s_from, s_to, with_copies, layer_of=lambda g: g % 4):
        g = s_from * 4
        gate = with_copies and wl.prefetch_start == "gate_up"
        wl.set_phases(wl.gate_ev if gate else None)
        wl.gated_by = wl.gate_ev if gate else None
        for s in range(s_from, s_to):
            for l in range(4):
                lay = layer_of(g)
                stage = g % S if with_copies else lay % 2
                wl.layer_step(lay, stage, T=Ts[s])
                if with_copies:   # the layer S - 1 ahead into its stage
                    wl.prefetch(layer_of(g + S - 1), (g + S - 1) % S)
                attn_standin(layer_of(g + 1), s)
                g += 1

    ev = lambda: _events(torch, 2)
    # overlapped: prologue (the first S - 1 layers into their stages) outside the timed steps
    for j in range(S - 1):
        wl.prefetch(j, j)
    run(0, args.warmup, True)
    wl.sync()
    a, b = ev()
    with ClockSampler(0) as clk:
        a.record(wl.compute)
        for c in wl.copies:
            c.wait_stream(wl.compute)
        run(args.warmup, args.warmup + steps, True)
        for c in wl.copies:
            wl.compute.wait_stream(c)
        b.record(wl.compute)
        b.synchronize()
    assert wl.rt.device_status() == 0
    ms = a.elapsed_time(b)
    tokens = 4 * sum(Ts[args.warmup:])
    res = {"ms_step": ms / steps, "value": tokens / (ms / 1e3), "clocks": clk.summary()}
    if not args.no_extras:
        # compute only: the same sequence with layers 0 and 1 (staged once)
        # standing in for 2 and 3 (same shapes, same routing statistics)
        wl.sync()
        wl.prefetch(0, 0)
        wl.prefetch(1, 1)
        wl.sync()
        a, b = ev()
        a.record(wl.compute)
        run(args.warmup, args.warmup + steps, False, layer_of=lambda g: g % 2)
        b.record(wl.compute)
        b.synchronize()
        res["compute_only_ms"] = a.elapsed_time(b) / steps
        a, b = ev()
        a.record(wl.copies[0])
        for g in range(4 * steps):
            wl.prefetch(g % 4, g % 2)
        b.record(wl.copies[0])
        b.synchronize()
        res["copy_only_ms"] = a.elapsed_time(b) / steps
    res["tokens_per_step"] = [int(t) for t in Ts[args.warmup:]]
    res["wl"] = wl
    return res


def cpu_baseline_sample(wl, target_s=15.0, max_tokens=512):
    """The oracle as it stands on host cores, on a seeded token sample of the
    same workload (the layer's rows are independent, so a sample's cost per
    token is the layer's)."""
    import numpy as np

    import oracle
    from moe_expert_grouped_split_gb300 import inputs as I

    o = oracle.default()
    sh = wl.shape
    lw = wl.layers[0]
    x = I.bf16_bits(wl.x[0])
    rng = np.random.default_rng(1234)
    order = rng.permutation(sh.T)
    wr = I.bf16_bits(lw.wr)
    bias = None if lw.bias is None else lw.bias.cpu().numpy()
    cache = {}
    pl = lw.placement

    def weights_for(ids):
        need = sorted(set(int(e) for e in np.unique(ids)) - set(cache))
        for e in need:
            if pl.local_slot[e] >= 0:
                w13, w2 = lw.local_w13[pl.local_slot[e]], lw.local_w2[pl.local_slot[e]]
            else:
                w13, w2 = lw.peer_w13[pl.peer_id[e]][pl.peer_slot[e]], lw.peer_w2[pl.peer_id[e]][pl.peer_slot[e]]
            cache[e] = (conv13(w13), conv2(w2))
        w13s = [cache.get(e, (None, None))[0] for e in range(sh.E)]
        w2s = [cache.get(e, (None, None))[1] for e in range(sh.E)]
        return w13s, w2s

    wdtype = getattr(wl, "wdtype", "bf16")
    fp8, nvfp4 = wdtype == "fp8", wdtype == "nvfp4"
    conv = (lambda t: t.detach().contiguous().cpu().numpy().view(np.uint8)) if fp8 else I.bf16_bits
    conv13 = conv2 = conv
    if nvfp4:   # slots to math layout: (codes, block scales) of w13 / of w2
        conv13 = lambda t: I.unpack_nvfp4(t.detach().cpu(), 2 * sh.I, sh.H)
        conv2 = lambda t: I.unpack_nvfp4(t.detach().cpu(), sh.H, sh.I)
    sw13 = conv13(lw.shared_w13) if lw.shared_w13 is not None else None
    sw2 = conv2(lw.shared_w2) if lw.shared_w2 is not None else None

    def run(tokens):
        xs = np.ascontiguousarray(x[tokens])
        r_pre = o.route(xs, wr, bias, sh.k)            # routing, untimed pass to learn the experts
        w13s, w2s = weights_for(r_pre["ids"])          # host copies of those experts (untimed)
        t0 = time.perf_counter()
        r = o.route(xs, wr, bias, sh.k)
        if nvfp4:
            sh_t = None if sw13 is None else (sw13[0], sw13[1], lw.shared_s13, sw2[0], sw2[1], lw.shared_s2)
            o.moe_tokens_nvfp4(xs, np.arange(len(tokens)), r["ids"], r["w"],
                               [None if a is None else a[0] for a in w13s], [None if a is None else a[1] for a in w13s],
                               lw.w13_scale, [None if a is None else a[0] for a in w2s],
                               [None if a is None else a[1] for a in w2s], lw.w2_scale, shared=sh_t, mirrored=True)
        elif fp8:
            o.moe_tokens_fp8(xs, np.arange(len(tokens)), r["ids"], r["w"], w13s, w2s, lw.w13_scale, lw.w2_scale,
                             sw13, sw2, lw.shared_s13, lw.shared_s2, mirrored=True)
        else:
            o.moe_tokens(xs, np.arange(len(tokens)), r["ids"], r["w"], w13s, w2s, sw13, sw2, mirrored=True)
        return time.perf_counter() - t0

    n = 8
    dt = run(order[:n])
    per_tok = dt / n
    n2 = int(min(max_tokens, sh.T, max(n, target_s / max(per_tok, 1e-9))))
    if n2 > n:
        dt = run(order[:n2])
        n = n2
    cores = o.num_threads()
    # the same oracle on one thread, on one or two of the sampled tokens
    o.set_num_threads(1)
    try:
        n1 = 2 if per_tok * cores < 2.0 else 1
        dt1 = run(order[:n1])
    finally:
        o.set_num_threads(cores)
    return {"value": round(n / dt, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "value_1thread": round(n1 / dt1, 3),
            "sample": f"{n} seeded tokens of the {sh.T}-token R1-shaped layer (routing + {sh.k} routed experts"
                      f"{' + shared expert' if sh.S else ''} per token, fp64, {dt:.1f} s; one thread: {n1} "
                      f"tokens, {dt1:.1f} s)"}


def parse_variant(main_workload: str, variant: str):
    """(workload, weight type, wide epilogue) of a --variants entry."""
    workload, wdtype = main_workload, variant
    if variant.split(":")[0] in WORKLOADS:
        workload, _, wdtype = variant.partition(":")
        wdtype = wdtype or "bf16"
    wide = wdtype.endswith("_wide")
    wdtype = wdtype[: -len("_wide")] if wide else wdtype
    if wdtype not in WEIGHT_BYTES:
        raise ValueError(f"unknown variant {variant!r}")
    return workload, wdtype, wide


def variant_summary(args, variant: str) -> dict:
    """One more measurement in the same run, in compact form.  variant is
    "<dtype>[_wide]" (the main line's workload with E4M3 or NVFP4 weights,
    _wide = NVFP4 with the eight-warp gate/up epilogue) or
    "<workload>[:<dtype>]" (another workload of WORKLOADS, bf16 unless
    given; the bf16 256-token layer adds the chunk sweep over 1, 4, 16 and
    64 MB slices), timed like the main line: overlapped steps, compute-only
    and copy-only legs, and (single layers) end to end with host buffers."""
    import copy as _copy

    import torch
    a = _copy.copy(args)
    workload, wdtype, wide = parse_variant(args.workload, variant)
    # the merge-copy baseline also for the main workload in the pages' weight format
    merge = workload == "r1_moe_layer_8k" and wdtype == "nvfp4" and not wide and args.group == 4
    a.workload, a.dtype, a.merge_copy, a.wide_epilogue = workload, wdtype, merge, wide
    if not args.copy_streams_given:
        a.copy_streams = default_copy_streams(workload, wdtype)
    a.chunk_sweep = "1,4,16,64" if workload == "r1_moe_layer_256" and wdtype == "bf16" else ""
    a.chunk_mb = default_chunk_mb(workload, wdtype)
    pipeline = workload == "r1_pipeline_4layer"
    if pipeline:
        a.steps = 16        # the 4-layer workload's own step count
    res = (run_pipeline_bench if pipeline else run_layer_bench)(a)
    wl = res.pop("wl")
    sh = wl.shape
    comp, copy_ms = res["compute_only_ms"], res["copy_only_ms"]
    exposed = max(0.0, res["ms_step"] - comp)
    out = {
        "workload": workload, "T": sh.T, "expert_weights": wdtype, "wide_epilogue": wide,
        "value": round(res["value"], 1), "unit": UNIT + (" (layer-tokens, 4 layers per step)" if pipeline else ""),
        "ms_per_step": round(res["ms_step"], 4),
        "prefetch": {"compute_only_ms": round(comp, 4), "copy_only_ms": round(copy_ms, 4),
                     "exposed_ms": round(exposed, 4),
                     "hidden_frac": round(max(0.0, 1.0 - exposed / copy_ms), 4) if copy_ms > 0 else None},
        "clocks": res["clocks"], "chunk_mb": a.chunk_mb, "copy_streams": a.copy_streams,
    }
    if pipeline:
        flops = sum(4 * (layer_flops(T, sh.H, sh.I, sh.E, sh.k, sh.S) + 2 * T * sh.H * sh.H)
                    for T in res["tokens_per_step"]) / len(res["tokens_per_step"])
        out["tflops"] = round(flops / (res["ms_step"] / 1e3) / 1e12, 1)
        out["tokens_per_step"] = res["tokens_per_step"]
        out["gpu_launches"] = args.steps * 4 * kernels_per_layer(wdtype)
    else:
        peaks, src = measured_peaks()
        tc_peak, hbm, tc_note = roofline_peaks(peaks, src, wdtype)
        wb = WEIGHT_BYTES[wdtype]
        g1 = g1_flops(sh.T, sh.H, sh.I, sh.k, sh.S)
        g1b = g1_bytes(sh.T, sh.H, sh.I, res["e_active"], sh.k, sh.S, wb)
        out.update({
            "e2e": res["e2e"],
            "tflops": round(layer_flops(sh.T, sh.H, sh.I, sh.E, sh.k, sh.S) / (res["ms_step"] / 1e3) / 1e12, 1),
            "phase_ms": res["phase_ms"], "compute_only_phase_ms": res["compute_only_phase_ms"],
            "roofline": roofline_entry("gate_up_grouped_gemm", g1, g1b, res["phase_ms"]["gate_up_gemm"] / 1e3,
                                       tc_peak, hbm, tc_note, f"{src} hbm_gbs"),
            "roofline_alone": roofline_entry("gate_up_grouped_gemm", g1, g1b,
                                             res["compute_only_phase_ms"]["gate_up_gemm"] / 1e3, tc_peak, hbm,
                                             tc_note, f"{src} hbm_gbs"),
            "step_hbm_frac": round(step_bytes(sh.T, sh.H, sh.I, res["e_active"], sh.k, sh.S,
                                              wl.placement.n_remote(), wb) / (res["ms_step"] / 1e3) / 1e9 / hbm, 4),
            "experts_active": res["e_active"],
            "gpu_launches": kernels_per_layer(wdtype) * args.steps,
        })
        if "chunk_sweep" in res:
            out["chunk_sweep"] = res["chunk_sweep"]
        if res.get("merge_copy"):
            out["merge_copy_baseline"] = res["merge_copy"]
    wl.rt.close()
    del wl, res
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        return main_reference(args, rank, world)
    refusal = single_gpu_refusal(args, world)
    if refusal is not None:
        # nothing is built or loaded: no kernel of this library runs on more than one GPU
        if rank == 0:
            print(json.dumps(refusal), flush=True)
        return

    from moe_expert_grouped_split_gb300.build import build
    build()
    pipeline = args.workload == "r1_pipeline_4layer"
    res = (run_pipeline_bench if pipeline else run_layer_bench)(args)
    wl = res.pop("wl")
    sh = wl.shape
    peaks, src = measured_peaks()
    tc_peak, hbm, tc_note = roofline_peaks(peaks, src, args.dtype)
    hbm_note = f"{src} hbm_gbs"
    wb = WEIGHT_BYTES[args.dtype]
    line = {
        "metric": METRIC, "value": round(res["value"], 1), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_step"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": {"bf16": "bf16", "fp8": "e4m3", "nvfp4": "nvfp4"}[args.dtype],
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02) weights; R1 MoE layer shapes)",
        "config": workload_config(args, sh, wl.placement, wl.n_layers),
        "clocks": res["clocks"],
    }
    if pipeline:
        flops = sum(4 * (layer_flops(T, sh.H, sh.I, sh.E, sh.k, sh.S) + 2 * T * sh.H * sh.H)
                    for T in res["tokens_per_step"]) / len(res["tokens_per_step"])
        line["config"]["tokens_per_step"] = res["tokens_per_step"]
        line["config"]["attention_standin"] = "bf16 GEMM T x 7168 x 7168 after every MoE layer"
        line["config"]["expert_weights"] = args.dtype
        line["tflops"] = round(flops / (res["ms_step"] / 1e3) / 1e12, 1)
        line["gpu_launches"] = args.steps * 4 * kernels_per_layer(args.dtype)
    else:
        flops_layer = layer_flops(sh.T, sh.H, sh.I, sh.E, sh.k, sh.S)
        g1 = g1_flops(sh.T, sh.H, sh.I, sh.k, sh.S)
        g1b = g1_bytes(sh.T, sh.H, sh.I, res["e_active"], sh.k, sh.S, wb)
        sb = step_bytes(sh.T, sh.H, sh.I, res["e_active"], sh.k, sh.S, wl.placement.n_remote(), wb)
        layer_tflops = flops_layer / (res["ms_step"] / 1e3) / 1e12
        traffic = None
        if args.workload == "r1_moe_layer_8k" and args.dtype == "bf16":
            traffic = measured_traffic(os.path.join(ROOT, "moe_expert_grouped_split_gb300", "csrc", "gemm.cu"), g1b)
        roof = roofline_entry("gate_up_grouped_gemm", g1, g1b, res["phase_ms"]["gate_up_gemm"] / 1e3, tc_peak, hbm,
                              tc_note, hbm_note)
        roof.update({"traffic": traffic, "algorithmic_flops_per_launch": g1, "algorithmic_bytes_per_launch": g1b,
                     "traffic_source": "ncu DRAM bytes (read + write) of this kernel's launch at this workload, "
                                       "1-pass capture of the same source (profiles/"
                                       "gate_up_gemm_traffic_r1_moe_layer_8k.json)" if traffic else None,
                     "timed": "CUDA events around the kernel on the compute stream, inside the overlapped step"})
        line.update({
            "tflops": round(layer_tflops, 1),
            "tc_peak_frac": round(layer_tflops / tc_peak, 4),
            "tc_peak": {"value": tc_peak, "unit": "TFLOP/s", "source": tc_note},
            "phase_ms": res["phase_ms"],
            "roofline": roof,
            "step_hbm": {"bound": "hbm", "achieved": round(sb / (res["ms_step"] / 1e3) / 1e9, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(sb / (res["ms_step"] / 1e3) / 1e9 / hbm, 4),
                         "algorithmic_bytes_per_step": sb, "peak_source": hbm_note},
            "host_issue_ms_per_prefetch": res["issue_ms"],
            "merge_copy_baseline": res.get("merge_copy"),
            "gpu_launches": kernels_per_layer(args.dtype) * args.steps,
        })
        if "chunk_sweep" in res:
            line["chunk_sweep"] = res["chunk_sweep"]
        if "duration_study" in res:
            line["duration_study"] = res["duration_study"]
    if "compute_only_ms" in res:
        comp, copy = res["compute_only_ms"], res["copy_only_ms"]
        exposed = max(0.0, res["ms_step"] - comp)
        pre = {"compute_only_ms": round(comp, 4), "copy_only_ms": round(copy, 4),
               "overlapped_ms": round(res["ms_step"], 4), "exposed_ms": round(exposed, 4),
               "hidden_frac": round(max(0.0, 1.0 - exposed / copy), 4) if copy > 0 else None,
               "model_max_ms": round(max(comp, copy), 4)}
        if not pipeline:
            pre["copy_gbs"] = round(wl.placement.n_remote() * 3 * sh.H * sh.I * wb / (copy / 1e3) / 1e9, 1)
            pre["compute_only_phase_ms"] = res["compute_only_phase_ms"]
            # kernel slowdown while the copy engine runs (analogue of the pages'
            # communication-computation interference, DWDP appendix A)
            pre["interference"] = {n_: round(res["phase_ms"][n_] / max(res["compute_only_phase_ms"][n_], 1e-9), 3)
                                   for n_ in PHASES if n_ != "wait_stage"}
            # the roofline kernel again, timed in the compute-only leg (no copy
            # sharing the memory system), against the same roof
            r = line["roofline"]
            alone = roofline_entry(r["kernel"], r["algorithmic_flops_per_launch"], r["algorithmic_bytes_per_launch"],
                                   res["compute_only_phase_ms"]["gate_up_gemm"] / 1e3, tc_peak, hbm, tc_note,
                                   hbm_note)
            alone["timed"] = "CUDA events around the kernel on the compute stream, compute-only leg (no copy)"
            line["roofline_alone"] = alone
        line["prefetch"] = pre
    if "e2e" in res:
        line["e2e"] = res["e2e"]
    if not args.no_cpu_baseline and not pipeline:
        line["cpu_baseline"] = cpu_baseline_sample(wl)
    if args.variants and not pipeline:
        import torch
        wl.rt.close()
        del wl, res
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["variants"] = {v: variant_summary(args, v) for v in args.variants.split(",") if v}
    print(json.dumps(line), flush=True)


def main_reference(args, rank, world):
    """The oracle as it stands, timed on host cores, same metric, unit and
    expert weight format; each step is one seeded token per oracle thread."""
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from moe_expert_grouped_split_gb300 import inputs as I

    spec = WORKLOADS[args.workload](group=args.group)
    shape = spec.shape
    T = shape.T
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    o = oracle.default()
    x_all = I.bf16_bits(I.make_tokens(T, shape.H, 0, device=dev))
    wr = I.bf16_bits(I.randn_bf16((shape.E, shape.H), spec.router_std, I.seed_for(0, "Wr", 0), dev))
    rng = np.random.default_rng(99)
    per_step = max(1, o.num_threads())
    wd = args.dtype
    cache = {}

    def host(w):
        """Math-layout host arrays of one expert as the oracle takes them."""
        if wd == "bf16":
            return I.bf16_bits(w[0]), I.bf16_bits(w[1])
        if wd == "fp8":
            return w[0].cpu().numpy(), w[1].cpu().numpy()
        return tuple(t.cpu().numpy() for t in (*w[0], *w[1]))     # codes13, sf13, codes2, sf2

    def expert(e):
        if e not in cache:
            cache[e] = host(I.expert_weights(wd, shape, 0, 0, e, dev))
        return cache[e]

    shared = host(I.expert_weights(wd, shape, 0, 0, None, dev)) if shape.S else None
    scales = I.expert_scales(wd, 0, 0, shape.E) if wd != "bf16" else None

    def layer(xs, r, n):
        col = lambda i: [cache[e][i] if e in cache else None for e in range(shape.E)]
        if wd == "bf16":
            return o.moe_tokens(xs, np.arange(n), r["ids"], r["w"], col(0), col(1),
                                *(shared if shared else (None, None)), mirrored=True)
        s13, s2, ss13, ss2 = scales
        if wd == "fp8":
            kw = dict(shared_w13=shared[0], shared_w2=shared[1], shared_s13=ss13, shared_s2=ss2) if shared else {}
            return o.moe_tokens_fp8(xs, np.arange(n), r["ids"], r["w"], col(0), col(1), s13, s2, mirrored=True, **kw)
        sh = (shared[0], shared[1], ss13, shared[2], shared[3], ss2) if shared else None
        return o.moe_tokens_nvfp4(xs, np.arange(n), r["ids"], r["w"], col(0), col(1), s13, col(2), col(3), s2,
                                  shared=sh, mirrored=True)

    times = []
    ntok = 0
    for s in range(args.warmup + args.steps):
        tok = rng.choice(T, size=per_step, replace=False)
        xs = np.ascontiguousarray(x_all[tok])
        pre = o.route(xs, wr, spec.bias, shape.k)
        for e in np.unique(pre["ids"]):
            expert(int(e))
        t0 = time.perf_counter()
        r = o.route(xs, wr, spec.bias, shape.k)
        layer(xs, r, per_step)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
            ntok += per_step
    total = sum(times)
    value = ntok / total
    ms_step = total / len(times) * 1e3     # one timed step = one bounded token sample
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 1),
        "ms_per_layer_extrapolated": round(T / value * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, R1 MoE layer shapes)",
        # the same workload as the GPU arm's line (the oracle's result does not
        # depend on the placement or the prefetch settings)
        "config": workload_config(args, shape, spec.placement, 4 if args.workload == "r1_pipeline_4layer" else 2),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": o.num_threads(), "kind": "oracle",
                         "sample": f"{per_step} seeded tokens per step (one per oracle thread) of the {T}-token "
                                   f"layer, {args.steps} timed steps ({total:.1f} s); ms_per_step is one such "
                                   f"step, ms_per_layer_extrapolated the whole {T}-token layer at this rate"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
