"""The benchmark's layer / stage schedule on the host (no GPU): with S
staging buffers, step i runs layer i % L from stage i % S and prefetches the
layer of step i + S - 1 into stage (i + S - 1) % S, after a prologue that
fills stages 0 .. S-2.  Checked on a recording stand-in for the runtime:
every layer step reads a stage whose last fill was that layer, and no stage
is refilled before the layer it holds has been consumed (the library's
ready / free events order the GPU work; this checks the order the host asks
for)."""
import pytest

import bench


class _FakeB:
    @staticmethod
    def dwdp_set_phase_events(ctx, events):
        pass


class _Rt:
    ctx = 1


def _workload(n_layers, n_stages, log):
    wl = object.__new__(bench.Workload)
    wl.n_layers, wl.n_stages = n_layers, n_stages
    wl.prefetch_start = "route"
    wl.B, wl.rt = _FakeB, _Rt()
    wl.gate_ev = None
    wl.gated_by = None
    wl._phases_set = False
    wl.layer_step = lambda layer, stage, **kw: log.append(("run", layer, stage))
    wl.prefetch = lambda layer, stage: log.append(("fill", layer, stage))
    return wl


@pytest.mark.parametrize("n_layers", [2, 4])
@pytest.mark.parametrize("n_stages", [2, 3, 4])
def test_each_step_reads_the_layer_its_stage_holds(n_layers, n_stages):
    log = []
    wl = _workload(n_layers, n_stages, log)
    wl.prologue()
    steps = 3 * n_layers * n_stages
    for i in range(steps):
        wl.step(i)
    holds = {}          # stage -> layer of its last fill
    pending = {}        # stage -> filled but not yet read
    runs = 0
    for op, layer, stage in log:
        assert 0 <= stage < n_stages
        if op == "fill":
            assert not pending.get(stage), f"stage {stage} refilled before its layer ran"
            holds[stage] = layer
            pending[stage] = True
        else:
            assert holds.get(stage) == layer, f"step {runs}: stage {stage} holds {holds.get(stage)}, not {layer}"
            assert layer == runs % n_layers and stage == runs % n_stages
            pending[stage] = False
            runs += 1
    assert runs == steps


def test_refill_goes_to_the_stage_the_previous_step_read():
    """The fill issued at step i targets the stage step i - 1 read, so the
    copy waits for exactly that step's down GEMM (the stage's free event)."""
    for n_stages in (2, 3, 4):
        log = []
        wl = _workload(2, n_stages, log)
        wl.prologue()
        for i in range(12):
            wl.step(i)
        runs = [e for e in log if e[0] == "run"]
        fills = [e for e in log if e[0] == "fill"][n_stages - 1:]   # after the prologue
        for i, (_, _, stage) in enumerate(fills):
            if i >= 1:
                assert stage == runs[i - 1][2]


def test_compute_only_steps_read_stage_equal_layer():
    log = []
    wl = _workload(2, 3, log)
    for i in range(4):
        wl.step(i, prefetch_next=False)
    assert log == [("run", 0, 0), ("run", 1, 1), ("run", 0, 0), ("run", 1, 1)]
