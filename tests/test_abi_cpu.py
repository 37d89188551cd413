"""Host-side checks of libdwdp.so that need no GPU: it builds for sm_103a,
loads, exports every function include/dwdp.h declares, and its host logic
(the prefetch copy plan, argument validation) matches the oracle."""
import ctypes
import re
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300.build import build

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    build()
    return B.lib()


def declared_functions():
    text = (ROOT / "include" / "dwdp.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dwdp_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    bound = {s[0] for s in B.SIGNATURES}
    assert set(names) == bound, "binding and header disagree"
    assert B.dwdp_version() == 5


def _random_map(rng, E, P, redundant=0.0):
    ls = np.full(E, -1, np.int32)
    pid = np.full(E, -1, np.int32)
    ps = np.full(E, -1, np.int32)
    n_local = int(rng.integers(0, E + 1))
    for i, e in enumerate(rng.permutation(E)[:n_local]):
        ls[e] = i
    used = [0] * max(1, P)
    for e in range(E):
        if P and (ls[e] < 0 or rng.random() < redundant):
            p = int(rng.integers(0, P))
            pid[e] = p
            ps[e] = used[p] + int(rng.integers(0, 2))   # gaps break contiguity
            used[p] = ps[e] + 1
    return ls, pid, ps


def test_plan_matches_oracle(lib):
    rng = np.random.default_rng(0)
    for trial in range(300):
        E = int(rng.integers(1, 20))
        P = int(rng.integers(1, 4))
        H = 64 * int(rng.integers(1, 3))
        I = 64 * int(rng.integers(1, 3))
        ls, pid, ps = _random_map(rng, E, P, redundant=0.2)
        chunk = int(rng.choice([1000, 4096, 65536, 10 ** 9, int(rng.integers(100, 300000))]))
        dt = int(rng.choice([B.DTYPE_BF16, B.DTYPE_E4M3, B.DTYPE_NVFP4]))
        got = B.dwdp_plan_prefetch(E, H, I, ls, pid, ps, P, chunk, weight_dtype=dt)
        # bytes per expert tensor as dwdp.h states them: bf16 2 per element,
        # E4M3 1, NVFP4 rows * K * 9 / 16 (codes + block scales)
        tb = {B.DTYPE_BF16: (4 * I * H, 2 * H * I), B.DTYPE_E4M3: (2 * I * H, H * I),
              B.DTYPE_NVFP4: (2 * I * H * 9 // 16, H * I * 9 // 16)}[dt]
        want = oracle.plan_prefetch(E, H, I, ls.tolist(), pid.tolist(), ps.tolist(), P, chunk, tensor_bytes=tb)
        assert got == want, f"trial {trial}"


def test_plan_r1_shape(lib):
    E, H, I = 256, 7168, 2048
    ls = np.array([e if e < 64 else -1 for e in range(E)], np.int32)
    pid = np.array([-1 if e < 64 else (e - 64) // 64 for e in range(E)], np.int32)
    ps = np.array([-1 if e < 64 else (e - 64) % 64 for e in range(E)], np.int32)
    for chunk in (1 << 20, 4 << 20, 16 << 20, 64 << 20):
        got = B.dwdp_plan_prefetch(E, H, I, ls, pid, ps, 3, chunk)
        assert got == oracle.plan_prefetch(E, H, I, ls.tolist(), pid.tolist(), ps.tolist(), 3, chunk)
        assert sum(s[4] for s in got) == 192 * 3 * H * I * 2


def test_plan_rejects_bad_maps(lib):
    with pytest.raises(B.DwdpError) as ei:
        B.dwdp_plan_prefetch(3, 64, 64, [0, -1, 1], [-1, -1, -1], [-1, -1, -1], 1, 1024)
    assert ei.value.code == -1 and "expert 1" in str(ei.value)
    with pytest.raises(B.DwdpError):
        B.dwdp_plan_prefetch(2, 64, 64, [-1, -1], [0, 3], [0, 0], 2, 1024)   # peer 3 of 2
    with pytest.raises(B.DwdpError):
        B.dwdp_plan_prefetch(2, 64, 64, [-1, -1], [0, 0], [0, 1], 1, 0)      # zero chunk


def test_host_validation_without_gpu(lib):
    # NULL config / out are rejected before any CUDA call
    out = ctypes.c_void_p()
    assert lib.dwdp_create(None, None, None, ctypes.byref(out)) == -1
    cfg = B.dwdp_config(256, 128, 8, 2, 0, 64, 1, 0, 7)       # unknown weight type
    assert lib.dwdp_create(ctypes.byref(cfg), None, None, ctypes.byref(out)) == -1
    cfg = B.dwdp_config(100, 128, 8, 2, 0, 64, 1, 0)          # H not a multiple of 64
    assert lib.dwdp_create(ctypes.byref(cfg), None, None, ctypes.byref(out)) == -5
    cfg = B.dwdp_config(256, 128, 8, 9, 0, 64, 1, 0)          # k > E
    assert lib.dwdp_create(ctypes.byref(cfg), None, None, ctypes.byref(out)) == -5
    cfg = B.dwdp_config(320, 256, 8, 2, 0, 64, 1, 0, B.DTYPE_NVFP4)   # NVFP4: H not a multiple of 256
    assert lib.dwdp_create(ctypes.byref(cfg), None, None, ctypes.byref(out)) == -5
    assert "256" in B.dwdp_last_error(None)
    cfg = B.dwdp_config(256, 192, 8, 2, 0, 64, 1, 0, B.DTYPE_NVFP4)   # NVFP4: I not a multiple of 256
    assert lib.dwdp_create(ctypes.byref(cfg), None, None, ctypes.byref(out)) == -5
    cfg = B.dwdp_config(256, 128, 8, 2, 0, 64, 1, 4)          # staging without buffers
    assert lib.dwdp_create(ctypes.byref(cfg), None, None, ctypes.byref(out)) == -1
    assert "stage" in B.dwdp_last_error(None)
    for n_stages in (5, -1):                                    # stage count outside 0 (= 2), 1..4
        cfg = B.dwdp_config(256, 128, 8, 2, 0, 64, 1, 0, B.DTYPE_BF16, n_stages)
        assert lib.dwdp_create(ctypes.byref(cfg), None, None, ctypes.byref(out)) == -1
        assert "n_stages" in B.dwdp_last_error(None)
    # three stages, one missing buffer
    cfg = B.dwdp_config(256, 128, 8, 2, 0, 64, 1, 4, B.DTYPE_BF16, 3)
    bufs = (ctypes.c_void_p * 3)(256, 512, None)
    assert lib.dwdp_create(ctypes.byref(cfg), bufs, bufs, ctypes.byref(out)) == -1
    cfg = B.dwdp_config(256, 128, 8, 2, 0, 64, 1, 0, B.DTYPE_BF16, 0, 6)   # unknown flag bits
    assert lib.dwdp_create(ctypes.byref(cfg), None, None, ctypes.byref(out)) == -1
    assert "flags" in B.dwdp_last_error(None)
    assert lib.dwdp_workspace_bytes(None, 10) == 0
    assert lib.dwdp_selftest_bounded_wait(None, 1000, None) == -1            # no context: nothing enqueued
    # activation quantization: argument checks come before any CUDA call
    x = ctypes.c_void_p(16)
    assert lib.dwdp_quantize_rows(B.DTYPE_BF16, x, 4, 64, x, x, x, None) == -1      # not a quantized type
    assert lib.dwdp_quantize_rows(B.DTYPE_NVFP4, x, 4, 96, x, x, x, None) == -1     # K not a multiple of 64
    assert lib.dwdp_quantize_rows(B.DTYPE_NVFP4, x, 4, 64, x, None, x, None) == -1  # NVFP4 needs block scales
    assert lib.dwdp_quantize_rows(B.DTYPE_NVFP4, x, 0, 64, None, None, None, None) == 0  # nothing to do
    assert lib.dwdp_stage_layer(None, 0) == -1
    if not torch.cuda.is_available():
        cfg = B.dwdp_config(256, 128, 8, 2, 0, 64, 1, 0)
        rc = lib.dwdp_create(ctypes.byref(cfg), None, None, ctypes.byref(out))
        assert rc == -3, B.dwdp_last_error(None)               # no CUDA device here


def test_group_map_matches_oracle(lib):
    for E in (1, 7, 16, 256):
        for N in range(1, min(E, 9) + 1):
            for r in range(N):
                got = [a.tolist() for a in B.dwdp_group_map(E, N, r)]
                assert got == [list(v) for v in oracle.group_map(E, N, r)], (E, N, r)
    for bad in ((8, 0, 0), (8, 3, 3), (8, 9, 0), (0, 1, 0)):
        with pytest.raises(B.DwdpError):
            B.dwdp_group_map(*bad)
