"""Split-pointer grouped GEMM (dwdp_grouped_gemm, tcgen05 + TMA) against the
oracle's grouped GEMM, element by element: several tiles in M, N and K,
ragged and empty groups, several weight buffers, the three epilogues, and
rows outside every group left untouched."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, to_f64
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I
from moe_expert_grouped_split_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rt():
    build()
    r = B.Runtime(256, 128, 8, 2, 0, 64, 1, 0)
    yield r
    r.close()


def _case(rt, epi, K, N, sizes, n_bufs, slots, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(off[-1]) + 7                       # trailing rows outside every group
    a = (torch.randn((rows, K), generator=g) * 1.0).to(torch.bfloat16)
    brows = 2 * N if epi == B.EPI_SILU else N
    bufs = [(torch.randn((slots, brows, K), generator=g) * 0.1).to(torch.bfloat16) for _ in range(n_bufs)]
    G = len(sizes)
    rng = np.random.default_rng(seed)
    bs = np.array([[rng.integers(0, n_bufs), rng.integers(0, slots)] for _ in range(G)], dtype=np.int32)
    out_dtype = torch.float32 if epi == B.EPI_F32 else torch.bfloat16
    d = torch.full((rows, N), 7.0, dtype=out_dtype, device="cuda")
    da = a.cuda()
    dbufs = [b.cuda() for b in bufs]
    doff = torch.from_numpy(off).cuda()
    B.dwdp_grouped_gemm(rt.ctx, epi, da, rows, K, N, doff, G, dbufs, bs.reshape(-1), d)
    torch.cuda.synchronize()
    assert rt.device_status() == 0
    o = oracle.default()
    blist = [I.bf16_bits(bufs[b][s]) for b, s in bs]
    ref = o.grouped_gemm(I.bf16_bits(a), off, blist, N, epi)
    got = to_f64(d)
    n_in = int(off[-1])
    if epi == B.EPI_F32:
        err = np.abs(got[:n_in] - ref[:n_in]).max(initial=0.0)
        assert err <= 1e-4 * max(1.0, np.abs(ref).max()), f"fp32 epilogue error {err}"
    else:
        # the kernel rounds each fp32 result to bf16 once; compare with the
        # oracle's fp64 result rounded to bf16 by the oracle
        refb = np.array([o.bf16_to_double(int(b)) for b in o.round_bf16_array(ref[:n_in]).ravel()])
        refb = refb.reshape(ref[:n_in].shape)
        assert_close(got[:n_in], refb, rel_max=1e-2, mae_max=1e-3, what=f"epilogue {epi}")
        # at least 95% of elements are the identical bf16 value
        assert (got[:n_in] == refb).mean() >= 0.95
    assert (got[n_in:] == 7.0).all(), "rows outside every group were written"


@pytest.mark.parametrize("epi", [B.EPI_BF16, B.EPI_SILU, B.EPI_F32])
def test_ragged_groups(rt, epi):
    # K spans 4 k-blocks, N spans 2+ n-tiles, groups: ragged, empty, > 1 m-tile
    N = 320 if epi != B.EPI_F32 else 300
    _case(rt, epi, K=256, N=N, sizes=[130, 0, 1, 257, 64, 0, 128], n_bufs=3, slots=4, seed=epi + 1)


def test_single_row_and_single_group(rt):
    _case(rt, B.EPI_BF16, K=64, N=64, sizes=[1], n_bufs=1, slots=1, seed=11)


def test_many_groups(rt):
    rng = np.random.default_rng(5)
    sizes = rng.integers(0, 40, size=150).tolist()
    _case(rt, B.EPI_SILU, K=128, N=128, sizes=sizes, n_bufs=2, slots=8, seed=12)


def test_device_check_reports_rows_outside_the_output(rt):
    """Group rows live in device memory, so the host cannot check them: rows
    at or past a_rows are not stored, the kernel sets the context's device
    error word, and dwdp_device_status reports DEVICE_CHECK once (then
    clears it); the context stays usable."""
    a = torch.ones((64, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.ones((1, 64, 64), dtype=torch.bfloat16, device="cuda")
    d = torch.zeros((200, 64), dtype=torch.bfloat16, device="cuda")
    off = torch.tensor([0, 100], dtype=torch.int32, device="cuda")     # 100 rows, but a_rows = 64
    B.dwdp_grouped_gemm(rt.ctx, 0, a, 64, 64, 64, off, 1, [b], [0, 0], d)
    torch.cuda.synchronize()
    assert rt.device_status() == -6
    assert "error bits" in B.dwdp_last_error(rt.ctx)
    assert (d[64:].float() == 0).all(), "rows past a_rows were written"
    assert (d[:64].float() == 64).all()
    assert rt.device_status() == 0                                     # cleared, context usable
    off2 = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    B.dwdp_grouped_gemm(rt.ctx, 0, a, 64, 64, 64, off2, 1, [b], [0, 0], d)
    torch.cuda.synchronize()
    assert rt.device_status() == 0


def test_rejects_bad_arguments(rt):
    a = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((1, 64, 64), dtype=torch.bfloat16, device="cuda")
    off = torch.tensor([0, 8], dtype=torch.int32, device="cuda")
    d = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.DwdpError):   # K not a multiple of 64
        B.dwdp_grouped_gemm(rt.ctx, 0, a, 8, 48, 64, off, 1, [b], [0, 0], d)
    with pytest.raises(B.DwdpError):   # slot out of range
        B.dwdp_grouped_gemm(rt.ctx, 0, a, 8, 64, 64, off, 1, [b], [0, 3], d)
    with pytest.raises(B.DwdpError):   # epilogue out of range
        B.dwdp_grouped_gemm(rt.ctx, 5, a, 8, 64, 64, off, 1, [b], [0, 0], d)
