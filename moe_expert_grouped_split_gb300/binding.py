"""Thin ctypes binding of libdwdp.so (include/dwdp.h): same names, argument
marshalling only.  Every step of the hot path runs in the library's CUDA
kernels; nothing here computes.  Device buffers are torch tensors (PyTorch
provides memory and streams); a missing library raises instead of falling
back to anything else.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import numpy as np

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libdwdp.so"

DWDP_OK = 0
STATUS = {0: "OK", -1: "INVALID_ARG", -2: "NOT_MAPPED", -3: "CUDA", -4: "TIMEOUT", -5: "UNSUPPORTED",
          -6: "DEVICE_CHECK"}
EPI_BF16, EPI_SILU, EPI_F32 = 0, 1, 2
DWDP_PHASE_EVENTS = 7  # dwdp_set_phase_events: route start/end, rows in expert order, stage waited for, gate/up, down, combine
DTYPE_BF16, DTYPE_E4M3, DTYPE_NVFP4 = 0, 1, 2
FLAG_WIDE_EPILOGUE = 1


def weight_slot_bytes(rows: int, K: int, weight_dtype: int) -> int:
    """Bytes of one [rows][K] expert tensor (one pool slot) in weight_dtype:
    bf16 2 per element, E4M3 1, NVFP4 half a byte of E2M1 code plus 1/16
    byte of E4M3 block scale (dwdp.h, DWDP_DTYPE_NVFP4)."""
    if weight_dtype == DTYPE_NVFP4:
        return rows * K // 2 + rows * K // 16
    return rows * K * (1 if weight_dtype == DTYPE_E4M3 else 2)


class DwdpError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class dwdp_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("stage_slots", ctypes.c_int32), ("weight_dtype", ctypes.c_int32),
                ("n_stages", ctypes.c_int32), ("flags", ctypes.c_int32)]


class dwdp_pool(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("n_slots", ctypes.c_int32)]


class dwdp_route_out(ctypes.Structure):
    _fields_ = [("topk_ids", ctypes.c_void_p), ("topk_w", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("perm", ctypes.c_void_p), ("inv_perm", ctypes.c_void_p),
                ("logits", ctypes.c_void_p)]


class dwdp_copy_slice(ctypes.Structure):
    _fields_ = [("peer", ctypes.c_int32), ("tensor", ctypes.c_int32), ("src_offset", ctypes.c_int64),
                ("dst_offset", ctypes.c_int64), ("nbytes", ctypes.c_int64)]


_I32 = ctypes.c_int32
_VP = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)

# (name, restype, argtypes) for every symbol dwdp.h declares
SIGNATURES = [
    ("dwdp_version", _I32, []),
    ("dwdp_create", _I32, [ctypes.POINTER(dwdp_config), ctypes.POINTER(_VP), ctypes.POINTER(_VP),
                           ctypes.POINTER(_VP)]),
    ("dwdp_destroy", None, [_VP]),
    ("dwdp_last_error", ctypes.c_char_p, [_VP]),
    ("dwdp_workspace_bytes", ctypes.c_size_t, [_VP, _I32]),
    ("dwdp_set_expert_map", _I32, [_VP, _I32, ctypes.POINTER(dwdp_pool), ctypes.POINTER(dwdp_pool), _I32,
                                   _I32P, _I32P, _I32P, _VP, _VP]),
    ("dwdp_route", _I32, [_VP, _VP, _I32, _VP, _VP, ctypes.POINTER(dwdp_route_out), _VP, ctypes.c_size_t, _VP]),
    ("dwdp_prefetch_layer", _I32, [_VP, _I32, _I32, ctypes.c_size_t, ctypes.POINTER(_VP), _I32]),
    ("dwdp_moe_layer", _I32, [_VP, _I32, _I32, _VP, _I32, ctypes.POINTER(dwdp_route_out), _VP, _VP,
                              ctypes.c_size_t, _VP]),
    ("dwdp_wait_stage", _I32, [_VP, _I32, _I32]),
    ("dwdp_stage_layer", _I32, [_VP, _I32]),
    ("dwdp_device_status", _I32, [_VP]),
    ("dwdp_set_phase_events", _I32, [_VP, ctypes.POINTER(_VP), _I32]),
    ("dwdp_selftest_bounded_wait", _I32, [_VP, ctypes.c_uint32, _VP]),
    ("dwdp_set_expert_scales", _I32, [_VP, _I32, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float),
                                      ctypes.c_float, ctypes.c_float]),
    ("dwdp_grouped_gemm", _I32, [_VP, _I32, _VP, ctypes.c_int64, _I32, _I32, _VP, _I32, ctypes.POINTER(dwdp_pool),
                                 _I32, _I32P, _VP, _VP]),
    ("dwdp_route_static", _I32, [_VP, _I32, _I32, _I32, _I32, _VP, _VP, ctypes.POINTER(dwdp_route_out), _VP]),
    ("dwdp_route_static_status", _I32, [_VP, _I32P]),
    ("dwdp_group_map", _I32, [_I32, _I32, _I32, _I32P, _I32P, _I32P]),
    ("dwdp_workspace_region", _I32, [_VP, _I32, _I32, ctypes.POINTER(ctypes.c_size_t),
                                     ctypes.POINTER(ctypes.c_size_t)]),
    ("dwdp_quantize_rows", _I32, [_I32, _VP, ctypes.c_int64, _I32, _VP, _VP, _VP, _VP]),
    ("dwdp_plan_prefetch", _I32, [_I32, _I32, _I32, _I32, _I32P, _I32P, _I32P, _I32, ctypes.c_size_t,
                                  ctypes.POINTER(dwdp_copy_slice), ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]),
]

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libdwdp.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is missing: build it with moe_expert_grouped_split_gb300.build.build()")
        L = ctypes.CDLL(str(LIB_PATH))
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(ctx, rc: int) -> int:
    if rc < 0:
        raise DwdpError(rc, lib().dwdp_last_error(ctx).decode())
    return rc


def _i32(a) -> ctypes.Array:
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr, arr.ctypes.data_as(_I32P)


# ---------------------------------------------------------------- calls --
def dwdp_version() -> int:
    return lib().dwdp_version()


def dwdp_create(hidden, inter, n_experts, top_k, n_shared, max_tokens, n_layers, stage_slots,
                stage_w13=(None, None), stage_w2=(None, None), weight_dtype=DTYPE_BF16, n_stages=0, flags=0) -> int:
    """n_stages 0 means 2; stage_w13 / stage_w2 hold one buffer (or None) per stage."""
    cfg = dwdp_config(hidden, inter, n_experts, top_k, n_shared, max_tokens, n_layers, stage_slots, weight_dtype,
                      n_stages, flags)
    n = max(len(stage_w13), len(stage_w2), n_stages or 2)
    s13 = (_VP * n)(*[_ptr(stage_w13[i]) if i < len(stage_w13) else None for i in range(n)])
    s2 = (_VP * n)(*[_ptr(stage_w2[i]) if i < len(stage_w2) else None for i in range(n)])
    out = _VP()
    _check(None, lib().dwdp_create(ctypes.byref(cfg), s13, s2, ctypes.byref(out)))
    return out.value


def dwdp_destroy(ctx: int) -> None:
    lib().dwdp_destroy(ctx)


def dwdp_last_error(ctx: int | None) -> str:
    return lib().dwdp_last_error(ctx).decode()


def dwdp_workspace_bytes(ctx: int, T: int) -> int:
    return lib().dwdp_workspace_bytes(ctx, T)


def pool(w13, w2, n_slots=None) -> dwdp_pool:
    """A dwdp_pool over two device tensors [slots][2I][H] and [slots][H][I]."""
    if n_slots is None:
        n_slots = w13.shape[0] if w13 is not None else 0
    return dwdp_pool(_ptr(w13), _ptr(w2), int(n_slots))


def dwdp_set_expert_map(ctx, layer, local, peers, local_slot, peer_id, peer_slot, shared_w13=None,
                        shared_w2=None) -> None:
    n_peers = len(peers)
    parr = (dwdp_pool * max(1, n_peers))(*peers) if n_peers else None
    ls, lsp = _i32(local_slot)
    pi, pip = _i32(peer_id)
    ps, psp = _i32(peer_slot)
    _check(ctx, lib().dwdp_set_expert_map(ctx, layer, ctypes.byref(local) if local is not None else None,
                                          parr, n_peers, lsp, pip, psp, _ptr(shared_w13), _ptr(shared_w2)))


def route_out(topk_ids, topk_w, counts, offsets, perm, inv_perm, logits=None) -> dwdp_route_out:
    return dwdp_route_out(_ptr(topk_ids), _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(perm),
                          _ptr(inv_perm), _ptr(logits))


def dwdp_route(ctx, x, T, w_router, logit_bias, out: dwdp_route_out, ws, ws_bytes, stream=None) -> None:
    _check(ctx, lib().dwdp_route(ctx, _ptr(x), T, _ptr(w_router), _ptr(logit_bias), ctypes.byref(out),
                                 _ptr(ws), ws_bytes, _stream(stream)))


def dwdp_prefetch_layer(ctx, layer, stage, chunk_bytes, copy_streams) -> None:
    arr = (_VP * len(copy_streams))(*[_stream(s) for s in copy_streams])
    _check(ctx, lib().dwdp_prefetch_layer(ctx, layer, stage, chunk_bytes, arr, len(copy_streams)))


def dwdp_moe_layer(ctx, layer, stage, x, T, route: dwdp_route_out, out, ws, ws_bytes, stream=None) -> None:
    _check(ctx, lib().dwdp_moe_layer(ctx, layer, stage, _ptr(x), T, ctypes.byref(route), _ptr(out), _ptr(ws),
                                     ws_bytes, _stream(stream)))


def dwdp_wait_stage(ctx, stage, timeout_ms) -> int:
    """Returns the status code (OK or TIMEOUT) instead of raising on TIMEOUT."""
    rc = lib().dwdp_wait_stage(ctx, stage, timeout_ms)
    if rc not in (0, -4):
        _check(ctx, rc)
    return rc


def dwdp_stage_layer(ctx, stage) -> int:
    return lib().dwdp_stage_layer(ctx, stage)


def dwdp_device_status(ctx) -> int:
    rc = lib().dwdp_device_status(ctx)
    if rc not in (0, -6):
        _check(ctx, rc)
    return rc


def dwdp_set_phase_events(ctx, events) -> None:
    """events: a list of DWDP_PHASE_EVENTS torch.cuda.Event (timing enabled)
    or None."""
    if events is None:
        _check(ctx, lib().dwdp_set_phase_events(ctx, None, 0))
        return
    arr = (_VP * len(events))(*[e.cuda_event for e in events])
    _check(ctx, lib().dwdp_set_phase_events(ctx, arr, len(events)))


def dwdp_selftest_bounded_wait(ctx, limit_us: int, stream=None) -> None:
    """Enqueue the bounded-wait diagnostic (its wait runs out by design)."""
    _check(ctx, lib().dwdp_selftest_bounded_wait(ctx, int(limit_us), _stream(stream)))


def dwdp_grouped_gemm(ctx, epilogue, a, a_rows, K, N, row_offsets, G, bufs, buf_slot, d, stream=None) -> None:
    barr = (dwdp_pool * len(bufs))(*[dwdp_pool(_ptr(b), None, int(b.shape[0])) for b in bufs])
    bs, bsp = _i32(buf_slot)
    _check(ctx, lib().dwdp_grouped_gemm(ctx, epilogue, _ptr(a), a_rows, K, N, _ptr(row_offsets), G, barr,
                                        len(bufs), bsp, _ptr(d), _stream(stream)))


def dwdp_route_static(x, T, hidden, n_experts, top_k, w_router, logit_bias, out: dwdp_route_out,
                      stream=None) -> None:
    """Routing without a context or workspace (no device allocation)."""
    _check(None, lib().dwdp_route_static(_ptr(x), T, hidden, n_experts, top_k, _ptr(w_router), _ptr(logit_bias),
                                         ctypes.byref(out), _stream(stream)))


def dwdp_route_static_status(stream=None) -> int:
    """The error bits dwdp_route_static left on the current device (read and
    cleared after the stream's work); raises DwdpError (DEVICE_CHECK) when
    they are non-zero, with the bits in ``.bits``."""
    bits = ctypes.c_int32(0)
    rc = lib().dwdp_route_static_status(_stream(stream), ctypes.byref(bits))
    if rc != 0:
        err = DwdpError(rc, dwdp_last_error(None))
        err.bits = bits.value
        raise err
    return bits.value


WS_REGIONS = {"xp": 0, "a": 1, "y": 2, "xq": 3, "sx": 4, "sxp": 5, "aq": 6, "sa": 7, "sfx": 8, "sfa": 9}


def dwdp_workspace_region(ctx, T, region) -> tuple:
    """(byte offset, bytes) of a named intermediate in dwdp_moe_layer's workspace."""
    off, n = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(ctx, lib().dwdp_workspace_region(ctx, T, WS_REGIONS[region] if isinstance(region, str) else region,
                                            ctypes.byref(off), ctypes.byref(n)))
    return off.value, n.value


def dwdp_quantize_rows(weight_dtype, x, rows, K, codes, block_scales, row_scale, stream=None) -> None:
    _check(None, lib().dwdp_quantize_rows(weight_dtype, _ptr(x), rows, K, _ptr(codes), _ptr(block_scales),
                                          _ptr(row_scale), _stream(stream)))


def dwdp_set_expert_scales(ctx, layer, w13_scale, w2_scale, shared_w13_scale=1.0, shared_w2_scale=1.0) -> None:
    s13 = np.ascontiguousarray(w13_scale, dtype=np.float32)
    s2 = np.ascontiguousarray(w2_scale, dtype=np.float32)
    fp = ctypes.POINTER(ctypes.c_float)
    _check(ctx, lib().dwdp_set_expert_scales(ctx, layer, s13.ctypes.data_as(fp), s2.ctypes.data_as(fp),
                                             float(shared_w13_scale), float(shared_w2_scale)))


def dwdp_group_map(n_experts, n_ranks, rank):
    """(local_slot, peer_id, peer_slot) int32 arrays [E] of rank `rank` in a
    DWDP group of n_ranks ranks (host only)."""
    ls = np.empty(n_experts, dtype=np.int32)
    pid = np.empty(n_experts, dtype=np.int32)
    ps = np.empty(n_experts, dtype=np.int32)
    _check(None, lib().dwdp_group_map(n_experts, n_ranks, rank, ls.ctypes.data_as(_I32P), pid.ctypes.data_as(_I32P),
                                      ps.ctypes.data_as(_I32P)))
    return ls, pid, ps


def dwdp_plan_prefetch(n_experts, hidden, inter, local_slot, peer_id, peer_slot, n_peers, chunk_bytes,
                       weight_dtype=DTYPE_BF16):
    """The copy plan as a list of (peer, tensor, src_offset, dst_offset, nbytes)."""
    ls, lsp = _i32(local_slot)
    pi, pip = _i32(peer_id)
    ps, psp = _i32(peer_slot)
    n = ctypes.c_int64()
    _check(None, lib().dwdp_plan_prefetch(n_experts, hidden, inter, weight_dtype, lsp, pip, psp, n_peers, chunk_bytes,
                                          None, 0, ctypes.byref(n)))
    arr = (dwdp_copy_slice * max(1, n.value))()
    _check(None, lib().dwdp_plan_prefetch(n_experts, hidden, inter, weight_dtype, lsp, pip, psp, n_peers, chunk_bytes,
                                          arr, n.value, ctypes.byref(n)))
    return [(s.peer, s.tensor, s.src_offset, s.dst_offset, s.nbytes) for s in arr[: n.value]]


# ------------------------------------------------------------ helpers ----
class RouteBuffers:
    """Device tensors for dwdp_route's outputs (allocation only)."""

    def __init__(self, T: int, E: int, k: int, device="cuda", keep_logits: bool = False):
        import torch
        i32 = dict(dtype=torch.int32, device=device)
        self.T, self.E, self.k = T, E, k
        self.topk_ids = torch.empty((max(1, T), k), **i32)
        self.topk_w = torch.empty((max(1, T), k), dtype=torch.float32, device=device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.perm = torch.empty(max(1, T * k), **i32)
        self.inv_perm = torch.empty(max(1, T * k), **i32)
        self.logits = torch.empty((max(1, T), E), dtype=torch.float32, device=device) if keep_logits else None
        self.c = route_out(self.topk_ids, self.topk_w, self.counts, self.offsets, self.perm, self.inv_perm,
                           self.logits)


class Runtime:
    """One dwdp context with its stage buffers (two by default) and a
    workspace (torch allocations); methods forward to the C ABI."""

    def __init__(self, hidden, inter, n_experts, top_k, n_shared, max_tokens, n_layers, stage_slots,
                 device="cuda", weight_dtype=DTYPE_BF16, n_stages=2, flags=0):
        import torch
        self.cfg = dict(hidden=hidden, inter=inter, n_experts=n_experts, top_k=top_k, n_shared=n_shared,
                        max_tokens=max_tokens, n_layers=n_layers, stage_slots=stage_slots)
        self.weight_dtype = weight_dtype
        self.n_stages = n_stages
        if stage_slots > 0:
            b13 = weight_slot_bytes(2 * inter, hidden, weight_dtype)
            b2 = weight_slot_bytes(hidden, inter, weight_dtype)
            self.stage_w13 = [torch.empty((stage_slots, b13), dtype=torch.uint8, device=device)
                              for _ in range(n_stages)]
            self.stage_w2 = [torch.empty((stage_slots, b2), dtype=torch.uint8, device=device) for _ in range(n_stages)]
        else:
            self.stage_w13 = [None] * n_stages
            self.stage_w2 = [None] * n_stages
        self.ctx = dwdp_create(hidden, inter, n_experts, top_k, n_shared, max_tokens, n_layers, stage_slots,
                               self.stage_w13, self.stage_w2, weight_dtype, n_stages, flags)
        self.ws_bytes = max(256, dwdp_workspace_bytes(self.ctx, max_tokens))
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self._keep = {}

    def set_layer(self, layer: int, lw) -> None:
        """Map layer `layer` from an inputs.LayerWeights (pools + placement)."""
        pl = lw.placement
        local = pool(lw.local_w13, lw.local_w2)
        peers = [pool(a, b) for a, b in zip(lw.peer_w13, lw.peer_w2)]
        dwdp_set_expert_map(self.ctx, layer, local, peers, pl.local_slot, pl.peer_id, pl.peer_slot,
                            lw.shared_w13, lw.shared_w2)
        if getattr(lw, "w13_scale", None) is not None:
            dwdp_set_expert_scales(self.ctx, layer, lw.w13_scale, lw.w2_scale, lw.shared_s13, lw.shared_s2)
        self._keep[layer] = lw

    def route(self, x, w_router, bias, rb: RouteBuffers, stream=None) -> None:
        dwdp_route(self.ctx, x, x.shape[0], w_router, bias, rb.c, self.ws, self.ws_bytes, stream)

    def moe(self, layer, stage, x, rb: RouteBuffers, out, stream=None) -> None:
        dwdp_moe_layer(self.ctx, layer, stage, x, x.shape[0], rb.c, out, self.ws, self.ws_bytes, stream)

    def prefetch(self, layer, stage, chunk_bytes, copy_streams) -> None:
        dwdp_prefetch_layer(self.ctx, layer, stage, chunk_bytes, copy_streams)

    def ws_region(self, T: int, region: str):
        """The bytes of one intermediate of the last T-token layer in the
        workspace (a uint8 view, no copy)."""
        off, n = dwdp_workspace_region(self.ctx, T, region)
        return self.ws[off:off + n]

    def wait_stage(self, stage, timeout_ms) -> int:
        return dwdp_wait_stage(self.ctx, stage, timeout_ms)

    def device_status(self) -> int:
        return dwdp_device_status(self.ctx)

    def close(self) -> None:
        if self.ctx:
            dwdp_destroy(self.ctx)
            self.ctx = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
