"""CPU oracle of one DWDP MoE layer: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
(``moe_expert_grouped_split_gb300``) and the CUDA path never imports it.

The arithmetic lives in ``dwdp_oracle.c`` (plain loops, fp64); this module
compiles it with gcc, loads it with ctypes and marshals numpy arrays.  The
prefetch-plan oracle is plain Python in ``prefetch_plan.py``.

Sources: "DWDP: Distributed Weight Data Parallelism for High-Performance LLM
Inference on NVL72" (summary pages), §2 Methodology Overview (placement does
not change the layer's result; redundant placement allowed), §4.2 (grouped
GEMM over several weight buffers) and §4.3.2 (fixed-size slices issued
round-robin).  The router and the expert FFN are not printed on the pages;
``dwdp_oracle.c`` states the reading taken.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, invariants and special cases) and by the mutation
test in ``tests/test_oracle_mutants.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from pathlib import Path

import numpy as np

from .prefetch_plan import group_map, plan_prefetch, stage_slots  # noqa: F401

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "dwdp_oracle.c"
_BUILD = _HERE / "_build"


def build(mutant: int = 0, out_dir: Path | None = None, force: bool = False) -> Path:
    """Compile the oracle (optionally with one planted mistake) and return the
    path of the shared library.  gcc, -O2, OpenMP over tokens."""
    out_dir = Path(out_dir) if out_dir is not None else _BUILD
    out_dir.mkdir(parents=True, exist_ok=True)
    name = "liboracle.so" if mutant == 0 else f"liboracle_m{mutant}.so"
    lib = out_dir / name
    if force or not lib.exists() or lib.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = tempfile.NamedTemporaryFile(dir=out_dir, suffix=".so", delete=False).name
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               f"-DORACLE_MUTANT={mutant}", str(_SRC), "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


_U16P = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_F64P = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_F32P = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_I32P = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_I64P = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_I64 = ctypes.c_int64
_U8P = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


class Oracle:
    """ctypes view of one build of ``dwdp_oracle.c``."""

    def __init__(self, lib_path: Path | str | None = None):
        self.path = Path(lib_path) if lib_path is not None else build()
        L = ctypes.CDLL(str(self.path))
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_round_bf16.restype = ctypes.c_uint16
        L.oracle_round_bf16.argtypes = [ctypes.c_double]
        L.oracle_router_logits.restype = None
        L.oracle_router_logits.argtypes = [_U16P, _I64, _I64, _U16P, _I64, ctypes.c_void_p, _F64P]
        L.oracle_topk.restype = None
        L.oracle_topk.argtypes = [_F64P, _I64, _I64, _I64, ctypes.c_int, _I32P, _F64P]
        L.oracle_group.restype = None
        L.oracle_group.argtypes = [_I32P, _I64, _I64, _I64, _I32P, _I32P, _I32P, _I32P]
        L.oracle_expert_ffn.restype = None
        L.oracle_expert_ffn.argtypes = [_U16P, _I64, _I64, _U16P, _U16P, ctypes.c_int, _F64P]
        L.oracle_moe_tokens.restype = None
        L.oracle_moe_tokens.argtypes = [
            _U16P, _I64, _I64, _I64, _I64P, _I64, _I32P, _F64P,
            ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, _F64P]
        L.oracle_grouped_gemm.restype = None
        L.oracle_grouped_gemm.argtypes = [_U16P, _I64, _I32P, _I64, ctypes.POINTER(ctypes.c_void_p), _I64,
                                          ctypes.c_int, _F64P]
        L.oracle_e4m3_to_double.restype = ctypes.c_double
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        L.oracle_quantize_row_e4m3.restype = None
        L.oracle_quantize_row_e4m3.argtypes = [_F32P, _I64, _U8P, ctypes.POINTER(ctypes.c_float)]
        L.oracle_moe_tokens_fp8.restype = None
        L.oracle_moe_tokens_fp8.argtypes = [
            _U16P, _I64, _I64, _I64, _I64P, _I64, _I32P, _F64P,
            ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), _F32P, _F32P,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_float, ctypes.c_int, _F64P]
        L.oracle_e2m1_to_double.restype = ctypes.c_double
        L.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_encode.restype = ctypes.c_uint8
        L.oracle_e2m1_encode.argtypes = [ctypes.c_double]
        L.oracle_quantize_row_nvfp4.restype = None
        L.oracle_quantize_row_nvfp4.argtypes = [_F32P, _I64, _U8P, _U8P, ctypes.POINTER(ctypes.c_float)]
        L.oracle_moe_tokens_nvfp4.restype = None
        vpp = ctypes.POINTER(ctypes.c_void_p)
        L.oracle_moe_tokens_nvfp4.argtypes = [
            _U16P, _I64, _I64, _I64, _I64P, _I64, _I32P, _F64P,
            vpp, vpp, _F32P, vpp, vpp, _F32P,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
            ctypes.c_int, _F64P]
        L.oracle_e4m3_linear.restype = None
        L.oracle_e4m3_linear.argtypes = [_U8P, _F32P, _I64, _I64, _U8P, ctypes.c_float, _I64, ctypes.c_int,
                                         ctypes.c_int, _F64P]
        L.oracle_nvfp4_linear.restype = None
        L.oracle_nvfp4_linear.argtypes = [_U8P, _U8P, _F32P, _I64, _I64, _U8P, _U8P, ctypes.c_float, _I64,
                                          ctypes.c_int, ctypes.c_int, _F64P]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        self.lib = L

    # -- bf16 -------------------------------------------------------------
    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(int(bits))

    def round_bf16(self, v: float) -> int:
        return int(self.lib.oracle_round_bf16(float(v)))

    def round_bf16_array(self, v: np.ndarray) -> np.ndarray:
        flat = np.asarray(v, dtype=np.float64).ravel()
        out = np.fromiter((self.lib.oracle_round_bf16(float(a)) for a in flat),
                          dtype=np.uint16, count=flat.size)
        return out.reshape(np.shape(v))

    # -- routing ----------------------------------------------------------
    def router_logits(self, x, wr, bias=None) -> np.ndarray:
        """fp64 logits z[t, e] = x[t] . Wr[:, e] (+ bias[e])."""
        x, wr = _u16(x), _u16(wr)
        T, H = x.shape
        E, H2 = wr.shape
        assert H == H2
        z = np.zeros((T, E), dtype=np.float64)
        b = None
        if bias is not None:
            b = np.ascontiguousarray(bias, dtype=np.float32)
            assert b.shape == (E,)
        self.lib.oracle_router_logits(x, T, H, wr, E,
                                      b.ctypes.data if b is not None else None, z)
        return z

    def topk(self, z, k: int, decide_fp32: bool = True):
        """Chosen experts (ascending id) and renormalised fp64 weights."""
        z = np.ascontiguousarray(z, dtype=np.float64)
        T, E = z.shape
        if not (1 <= k <= E):
            raise ValueError("need 1 <= k <= E")
        ids = np.zeros((T, k), dtype=np.int32)
        w = np.zeros((T, k), dtype=np.float64)
        self.lib.oracle_topk(z, T, E, k, int(bool(decide_fp32)), ids, w)
        return ids, w

    def group(self, ids, E: int):
        """counts [E], offsets [E+1], perm [T*k], inv [T*k]."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T, k = ids.shape
        counts = np.zeros(E, dtype=np.int32)
        offsets = np.zeros(E + 1, dtype=np.int32)
        perm = np.zeros(T * k, dtype=np.int32)
        inv = np.zeros(T * k, dtype=np.int32)
        self.lib.oracle_group(ids, T, E, k, counts, offsets, perm, inv)
        return counts, offsets, perm, inv

    def route(self, x, wr, bias, k: int, decide_fp32: bool = True) -> dict:
        z = self.router_logits(x, wr, bias)
        ids, w = self.topk(z, k, decide_fp32)
        counts, offsets, perm, inv = self.group(ids, z.shape[1])
        return dict(logits=z, ids=ids, w=w, counts=counts, offsets=offsets,
                    perm=perm, inv=inv)

    # -- FFN --------------------------------------------------------------
    def expert_ffn(self, xrow, w13, w2, mirrored: bool = True) -> np.ndarray:
        xrow, w13, w2 = _u16(xrow), _u16(w13), _u16(w2)
        H = xrow.shape[-1]
        I = w13.shape[0] // 2
        assert w13.shape == (2 * I, H) and w2.shape == (H, I)
        y = np.zeros(H, dtype=np.float64)
        self.lib.oracle_expert_ffn(xrow, H, I, w13, w2, int(bool(mirrored)), y)
        return y

    def moe_tokens(self, x, tokens, ids, w, expert_w13, expert_w2,
                   shared_w13=None, shared_w2=None, mirrored: bool = True) -> np.ndarray:
        """Layer output rows for the given tokens (fp64; bf16-valued when
        mirrored).  expert_w13[e] / expert_w2[e]: expert e's weights, already
        resolved through the placement map (see ``resolve_experts``)."""
        x = _u16(x)
        T, H = x.shape
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        w = np.ascontiguousarray(w, dtype=np.float64)
        k = ids.shape[1]
        tok = np.ascontiguousarray(tokens, dtype=np.int64)
        E = len(expert_w13)
        I = None
        keep = []
        p13 = (ctypes.c_void_p * E)()
        p2 = (ctypes.c_void_p * E)()
        for e in range(E):
            a13, a2 = expert_w13[e], expert_w2[e]
            if a13 is None:
                p13[e] = None
                p2[e] = None
                continue
            a13, a2 = _u16(a13), _u16(a2)
            I = a13.shape[0] // 2
            assert a13.shape == (2 * I, H) and a2.shape == (H, I)
            keep += [a13, a2]
            p13[e] = a13.ctypes.data
            p2[e] = a2.ctypes.data
        used = np.unique(ids[tok]) if tok.size else np.zeros(0, dtype=np.int32)
        for e in used:
            if p13[int(e)] is None:
                raise ValueError(f"expert {int(e)} is routed to but has no weights")
        s13 = s2 = None
        if shared_w13 is not None:
            s13, s2 = _u16(shared_w13), _u16(shared_w2)
            I = s13.shape[0] // 2
        if I is None:
            raise ValueError("no expert weights given")
        out = np.zeros((tok.size, H), dtype=np.float64)
        self.lib.oracle_moe_tokens(x, H, I, k, tok, tok.size, ids, w, p13, p2,
                                   s13.ctypes.data if s13 is not None else None,
                                   s2.ctypes.data if s2 is not None else None,
                                   int(bool(mirrored)), out)
        del keep
        return out

    def grouped_gemm(self, a, row_offsets, b_list, N: int, epilogue: int) -> np.ndarray:
        """fp64 result [rows, N] of the grouped GEMM (rows outside every
        group stay 0).  b_list[g]: group g's weights [N or 2N][K] uint16."""
        a = _u16(a)
        rows, K = a.shape
        off = np.ascontiguousarray(row_offsets, dtype=np.int32)
        G = off.size - 1
        assert len(b_list) == G
        keep = [_u16(b) for b in b_list]
        ptrs = (ctypes.c_void_p * max(1, G))(*[b.ctypes.data for b in keep])
        d = np.zeros((rows, N), dtype=np.float64)
        self.lib.oracle_grouped_gemm(a, K, off, G, ptrs, N, int(epilogue), d)
        return d

    # -- FP8 (E4M3) ---------------------------------------------------------
    def e4m3_encode(self, v: float) -> int:
        return int(self.lib.oracle_e4m3_encode(float(v)))

    def e4m3_decode(self, code: int) -> float:
        return self.lib.oracle_e4m3_to_double(int(code))

    def quantize_row_e4m3(self, row) -> tuple:
        """(codes uint8 [n], scale) of one row of binary32 values."""
        r = np.ascontiguousarray(row, dtype=np.float32)
        codes = np.zeros(r.size, dtype=np.uint8)
        s = ctypes.c_float()
        self.lib.oracle_quantize_row_e4m3(r, r.size, codes, ctypes.byref(s))
        return codes, float(s.value)

    def moe_tokens_fp8(self, x, tokens, ids, w, expert_w13, expert_w2, w13_scale, w2_scale,
                       shared_w13=None, shared_w2=None, shared_s13=1.0, shared_s2=1.0,
                       mirrored: bool = True) -> np.ndarray:
        """Layer output rows with E4M3 expert weights (uint8 codes, per-tensor
        scales) and per-row E4M3 activations; see dwdp_oracle.c."""
        x = _u16(x)
        T, H = x.shape
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        w = np.ascontiguousarray(w, dtype=np.float64)
        k = ids.shape[1]
        tok = np.ascontiguousarray(tokens, dtype=np.int64)
        E = len(expert_w13)
        keep, I = [], None
        p13 = (ctypes.c_void_p * E)()
        p2 = (ctypes.c_void_p * E)()
        for e in range(E):
            if expert_w13[e] is None:
                continue
            a13 = np.ascontiguousarray(expert_w13[e], dtype=np.uint8)
            a2 = np.ascontiguousarray(expert_w2[e], dtype=np.uint8)
            I = a13.shape[0] // 2
            assert a13.shape == (2 * I, H) and a2.shape == (H, I)
            keep += [a13, a2]
            p13[e], p2[e] = a13.ctypes.data, a2.ctypes.data
        for e in (np.unique(ids[tok]) if tok.size else []):
            if p13[int(e)] is None:
                raise ValueError(f"expert {int(e)} is routed to but has no weights")
        s13 = s2 = None
        if shared_w13 is not None:
            s13 = np.ascontiguousarray(shared_w13, dtype=np.uint8)
            s2 = np.ascontiguousarray(shared_w2, dtype=np.uint8)
            I = s13.shape[0] // 2
        sc13 = np.ascontiguousarray(w13_scale, dtype=np.float32)
        sc2 = np.ascontiguousarray(w2_scale, dtype=np.float32)
        out = np.zeros((tok.size, H), dtype=np.float64)
        self.lib.oracle_moe_tokens_fp8(x, H, I, k, tok, tok.size, ids, w, p13, p2, sc13, sc2,
                                       s13.ctypes.data if s13 is not None else None,
                                       s2.ctypes.data if s2 is not None else None,
                                       float(shared_s13), float(shared_s2), int(bool(mirrored)), out)
        del keep
        return out

    # -- NVFP4 (E2M1 codes, E4M3 scales per 16-element block) ---------------
    def e2m1_encode(self, v: float) -> int:
        return int(self.lib.oracle_e2m1_encode(float(v)))

    def e2m1_decode(self, code: int) -> float:
        return self.lib.oracle_e2m1_to_double(int(code))

    def quantize_row_nvfp4(self, row) -> tuple:
        """(codes uint8 [n] one per element, block scales uint8 [n / 16],
        row scale) of one row of binary32 values (n a multiple of 16)."""
        r = np.ascontiguousarray(row, dtype=np.float32)
        if r.size % 16:
            raise ValueError("NVFP4 rows are whole 16-element blocks")
        codes = np.zeros(r.size, dtype=np.uint8)
        sf = np.zeros(r.size // 16, dtype=np.uint8)
        s = ctypes.c_float()
        self.lib.oracle_quantize_row_nvfp4(r, r.size, codes, sf, ctypes.byref(s))
        return codes, sf, float(s.value)

    def moe_tokens_nvfp4(self, x, tokens, ids, w, w13, w13_sf, w13_scale, w2, w2_sf, w2_scale,
                         shared=None, mirrored: bool = True) -> np.ndarray:
        """Layer output rows with NVFP4 expert weights.  Per expert e (None for
        experts no selected token uses): w13[e] codes [2I][H] and w13_sf[e]
        block scales [2I][H/16], w2[e] codes [H][I] and w2_sf[e] [H][I/16],
        one code or E4M3 scale per byte; w13_scale / w2_scale [E] tensor
        scales.  shared = (w13, w13_sf, s13, w2, w2_sf, s2) or None.
        Activations are quantized per row; see dwdp_oracle.c."""
        x = _u16(x)
        T, H = x.shape
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        w = np.ascontiguousarray(w, dtype=np.float64)
        k = ids.shape[1]
        tok = np.ascontiguousarray(tokens, dtype=np.int64)
        E = len(w13)
        keep, I = [], None
        ptrs = [(ctypes.c_void_p * E)() for _ in range(4)]
        for e in range(E):
            if w13[e] is None:
                continue
            arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (w13[e], w13_sf[e], w2[e], w2_sf[e])]
            I = arrs[0].shape[0] // 2
            assert arrs[0].shape == (2 * I, H) and arrs[1].shape == (2 * I, H // 16)
            assert arrs[2].shape == (H, I) and arrs[3].shape == (H, I // 16)
            keep += arrs
            for p, a in zip(ptrs, arrs):
                p[e] = a.ctypes.data
        for e in (np.unique(ids[tok]) if tok.size else []):
            if ptrs[0][int(e)] is None:
                raise ValueError(f"expert {int(e)} is routed to but has no weights")
        sh = [None] * 4
        ss13 = ss2 = 1.0
        if shared is not None:
            sh = [np.ascontiguousarray(shared[i], dtype=np.uint8) for i in (0, 1, 3, 4)]
            ss13, ss2 = float(shared[2]), float(shared[5])
            I = sh[0].shape[0] // 2
        if H % 16 or (I is not None and I % 16):
            raise ValueError("NVFP4 needs H and I multiples of 16")
        sc13 = np.ascontiguousarray(w13_scale, dtype=np.float32)
        sc2 = np.ascontiguousarray(w2_scale, dtype=np.float32)
        out = np.zeros((tok.size, H), dtype=np.float64)
        dp = lambda a: a.ctypes.data if a is not None else None
        self.lib.oracle_moe_tokens_nvfp4(x, H, I, k, tok, tok.size, ids, w, ptrs[0], ptrs[1], sc13, ptrs[2], ptrs[3],
                                         sc2, dp(sh[0]), dp(sh[1]), ss13, dp(sh[2]), dp(sh[3]), ss2,
                                         int(bool(mirrored)), out)
        del keep
        return out

    def e4m3_linear(self, codes, row_scale, w, w_scale, epilogue: int = 0, mirrored: bool = True) -> np.ndarray:
        """One E4M3 linear layer on rows given as codes [n][K] and row scales
        [n], against weight codes w [N][K] (epilogue 1: [2N][K], gate rows
        then up rows) with tensor scale w_scale.  Epilogue 0: the product;
        1: SiLU(gate) * up.  fp64, bf16-rounded when mirrored."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        rs = np.ascontiguousarray(row_scale, dtype=np.float32)
        w = np.ascontiguousarray(w, dtype=np.uint8)
        n, K = codes.shape
        N = w.shape[0] // (2 if epilogue == 1 else 1)
        assert w.shape[1] == K and rs.shape == (n,)
        out = np.zeros((n, N), dtype=np.float64)
        self.lib.oracle_e4m3_linear(codes, rs, n, K, w, float(w_scale), N, int(epilogue), int(bool(mirrored)), out)
        return out

    def nvfp4_linear(self, codes, sf, row_scale, w, wsf, w_scale, epilogue: int = 0,
                     mirrored: bool = True) -> np.ndarray:
        """One NVFP4 linear layer on rows given as codes [n][K] (one E2M1
        code per byte), block scales [n][K/16] and row scales [n], against
        weights w [N][K] (epilogue 1: [2N][K], gate rows then up rows) with
        block scales wsf and tensor scale w_scale.  Epilogue 0: the product;
        1: SiLU(gate) * up.  fp64, bf16-rounded when mirrored."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        sf = np.ascontiguousarray(sf, dtype=np.uint8)
        rs = np.ascontiguousarray(row_scale, dtype=np.float32)
        w = np.ascontiguousarray(w, dtype=np.uint8)
        wsf = np.ascontiguousarray(wsf, dtype=np.uint8)
        n, K = codes.shape
        N = w.shape[0] // (2 if epilogue == 1 else 1)
        assert w.shape[1] == K and sf.shape == (n, K // 16) and wsf.shape == (w.shape[0], K // 16)
        assert rs.shape == (n,)
        out = np.zeros((n, N), dtype=np.float64)
        self.lib.oracle_nvfp4_linear(codes, sf, rs, n, K, w, wsf, float(w_scale), N, int(epilogue),
                                     int(bool(mirrored)), out)
        return out

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.oracle_set_num_threads(int(n))


def resolve_experts(n_experts, local_pool, peer_pools, local_slot, peer_id, peer_slot):
    """Expert weights through a placement map (DWDP §2: placement need not be
    disjoint; a redundant expert is read from its local copy).

    local_pool / peer_pools[p]: (w13 [slots, 2I, H], w2 [slots, H, I]) uint16
    arrays.  local_slot[e] >= 0 selects the local copy; otherwise
    peer_id[e] / peer_slot[e] select the peer copy.  Returns two lists
    (expert_w13, expert_w2) indexed by expert."""
    w13s, w2s = [], []
    for e in range(n_experts):
        if local_slot[e] >= 0:
            w13s.append(local_pool[0][local_slot[e]])
            w2s.append(local_pool[1][local_slot[e]])
        elif peer_id[e] >= 0:
            pool = peer_pools[peer_id[e]]
            w13s.append(pool[0][peer_slot[e]])
            w2s.append(pool[1][peer_slot[e]])
        else:
            raise ValueError(f"expert {e} has no copy")
    return w13s, w2s


_default: Oracle | None = None


def default() -> Oracle:
    """The unmutated oracle, built on first use."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
