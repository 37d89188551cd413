"""Seeded synthetic inputs for the DWDP MoE layer.

This module generates data only: it holds none of the layer's arithmetic and
is the one piece that both the CUDA path's tests/benchmark and the CPU oracle
consume.  Every tensor is drawn in fp32 from a ``torch.Generator`` seeded by
(base seed, tensor name, indices), scaled, then rounded to bf16 by
``Tensor.to`` (round-to-nearest-even).  An expert's weights depend only on
(base seed, layer, expert id), never on where the expert is placed, so the
same expert placed in several pools (redundant placement, DWDP §2) holds
identical bytes.

Shapes and distributions of the DeepSeek-R1-shaped workloads the pages
evaluate on (DWDP §5.1: DeepSeek-R1 on NVL72):
  * activations x ~ N(0, 1), [T, H]
  * router weight ~ N(0, 0.02) stored [E, H] (``router_std`` overrides it,
    e.g. 1/sqrt(H) for logits ~ N(0, 1))
  * expert weights ~ N(0, 0.02): w13 [2I, H] (gate rows, then up rows), w2 [H, I]
  * optional router bias that makes expert popularity follow a Zipf law over
    a seeded permutation of the experts.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field

import numpy as np
import torch


def seed_for(base: int, *names) -> int:
    """A 63-bit seed derived from the base seed and a tuple of names/indices."""
    h = hashlib.sha256(repr((int(base),) + tuple(names)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, std: float, seed: int, device="cpu", out: torch.Tensor | None = None):
    """N(0, std^2) drawn in fp32, rounded to bf16 (RNE).  If ``out`` is given
    the values are written into it (a bf16 view of the right shape)."""
    g = _gen(device, seed)
    v = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    if out is None:
        return v.to(torch.bfloat16)
    out.copy_(v)
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a bf16 tensor as its uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@dataclass
class LayerShape:
    T: int          # tokens
    H: int          # hidden
    I: int          # expert intermediate
    E: int          # routed experts
    k: int          # top-k
    S: int = 0      # shared experts (0 or 1)


@dataclass
class Placement:
    """Where each routed expert lives: local_slot[e] >= 0 -> resident local
    pool slot; otherwise peer_id[e] / peer_slot[e] name a peer pool slot.  A
    redundant expert has both."""
    local_slot: np.ndarray
    peer_id: np.ndarray
    peer_slot: np.ndarray
    n_local_slots: int
    n_peers: int
    peer_slots: int

    def n_remote(self) -> int:
        return int((self.local_slot < 0).sum())


def split_placement(E: int, n_local: int, n_peers: int, redundant=()) -> Placement:
    """Experts 0..n_local-1 resident (local slots 0..n_local-1); the rest
    spread over n_peers peer pools in contiguous blocks.  Each expert in
    ``redundant`` (a remote expert) also gets a local copy in an extra local
    slot after the first n_local."""
    local_slot = np.full(E, -1, dtype=np.int32)
    peer_id = np.full(E, -1, dtype=np.int32)
    peer_slot = np.full(E, -1, dtype=np.int32)
    local_slot[:n_local] = np.arange(n_local, dtype=np.int32)
    n_rem = E - n_local
    per = max(1, -(-n_rem // max(1, n_peers))) if n_rem else 0
    for r, e in enumerate(range(n_local, E)):
        peer_id[e] = r // per
        peer_slot[e] = r % per
    extra = n_local
    for e in sorted(int(v) for v in redundant):
        if local_slot[e] < 0:
            local_slot[e] = extra
            extra += 1
    return Placement(local_slot, peer_id, peer_slot, extra, n_peers if n_rem else 0, per)


def zipf_bias(E: int, s: float, seed: int) -> np.ndarray:
    """b_e = ln p_{pi(e)}, p_r = r^-s / sum_r' r'^-s (r = 1..E), pi a seeded
    permutation of the expert ids.  Returned as float32 [E]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    pi = rng.permutation(E)
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    p /= p.sum()
    b = np.empty(E, dtype=np.float64)
    b[np.arange(E)] = np.log(p[pi])
    return b.astype(np.float32)


def hottest_experts(bias: np.ndarray, n: int) -> list:
    """The n experts with the largest bias (the most popular under Zipf)."""
    return [int(e) for e in np.argsort(-bias.astype(np.float64), kind="stable")[:n]]


@dataclass
class LayerWeights:
    shape: LayerShape
    placement: Placement
    wr: torch.Tensor                      # [E, H] bf16
    bias: torch.Tensor | None             # [E] f32
    local_w13: torch.Tensor               # [n_local_slots, 2I, H]
    local_w2: torch.Tensor                # [n_local_slots, H, I]
    peer_w13: list = field(default_factory=list)   # [n_peers] of [peer_slots, 2I, H]
    peer_w2: list = field(default_factory=list)    # [n_peers] of [peer_slots, H, I]
    shared_w13: torch.Tensor | None = None         # [2I, H]
    shared_w2: torch.Tensor | None = None          # [H, I]


def make_layer(shape: LayerShape, placement: Placement, base_seed: int, layer: int,
               device="cpu", router_std: float = 0.02, weight_std: float = 0.02,
               bias: np.ndarray | None = None) -> LayerWeights:
    """All weights of one MoE layer, written into the pools the placement
    names."""
    H, I, E = shape.H, shape.I, shape.E
    bf = torch.bfloat16
    wr = randn_bf16((E, H), router_std, seed_for(base_seed, "Wr", layer), device)
    lw13 = torch.empty((max(1, placement.n_local_slots), 2 * I, H), dtype=bf, device=device)
    lw2 = torch.empty((max(1, placement.n_local_slots), H, I), dtype=bf, device=device)
    pw13 = [torch.empty((placement.peer_slots, 2 * I, H), dtype=bf, device=device)
            for _ in range(placement.n_peers)]
    pw2 = [torch.empty((placement.peer_slots, H, I), dtype=bf, device=device)
           for _ in range(placement.n_peers)]
    for e in range(E):
        dsts13, dsts2 = [], []
        if placement.local_slot[e] >= 0:
            dsts13.append(lw13[placement.local_slot[e]])
            dsts2.append(lw2[placement.local_slot[e]])
        if placement.peer_id[e] >= 0:
            dsts13.append(pw13[placement.peer_id[e]][placement.peer_slot[e]])
            dsts2.append(pw2[placement.peer_id[e]][placement.peer_slot[e]])
        if not dsts13:
            raise ValueError(f"expert {e} has no placement")
        randn_bf16((2 * I, H), weight_std, seed_for(base_seed, "W13", layer, e), device, out=dsts13[0])
        randn_bf16((H, I), weight_std, seed_for(base_seed, "W2", layer, e), device, out=dsts2[0])
        for d in dsts13[1:]:
            d.copy_(dsts13[0])
        for d in dsts2[1:]:
            d.copy_(dsts2[0])
    sw13 = sw2 = None
    if shape.S:
        sw13 = randn_bf16((2 * I, H), weight_std, seed_for(base_seed, "W13s", layer), device)
        sw2 = randn_bf16((H, I), weight_std, seed_for(base_seed, "W2s", layer), device)
    bt = None
    if bias is not None:
        bt = torch.as_tensor(np.asarray(bias, dtype=np.float32)).to(device)
    return LayerWeights(shape, placement, wr, bt, lw13, lw2, pw13, pw2, sw13, sw2)


@dataclass
class LayerWeightsFp8(LayerWeights):
    """As LayerWeights, with uint8 E4M3 weight codes in the pools and one
    scale per expert tensor (w = code * scale)."""
    w13_scale: np.ndarray | None = None   # [E] float32
    w2_scale: np.ndarray | None = None    # [E] float32
    shared_s13: float = 1.0
    shared_s2: float = 1.0


def e4m3_codes(shape, seed: int, device="cpu", out: torch.Tensor | None = None) -> torch.Tensor:
    """Synthetic E4M3 weight codes: N(0, 1) drawn in fp32 and converted by
    torch's float8_e4m3fn cast, returned (or written) as uint8."""
    g = _gen(device, seed)
    v = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    c = v.to(torch.float8_e4m3fn).view(torch.uint8)
    if out is None:
        return c
    out.copy_(c)
    return out


def make_layer_fp8(shape: LayerShape, placement: Placement, base_seed: int, layer: int, device="cpu",
                   router_std: float = 0.02, bias: np.ndarray | None = None) -> LayerWeightsFp8:
    """One MoE layer with E4M3 expert weights: codes ~ E4M3(N(0, 1)) and a
    per-tensor scale ~ 0.02 * U(0.8, 1.2) per expert, so w = code * scale has
    roughly the bf16 layers' N(0, 0.02^2) spread.  Codes and scales depend only
    on (base seed, layer, expert), not on placement."""
    H, I, E = shape.H, shape.I, shape.E
    u8 = torch.uint8
    wr = randn_bf16((E, H), router_std, seed_for(base_seed, "Wr", layer), device)
    lw13 = torch.empty((max(1, placement.n_local_slots), 2 * I, H), dtype=u8, device=device)
    lw2 = torch.empty((max(1, placement.n_local_slots), H, I), dtype=u8, device=device)
    pw13 = [torch.empty((placement.peer_slots, 2 * I, H), dtype=u8, device=device) for _ in range(placement.n_peers)]
    pw2 = [torch.empty((placement.peer_slots, H, I), dtype=u8, device=device) for _ in range(placement.n_peers)]
    for e in range(E):
        d13, d2 = [], []
        if placement.local_slot[e] >= 0:
            d13.append(lw13[placement.local_slot[e]])
            d2.append(lw2[placement.local_slot[e]])
        if placement.peer_id[e] >= 0:
            d13.append(pw13[placement.peer_id[e]][placement.peer_slot[e]])
            d2.append(pw2[placement.peer_id[e]][placement.peer_slot[e]])
        e4m3_codes((2 * I, H), seed_for(base_seed, "W13q", layer, e), device, out=d13[0])
        e4m3_codes((H, I), seed_for(base_seed, "W2q", layer, e), device, out=d2[0])
        for d in d13[1:]:
            d.copy_(d13[0])
        for d in d2[1:]:
            d.copy_(d2[0])
    s13, s2, ss13, ss2 = expert_scales("fp8", base_seed, layer, E)
    sw13 = sw2 = None
    if shape.S:
        sw13, sw2 = expert_weights("fp8", shape, base_seed, layer, None, device)
    else:
        ss13 = ss2 = 1.0
    bt = None
    if bias is not None:
        bt = torch.as_tensor(np.asarray(bias, dtype=np.float32)).to(device)
    return LayerWeightsFp8(shape, placement, wr, bt, lw13, lw2, pw13, pw2, sw13, sw2, s13, s2, ss13, ss2)


# ----------------------------------------------------------------- NVFP4 --
# Synthetic NVFP4 weights are drawn directly as codes: E2M1 magnitude codes
# 0..7 with these probabilities (a bell-shaped spread over 0 .. 6) and a
# uniform sign, E4M3 block-scale codes uniform in [0x30, 0x48) (0.5 .. 3.75),
# and a tensor scale ~ 0.004 * U(0.8, 1.2), which puts the weights' spread
# near the bf16 layers' 0.02.
E2M1_CODE_P = (0.10, 0.18, 0.18, 0.15, 0.14, 0.12, 0.08, 0.05)


@dataclass
class LayerWeightsNvfp4(LayerWeights):
    """As LayerWeights, with NVFP4 pool slots (uint8 [slots][slot bytes]:
    packed codes then block-scale chunks, as dwdp.h lays them out) and one
    tensor scale per expert tensor."""
    w13_scale: np.ndarray | None = None   # [E] float32
    w2_scale: np.ndarray | None = None    # [E] float32
    shared_s13: float = 1.0
    shared_s2: float = 1.0


def nvfp4_codes(rows: int, K: int, seed: int, device="cpu") -> tuple:
    """(codes uint8 [rows][K], one E2M1 code per byte; block scales uint8
    [rows][K / 16], E4M3 codes) of one synthetic expert tensor."""
    g = _gen(device, seed)
    edges = torch.tensor(np.cumsum(E2M1_CODE_P)[:-1], dtype=torch.float32, device=device)
    mag = torch.bucketize(torch.rand((rows, K), generator=g, device=device), edges).to(torch.uint8)
    sign = (torch.rand((rows, K), generator=g, device=device) < 0.5).to(torch.uint8) << 3
    sf = torch.randint(0x30, 0x48, (rows, K // 16), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    return mag | sign, sf


def pack_nvfp4(codes: torch.Tensor, sf: torch.Tensor) -> torch.Tensor:
    """One pool slot (uint8, rows * K * 9 / 16 bytes) from math-layout codes
    [rows][K] and block scales [rows][K / 16]: codes two per byte (element 2i
    in the low nibble), then the scales in 512-byte chunks per (128-row block
    rb, 64-element K step ks), row 128 rb + 32 m1 + m0 and block kb of the step
    at byte 16 m0 + 4 m1 + kb.  rows a multiple of 128, K of 64."""
    R, K = codes.shape
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    chunks = sf.reshape(R // 128, 4, 32, K // 64, 4).permute(0, 3, 2, 1, 4)
    return torch.cat([packed.reshape(-1), chunks.reshape(-1)])


def unpack_nvfp4(slot: torch.Tensor, rows: int, K: int) -> tuple:
    """Inverse of pack_nvfp4: (codes uint8 [rows][K], block scales uint8
    [rows][K / 16]) as numpy arrays from one slot's bytes."""
    b = slot.reshape(-1).to(torch.uint8)
    n = rows * K // 2
    packed = b[:n].reshape(rows, K // 2)
    codes = torch.stack([packed & 15, packed >> 4], dim=2).reshape(rows, K)
    sf = b[n:n + rows * K // 16].reshape(rows // 128, K // 64, 32, 4, 4).permute(0, 3, 2, 1, 4)
    return codes.numpy(), sf.reshape(rows, K // 16).numpy()


def make_layer_nvfp4(shape: LayerShape, placement: Placement, base_seed: int, layer: int, device="cpu",
                     router_std: float = 0.02, bias: np.ndarray | None = None) -> LayerWeightsNvfp4:
    """One MoE layer with NVFP4 expert weights in the pools the placement
    names.  Codes and scales depend only on (base seed, layer, expert)."""
    H, I, E = shape.H, shape.I, shape.E
    u8 = torch.uint8
    b13, b2 = 2 * I * H * 9 // 16, H * I * 9 // 16
    wr = randn_bf16((E, H), router_std, seed_for(base_seed, "Wr", layer), device)
    lw13 = torch.empty((max(1, placement.n_local_slots), b13), dtype=u8, device=device)
    lw2 = torch.empty((max(1, placement.n_local_slots), b2), dtype=u8, device=device)
    pw13 = [torch.empty((placement.peer_slots, b13), dtype=u8, device=device) for _ in range(placement.n_peers)]
    pw2 = [torch.empty((placement.peer_slots, b2), dtype=u8, device=device) for _ in range(placement.n_peers)]
    for e in range(E):
        d13, d2 = [], []
        if placement.local_slot[e] >= 0:
            d13.append(lw13[placement.local_slot[e]])
            d2.append(lw2[placement.local_slot[e]])
        if placement.peer_id[e] >= 0:
            d13.append(pw13[placement.peer_id[e]][placement.peer_slot[e]])
            d2.append(pw2[placement.peer_id[e]][placement.peer_slot[e]])
        c13, c2 = expert_weights("nvfp4", shape, base_seed, layer, e, device)
        p13, p2 = pack_nvfp4(*c13), pack_nvfp4(*c2)
        for d in d13:
            d.copy_(p13)
        for d in d2:
            d.copy_(p2)
    s13, s2, ss13, ss2 = expert_scales("nvfp4", base_seed, layer, E)
    sw13 = sw2 = None
    if shape.S:
        c13, c2 = expert_weights("nvfp4", shape, base_seed, layer, None, device)
        sw13, sw2 = pack_nvfp4(*c13), pack_nvfp4(*c2)
    else:
        ss13 = ss2 = 1.0
    bt = None
    if bias is not None:
        bt = torch.as_tensor(np.asarray(bias, dtype=np.float32)).to(device)
    return LayerWeightsNvfp4(shape, placement, wr, bt, lw13, lw2, pw13, pw2, sw13, sw2, s13, s2, ss13, ss2)


def expert_weights(wdtype: str, shape: LayerShape, base_seed: int, layer: int, e=None, device="cpu"):
    """One expert's weights in math layout, drawn exactly as the layer
    builders draw them (e = None: the shared expert): bf16 (w13, w2) tensors
    (the default weight spread 0.02); E4M3 (w13, w2) uint8 code tensors;
    NVFP4 ((codes13, scales13), (codes2, scales2)) as nvfp4_codes returns."""
    H, I = shape.H, shape.I
    idx = (layer,) if e is None else (layer, e)
    sfx = "s" if e is None else ""
    if wdtype == "bf16":
        return (randn_bf16((2 * I, H), 0.02, seed_for(base_seed, "W13" + sfx, *idx), device),
                randn_bf16((H, I), 0.02, seed_for(base_seed, "W2" + sfx, *idx), device))
    if wdtype == "fp8":
        return (e4m3_codes((2 * I, H), seed_for(base_seed, "W13q" + sfx, *idx), device),
                e4m3_codes((H, I), seed_for(base_seed, "W2q" + sfx, *idx), device))
    if wdtype == "nvfp4":
        return (nvfp4_codes(2 * I, H, seed_for(base_seed, "W13f" + sfx, *idx), device),
                nvfp4_codes(H, I, seed_for(base_seed, "W2f" + sfx, *idx), device))
    raise ValueError(wdtype)


def expert_scales(wdtype: str, base_seed: int, layer: int, E: int) -> tuple:
    """(w13 scales [E], w2 scales [E], shared w13 scale, shared w2 scale) of
    an E4M3 or NVFP4 layer, as the layer builders draw them."""
    base, tag, shared = {"fp8": (0.02, "fp8_scales", (0.02, 0.021)),
                         "nvfp4": (0.004, "nvfp4_scales", (0.004, 0.0042))}[wdtype]
    rng = np.random.Generator(np.random.PCG64(seed_for(base_seed, tag, layer)))
    s13 = (base * rng.uniform(0.8, 1.2, E)).astype(np.float32)
    s2 = (base * rng.uniform(0.8, 1.2, E)).astype(np.float32)
    return s13, s2, float(np.float32(shared[0])), float(np.float32(shared[1]))


def make_tokens(T: int, H: int, base_seed: int, step: int = 0, device="cpu") -> torch.Tensor:
    """Activations x ~ N(0, 1) as bf16 [T, H]."""
    return randn_bf16((T, H), 1.0, seed_for(base_seed, "x", step), device)


def step_token_counts(n_steps: int, lo: int, hi: int, base_seed: int) -> list:
    """Per-step token counts, integers uniform in [lo, hi] inclusive."""
    rng = np.random.Generator(np.random.PCG64(seed_for(base_seed, "T_steps")))
    return [int(v) for v in rng.integers(lo, hi + 1, size=n_steps)]


# The workloads, by what they are.  R1 = DeepSeek-R1 MoE layer shapes.
def tiny_layer() -> tuple:
    """T=64, H=256, I=128, E=8, top-2, no shared expert; experts 0-3 local,
    4-7 in one separate pool."""
    shape = LayerShape(T=64, H=256, I=128, E=8, k=2, S=0)
    return shape, split_placement(8, 4, 1)


def r1_layer(T: int = 8192) -> tuple:
    """R1-shaped layer: H=7168, I=2048, 256 routed top-8 + 1 shared; 64 local
    experts, 192 over three emulated peer pools of 64."""
    shape = LayerShape(T=T, H=7168, I=2048, E=256, k=8, S=1)
    return shape, split_placement(256, 64, 3)


def sqrt_inv(H: int) -> float:
    return 1.0 / math.sqrt(H)
