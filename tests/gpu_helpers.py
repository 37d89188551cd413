"""Shared pieces of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, and compare.

Tolerances (floating point): the layer output is bf16; with
rel_i = |g_i - o_i| / max(|o_i|, rms(o)) the bar is max rel <= 2e-2 and mean
absolute error <= 1e-3 against the oracle's mirrored mode (same bf16
rounding points as the kernels).  Integer outputs (expert ids, counts,
offsets, permutations) are compared bit for bit; the only exemption is a
token whose choice is a near-tie in fp32 (see ``near_tie_tokens``), for
which the GPU's choice is checked for validity instead.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_expert_grouped_split_gb300 import binding as B
from moe_expert_grouped_split_gb300 import inputs as I

REL_MAX = 2e-2
MAE_MAX = 1e-3


def rel_metrics(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    denom = np.maximum(np.abs(ref), rms if rms > 0 else 1e-30)
    rel = np.abs(got - ref) / denom
    return float(rel.max(initial=0.0)), float(np.abs(got - ref).mean()) if ref.size else 0.0


def assert_close(got, ref, rel_max=REL_MAX, mae_max=MAE_MAX, what=""):
    r, m = rel_metrics(got, ref)
    assert r <= rel_max and m <= mae_max, f"{what}: max rel {r:.3e} (<= {rel_max}), MAE {m:.3e} (<= {mae_max})"
    return r, m


def assert_close_requantized(got, ref, rel_max=REL_MAX, mae_max=MAE_MAX, flip_frac=1e-3, flip_rel=0.25, what=""):
    """The bar for a layer that quantizes its own intermediate activations
    (NVFP4 a rows): the GPU's bf16 a (fp32 accumulation) and the oracle's
    (fp64) differ by a bf16 ulp now and then, and a value on an E2M1 rounding
    boundary then takes the neighbouring code on one side, which moves the
    outputs that read it by up to one E2M1 step of that value times a weight.
    Both codes are correct quantizations.  So: MAE as always, at most
    flip_frac of the elements beyond rel_max, none beyond flip_rel."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), rms if rms > 0 else 1e-30)
    mae = float(np.abs(got - ref).mean()) if ref.size else 0.0
    over = float((rel > rel_max).mean()) if ref.size else 0.0
    r = float(rel.max(initial=0.0))
    print(f"\n{what}: MAE {mae:.3e}, max rel {r:.3e}, elements beyond {rel_max}: {over:.2e}")
    assert mae <= mae_max and over <= flip_frac and r <= flip_rel, \
        f"{what}: MAE {mae:.3e} (<= {mae_max}), beyond {rel_max}: {over:.2e} (<= {flip_frac}), max rel {r:.3e}"
    return r, mae


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def near_tie_tokens(z: np.ndarray, k: int, rel: float = 1e-5) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest logits (fp32-rounded oracle
    logits) are closer than rel * max|z|: a correct fp32 router may pick
    either side there."""
    T, E = z.shape
    if k >= E:
        return np.zeros(T, dtype=bool)
    z32 = z.astype(np.float32).astype(np.float64)
    s = -np.sort(-z32, axis=1)
    gap = s[:, k - 1] - s[:, k]
    scale = np.maximum(np.abs(z32).max(axis=1), 1e-30)
    return gap <= rel * scale


def check_choice_valid(z: np.ndarray, ids_gpu: np.ndarray, k: int, rel: float = 1e-5):
    """The GPU's chosen set is a valid top-k of the oracle logits up to a
    perturbation of rel * max|z|, and is listed in ascending id."""
    z32 = z.astype(np.float32).astype(np.float64)
    for t in range(z.shape[0]):
        row = ids_gpu[t]
        assert (np.diff(row) > 0).all(), f"token {t}: ids not ascending/distinct"
        kth = -np.sort(-z32[t])[k - 1]
        tol = rel * max(np.abs(z32[t]).max(), 1e-30)
        assert (z32[t, row] >= kth - tol).all(), f"token {t}: chose an expert below the k-th logit"


def check_grouping_properties(ids: np.ndarray, counts, offsets, perm, inv, E: int):
    """Grouping outputs are the stable grouping of the given ids (properties
    only; used when ids legitimately differ from the oracle's)."""
    flat = ids.reshape(-1)
    n = flat.size
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and np.array_equal(offsets[1:], np.cumsum(counts))
    assert np.array_equal(perm[inv], np.arange(n))
    for e in range(E):
        rows = perm[offsets[e]:offsets[e + 1]]
        assert (flat[rows] == e).all() and (np.diff(rows) > 0).all()


def host_layer(lw: I.LayerWeights):
    """Host copies (uint16 bits) of a layer's weights, resolved per expert
    through its placement by the oracle's resolver."""
    pl = lw.placement
    lpool = (I.bf16_bits(lw.local_w13), I.bf16_bits(lw.local_w2))
    ppools = [(I.bf16_bits(a), I.bf16_bits(b)) for a, b in zip(lw.peer_w13, lw.peer_w2)]
    w13s, w2s = oracle.resolve_experts(lw.shape.E, lpool, ppools, pl.local_slot, pl.peer_id, pl.peer_slot)
    sw13 = I.bf16_bits(lw.shared_w13) if lw.shared_w13 is not None else None
    sw2 = I.bf16_bits(lw.shared_w2) if lw.shared_w2 is not None else None
    return w13s, w2s, sw13, sw2


class GpuLayerRun:
    """Route + prefetch + MoE through the C ABI for one layer."""

    def __init__(self, shape: I.LayerShape, lw: I.LayerWeights, n_layers=1, stage_slots=None):
        self.shape = shape
        slots = stage_slots if stage_slots is not None else max(1, lw.placement.n_remote())
        self.rt = B.Runtime(shape.H, shape.I, shape.E, shape.k, shape.S, shape.T, n_layers, slots)
        self.rt.set_layer(0, lw)
        self.lw = lw

    def run(self, x: torch.Tensor, chunk_bytes=1 << 20, n_copy_streams=1, keep_logits=True):
        sh = self.shape
        T = x.shape[0]
        rb = B.RouteBuffers(T, sh.E, sh.k, keep_logits=keep_logits)
        out = torch.empty((max(1, T), sh.H), dtype=torch.bfloat16, device="cuda")
        if self.lw.placement.n_remote() > 0:
            streams = [torch.cuda.Stream() for _ in range(n_copy_streams)]
            self.rt.prefetch(0, 0, chunk_bytes, streams)
        self.rt.route(x, self.lw.wr, self.lw.bias, rb)
        self.rt.moe(0, 0, x, rb, out)
        torch.cuda.synchronize()
        assert self.rt.device_status() == 0
        return rb, out[:T]

    def close(self):
        self.rt.close()


def assert_route_same_logits(o, rb, T: int, k: int, E: int):
    """The oracle's steps after the logits (top-k on fp32 decisions, weights,
    grouping) fed the GPU's own fp32 logits for every token: expert ids,
    counts, offsets, perm and inv_perm must then be identical, bit for bit,
    and the weights equal within fp32 softmax rounding.  (The GPU's logits
    themselves are checked against the oracle's fp64 logits separately.)
    Returns the oracle's (ids, w) for those logits."""
    z = rb.logits.cpu().numpy()[:T].astype(np.float64)
    ids_o, w_o = o.topk(z, k, decide_fp32=True)
    counts, offsets, perm, inv = o.group(ids_o, E)
    ids = rb.topk_ids.cpu().numpy()[:T]
    bad = np.nonzero((ids != ids_o).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} of {T} tokens choose other experts than the oracle on the same logits " \
                          f"(first: token {bad[:5].tolist()})"
    assert np.array_equal(rb.counts.cpu().numpy(), counts)
    assert np.array_equal(rb.offsets.cpu().numpy(), offsets)
    assert np.array_equal(rb.perm.cpu().numpy()[: T * k], perm)
    assert np.array_equal(rb.inv_perm.cpu().numpy()[: T * k], inv)
    w = rb.topk_w.cpu().numpy()[:T].astype(np.float64)
    dw = np.abs(w - w_o).max()
    assert dw <= 2e-6, f"weights differ by {dw:.3e}"
    return ids_o, w_o


def last_tile_tokens(perm, offsets, k: int, T: int, eligible, n_shared: int = 0, bm: int = 128):
    """A small set of tokens that between them own at least one row of
    every routed expert's last (ragged) 128-row m-tile, and (n_shared) of
    the shared expert's last m-tile, chosen greedily from the tokens in
    `eligible` (a boolean mask over tokens).  Returns (sorted tokens,
    experts whose last tile has no eligible token)."""
    E = offsets.size - 1
    cover = {}
    missed = []
    for e in range(E):
        c = int(offsets[e + 1] - offsets[e])
        if c == 0:
            continue
        start = int(offsets[e]) + bm * ((c - 1) // bm)
        toks = {int(t) for t in perm[start:offsets[e + 1]] // k if eligible[t]}
        if not toks:
            missed.append(e)
            continue
        for t in toks:
            cover.setdefault(t, set()).add(e)
    left = set(e for s in cover.values() for e in s)
    chosen = []
    while left:
        t = max(cover, key=lambda u: (len(cover[u] & left), -u))
        chosen.append(t)
        left -= cover.pop(t)
    if n_shared:
        tail = [t for t in range(bm * ((T - 1) // bm), T) if eligible[t]]
        if tail and not any(t >= bm * ((T - 1) // bm) for t in chosen):
            chosen.append(tail[-1])
    return np.array(sorted(chosen), dtype=np.int64), missed
