"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with what the mathematics fixes: brute force on tiny inputs,
closed forms, invariants, special cases that reduce to a textbook or library
routine.  ``test_oracle_pins.py`` runs them against the oracle;
``test_oracle_mutants.py`` runs them against builds of the oracle with one
planted mistake each and checks that some pin fails.

Independent routines used here: numpy / torch fp64 matmuls, torch's own bf16
conversion, scipy's softmax, ``math.fsum`` and ``itertools.combinations``.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import scipy.special
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers --
def _bits_from_f32(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of fp32 values, by torch's conversion (RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _decode(bits: np.ndarray) -> np.ndarray:
    """fp64 values of bf16 bit patterns, by torch's conversion."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _rand_bits(rng, shape, std):
    return _bits_from_f32(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _silu(v):
    return v / (1.0 + np.exp(-v))


def _dense_moe(x, wr, bias, k, w13s, w2s, sw13, sw2, orc_ids, orc_w):
    """Dense brute force: out[t] = sum_e G[t, e] FFN_e(x_t) (+ shared), where
    G is the dense T x E gate matrix (zero outside the chosen set), and FFN_e
    is evaluated for EVERY expert on EVERY token with numpy fp64 matmuls."""
    X = _decode(x)
    T = X.shape[0]
    E = len(w13s)
    G = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            G[t, orc_ids[t, j]] += orc_w[t, j]
    out = np.zeros_like(X)
    for e in range(E):
        W13 = _decode(w13s[e])
        I = W13.shape[0] // 2
        Wg, Wu = W13[:I].T, W13[I:].T          # [H, I]
        Wd = _decode(w2s[e]).T                 # [I, H]
        Y = (_silu(X @ Wg) * (X @ Wu)) @ Wd
        out += G[:, e:e + 1] * Y
    if sw13 is not None:
        W13 = _decode(sw13)
        I = W13.shape[0] // 2
        out += (_silu(X @ W13[:I].T) * (X @ W13[I:].T)) @ _decode(sw2).T
    return out


def _random_layer(rng, T, H, I, E, k, S, wstd=0.1):
    x = _rand_bits(rng, (T, H), 1.0)
    wr = _rand_bits(rng, (E, H), 0.3)
    w13s = [_rand_bits(rng, (2 * I, H), wstd) for _ in range(E)]
    w2s = [_rand_bits(rng, (H, I), wstd) for _ in range(E)]
    sw13 = _rand_bits(rng, (2 * I, H), wstd) if S else None
    sw2 = _rand_bits(rng, (H, I), wstd) if S else None
    return x, wr, w13s, w2s, sw13, sw2


# ------------------------------------------------------------------- bf16 --
def pin_bf16(o):
    rng = np.random.default_rng(1)
    f = (rng.standard_normal(4000) * np.exp(rng.uniform(-30, 30, 4000))).astype(np.float32)
    ref = _bits_from_f32(f)
    got = np.array([o.round_bf16(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref), "round_bf16 disagrees with torch on binary32 inputs"
    dec = np.array([o.bf16_to_double(int(b)) for b in ref])
    assert np.array_equal(dec, _decode(ref)), "bf16 decode disagrees with torch"
    # ties to even, and no double rounding through binary32
    assert o.round_bf16(1.0 + 2.0 ** -8) == 0x3F80            # tie -> even (1.0)
    assert o.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82        # tie -> even (1 + 2^-6)
    assert o.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81  # just above the tie
    assert o.round_bf16(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    assert o.round_bf16(2.0 ** -133) == 0x0001                # smallest subnormal
    assert o.round_bf16(1e39) == 0x7F80                       # overflow -> inf


# ---------------------------------------------------------------- routing --
def pin_router_logits(o):
    rng = np.random.default_rng(2)
    T, H, E = 40, 96, 7
    x = _rand_bits(rng, (T, H), 1.0)
    wr = _rand_bits(rng, (E, H), 0.1)
    bias = rng.standard_normal(E).astype(np.float32)
    z = o.router_logits(x, wr, bias)
    ref = _decode(x) @ _decode(wr).T + bias.astype(np.float64)[None, :]
    assert np.allclose(z, ref, rtol=0, atol=1e-12), "router logits != x @ Wr + b"
    z0 = o.router_logits(x, wr, None)
    assert np.allclose(z0, _decode(x) @ _decode(wr).T, rtol=0, atol=1e-12)


def _bruteforce_topk(zrow32, k):
    """All k-subsets; the winner maximises the (correctly rounded) sum of p,
    ties to the lexicographically smallest id tuple."""
    p = np.exp(zrow32 - zrow32.max())
    best, best_key = None, None
    for sub in itertools.combinations(range(len(zrow32)), k):
        s = math.fsum(p[list(sub)])
        key = (-s, sub)
        if best_key is None or key < best_key:
            best, best_key = sub, key
    return list(best)


def pin_topk_bruteforce(o):
    rng = np.random.default_rng(3)
    for (T, E, k) in [(64, 8, 2), (30, 6, 3), (20, 5, 1), (12, 7, 4)]:
        z = rng.standard_normal((T, E))
        z[: T // 3] = np.round(z[: T // 3] * 2) / 2      # many exact ties
        ids, w = o.topk(z, k, decide_fp32=True)
        z32 = z.astype(np.float32).astype(np.float64)
        for t in range(T):
            assert list(ids[t]) == _bruteforce_topk(z32[t], k), f"top-{k} wrong at token {t}"


def pin_weights(o):
    rng = np.random.default_rng(4)
    T, E, k = 50, 16, 4
    z = rng.standard_normal((T, E)) * 3
    ids, w = o.topk(z, k)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-12), "weights do not sum to 1"
    for t in range(T):
        ref = scipy.special.softmax(z[t, ids[t]])        # renormalised over the chosen set
        assert np.allclose(w[t], ref, rtol=1e-12, atol=0)
        full = scipy.special.softmax(z[t])
        assert np.allclose(w[t], full[ids[t]] / full[ids[t]].sum(), rtol=1e-12, atol=0)


def pin_special_cases(o):
    rng = np.random.default_rng(5)
    z = rng.standard_normal((9, 6))
    ids, w = o.topk(z, 6)                                # k = E: full softmax
    assert (ids == np.arange(6)[None, :]).all()
    assert np.allclose(w, scipy.special.softmax(z, axis=1), rtol=1e-12, atol=0)
    ids, w = o.topk(rng.standard_normal((5, 1)), 1)      # E = 1
    assert (ids == 0).all() and np.array_equal(w, np.ones((5, 1)))
    ids, w = o.topk(np.full((4, 8), 0.25), 3)            # equal logits
    assert (ids == np.arange(3)[None, :]).all()
    assert np.allclose(w, 1.0 / 3.0, rtol=0, atol=1e-15)
    z = np.array([[0.0, 5.0, 1.0, 5.0, -1.0]])           # hand example
    ids, w = o.topk(z, 2)
    assert list(ids[0]) == [1, 3] and np.allclose(w[0], [0.5, 0.5], atol=1e-15)
    ids, w = o.topk(z, 3)
    e5, e1 = math.exp(5.0), math.exp(1.0)
    assert list(ids[0]) == [1, 2, 3]
    assert np.allclose(w[0], [e5 / (2 * e5 + e1), e1 / (2 * e5 + e1), e5 / (2 * e5 + e1)],
                       rtol=1e-14, atol=0)


def pin_group(o):
    rng = np.random.default_rng(6)
    for (T, E, k) in [(64, 8, 2), (33, 5, 5), (1, 4, 1), (100, 13, 3)]:
        z = rng.standard_normal((T, E))
        ids, _ = o.topk(z, k)
        counts, offsets, perm, inv = o.group(ids, E)
        flat = ids.reshape(-1)
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert offsets[0] == 0 and np.array_equal(offsets[1:], np.cumsum(counts))
        assert counts.sum() == T * k
        assert np.array_equal(perm[inv], np.arange(T * k)), "perm o inv != id"
        assert np.array_equal(inv[perm], np.arange(T * k)), "inv o perm != id"
        for e in range(E):
            rows = perm[offsets[e]:offsets[e + 1]]
            assert (flat[rows] == e).all(), "row in the wrong expert group"
            assert (np.diff(rows) > 0).all(), "group not in ascending flat index"
        # permute -> unpermute round trip on x
        x = rng.standard_normal((T, 3))
        xp = x[perm // k]
        back = xp[inv].reshape(T, k, 3)
        assert np.array_equal(back, np.repeat(x[:, None, :], k, axis=1))


# -------------------------------------------------------------------- FFN --
def pin_ffn_dense(o):
    rng = np.random.default_rng(7)
    for (T, H, I, E, k, S) in [(24, 32, 16, 6, 3, 1), (16, 48, 8, 4, 1, 0), (10, 16, 16, 3, 3, 1)]:
        x, wr, w13s, w2s, sw13, sw2 = _random_layer(rng, T, H, I, E, k, S)
        r = o.route(x, wr, None, k)
        out = o.moe_tokens(x, np.arange(T), r["ids"], r["w"], w13s, w2s, sw13, sw2, mirrored=False)
        ref = _dense_moe(x, wr, None, k, w13s, w2s, sw13, sw2, r["ids"], r["w"])
        scale = np.sqrt((ref ** 2).mean())
        assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, scale), "MoE != dense brute force"


def pin_swiglu_textbook(o):
    """E = k = 1, no shared expert: the layer is one SwiGLU MLP."""
    rng = np.random.default_rng(8)
    T, H, I = 12, 40, 24
    x, wr, w13s, w2s, _, _ = _random_layer(rng, T, H, I, 1, 1, 0)
    r = o.route(x, wr, None, 1)
    out = o.moe_tokens(x, np.arange(T), r["ids"], r["w"], w13s, w2s, mirrored=False)
    X = torch.from_numpy(_decode(x))
    W13 = torch.from_numpy(_decode(w13s[0]))
    Wd = torch.from_numpy(_decode(w2s[0]))
    lin_g = torch.nn.functional.linear(X, W13[:I])       # x W_gate
    lin_u = torch.nn.functional.linear(X, W13[I:])       # x W_up
    ref = torch.nn.functional.linear(torch.nn.functional.silu(lin_g) * lin_u, Wd).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12), "not the textbook SwiGLU MLP"


def pin_linearity_and_zero(o):
    rng = np.random.default_rng(9)
    T, H, I, E, k = 8, 32, 16, 4, 2
    x, wr, w13s, w2s, sw13, sw2 = _random_layer(rng, T, H, I, E, k, 1)
    r = o.route(x, wr, None, k)
    tok = np.arange(T)
    for mirrored in (False, True):
        base = o.moe_tokens(x, tok, r["ids"], r["w"], w13s, w2s, sw13, sw2, mirrored=mirrored)
        dbl = lambda b: _bits_from_f32(_decode(b).astype(np.float32) * 2)  # exact in bf16
        out2 = o.moe_tokens(x, tok, r["ids"], r["w"], w13s, [dbl(b) for b in w2s], sw13, dbl(sw2),
                            mirrored=mirrored)
        assert np.array_equal(out2, 2 * base), "not linear in W_down"
    zeros13 = [np.zeros_like(b) for b in w13s]
    out0 = o.moe_tokens(x, tok, r["ids"], r["w"], zeros13, w2s, np.zeros_like(sw13), sw2)
    assert not out0.any(), "zero weights must give zero output"


def pin_mirrored(o):
    """Mirrored outputs are bf16 values and sit within bf16 rounding of the
    strict ones; each expert's mirrored output equals the strict computation
    with a and y rounded (checked through a one-expert layer)."""
    rng = np.random.default_rng(10)
    T, H, I, E, k = 16, 64, 32, 5, 2
    x, wr, w13s, w2s, sw13, sw2 = _random_layer(rng, T, H, I, E, k, 1)
    r = o.route(x, wr, None, k)
    tok = np.arange(T)
    m = o.moe_tokens(x, tok, r["ids"], r["w"], w13s, w2s, sw13, sw2, mirrored=True)
    s = o.moe_tokens(x, tok, r["ids"], r["w"], w13s, w2s, sw13, sw2, mirrored=False)
    assert np.array_equal(_decode(_bits_from_f32(m.astype(np.float32))), m)
    rms = np.sqrt((s ** 2).mean())
    assert np.max(np.abs(m - s)) <= 0.03 * rms
    # one expert, by hand with torch fp64 and torch's bf16 rounding
    X = _decode(x)
    W13 = _decode(w13s[0])
    Wd = _decode(w2s[0])
    for t in range(3):
        a = _silu(X[t] @ W13[:I].T) * (X[t] @ W13[I:].T)
        a = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
        y = a @ Wd.T
        got = o.expert_ffn(x[t], w13s[0], w2s[0], mirrored=True)
        # y is rounded from fp64 by the oracle, from fp64 via torch here:
        # torch may round twice (fp64 -> fp32 -> bf16), so allow one ulp
        yb = torch.from_numpy(y).to(torch.bfloat16).to(torch.float64).numpy()
        ulp = np.abs(yb) * 2.0 ** -7 + 1e-30
        assert (np.abs(got - yb) <= ulp).all()


def pin_map_invariance(o):
    """DWDP §2: where an expert lives does not change the layer's output."""
    import oracle as _o
    rng = np.random.default_rng(11)
    T, H, I, E, k = 12, 32, 16, 8, 3
    x, wr, w13s, w2s, sw13, sw2 = _random_layer(rng, T, H, I, E, k, 1)
    r = o.route(x, wr, None, k)
    ref = o.moe_tokens(x, np.arange(T), r["ids"], r["w"], w13s, w2s, sw13, sw2)
    for trial in range(4):
        n_local = int(rng.integers(0, E + 1))
        order = rng.permutation(E)
        local = order[:n_local]
        n_peers = int(rng.integers(1, 4))
        lpool = (np.zeros((E, 2 * I, H), np.uint16), np.zeros((E, H, I), np.uint16))
        ppools = [(np.zeros((E, 2 * I, H), np.uint16), np.zeros((E, H, I), np.uint16))
                  for _ in range(n_peers)]
        ls = np.full(E, -1, np.int32)
        pid = np.full(E, -1, np.int32)
        ps = np.full(E, -1, np.int32)
        slots = rng.permutation(E)
        for i, e in enumerate(local):
            ls[e] = slots[i]
            lpool[0][slots[i]] = w13s[e]
            lpool[1][slots[i]] = w2s[e]
        for e in range(E):
            if ls[e] < 0 or rng.random() < 0.3:      # remote, or redundant copy
                p = int(rng.integers(0, n_peers))
                pid[e], ps[e] = p, int(rng.integers(0, E))
                while ppools[p][0][ps[e]].any():
                    ps[e] = (ps[e] + 1) % E
                ppools[p][0][ps[e]] = w13s[e]
                ppools[p][1][ps[e]] = w2s[e]
        r13, r2 = _o.resolve_experts(E, lpool, ppools, ls, pid, ps)
        got = o.moe_tokens(x, np.arange(T), r["ids"], r["w"], r13, r2, sw13, sw2)
        assert np.array_equal(got, ref), "output depends on placement"


def pin_closed_form_golden(o):
    """The hand-worked layer in golden/tiny_closed_form.json: every expected
    value is a closed form in sigma(v) = 1/(1+exp(-v))."""
    with open(os.path.join(GOLDEN, "tiny_closed_form.json")) as f:
        g = json.load(f)
    bits = lambda a: _bits_from_f32(np.array(a, dtype=np.float32))
    x = bits(g["x"])
    wr = bits(g["router_w"])
    w13s = [bits(a) for a in g["w13"]]
    w2s = [bits(a) for a in g["w2"]]
    k = g["k"]
    r = o.route(x, wr, None, k)
    assert r["ids"].tolist() == g["expected_ids"]
    env = {"sigma": lambda v: 1.0 / (1.0 + math.exp(-v)), "exp": math.exp}
    ew = np.array([[eval(s, {}, env) for s in row] for row in g["expected_w"]])
    assert np.allclose(r["w"], ew, rtol=1e-14, atol=0)
    out = o.moe_tokens(x, np.arange(x.shape[0]), r["ids"], r["w"], w13s, w2s, mirrored=False)
    eo = np.array([[eval(s, {}, env) for s in row] for row in g["expected_out"]])
    assert np.allclose(out, eo, rtol=1e-14, atol=1e-300)
    assert r["counts"].tolist() == g["expected_counts"]
    assert r["perm"].tolist() == g["expected_perm"]


ALL_PINS = [pin_bf16, pin_router_logits, pin_topk_bruteforce, pin_weights, pin_special_cases,
            pin_group, pin_ffn_dense, pin_swiglu_textbook, pin_linearity_and_zero, pin_mirrored,
            pin_map_invariance, pin_closed_form_golden]


def pin_grouped_gemm(o):
    """The grouped GEMM against numpy fp64 matmuls, group by group, for the
    three epilogues; empty groups and ragged sizes included."""
    rng = np.random.default_rng(12)
    K, N = 48, 20
    off = np.array([0, 5, 5, 17, 18, 30], dtype=np.int32)
    a = _rand_bits(rng, (32, K), 1.0)
    A = _decode(a)
    for epi in (0, 1, 2):
        bl = [_rand_bits(rng, ((2 if epi == 1 else 1) * N, K), 0.3) for _ in range(off.size - 1)]
        d = o.grouped_gemm(a, off, bl, N, epi)
        ref = np.zeros((32, N))
        for g in range(off.size - 1):
            Bg = _decode(bl[g])
            r0, r1 = off[g], off[g + 1]
            if epi == 1:
                ref[r0:r1] = _silu(A[r0:r1] @ Bg[:N].T) * (A[r0:r1] @ Bg[N:].T)
            else:
                ref[r0:r1] = A[r0:r1] @ Bg.T
        assert np.allclose(d, ref, rtol=1e-12, atol=1e-12), f"grouped GEMM epilogue {epi}"


ALL_PINS.append(pin_grouped_gemm)


# ------------------------------------------------------------ FP8 (E4M3) --
def _e4m3_torch(v32: np.ndarray) -> np.ndarray:
    """E4M3 codes of binary32 values by torch's conversion (RNE, no
    saturation: only used on values within +-464)."""
    return torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def _e4m3_decode_torch(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def pin_e4m3(o):
    rng = np.random.default_rng(13)
    v = (rng.standard_normal(6000) * np.exp(rng.uniform(-9, 6, 6000))).astype(np.float32)
    v = v[np.abs(v) <= 464]
    got = np.array([o.e4m3_encode(float(a)) for a in v], dtype=np.uint8)
    assert np.array_equal(got, _e4m3_torch(v)), "E4M3 encoding disagrees with torch"
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    dec = np.array([o.e4m3_decode(int(c)) for c in codes])
    assert np.array_equal(dec, _e4m3_decode_torch(codes)), "E4M3 decoding disagrees with torch"
    # saturation, ties to even, subnormals (by the format's definition)
    assert o.e4m3_encode(1000.0) == 0x7E and o.e4m3_encode(-470.0) == 0xFE
    assert o.e4m3_encode(1.0625) == 0x38          # tie between 1 and 1.125 -> even (1)
    assert o.e4m3_encode(1.1875) == 0x3A          # tie between 1.125 and 1.25 -> even (1.25)
    assert o.e4m3_encode(2.0 ** -9) == 0x01 and o.e4m3_encode(2.0 ** -10) == 0x00


def pin_quantize_rows(o):
    rng = np.random.default_rng(14)
    for n in (1, 7, 256, 2048):
        row = (rng.standard_normal(n) * rng.uniform(0.01, 50)).astype(np.float32)
        codes, scale = o.quantize_row_e4m3(row)
        amax = np.float32(np.abs(row).max())
        assert scale == np.float32(amax / np.float32(448.0))
        ref = _e4m3_torch(row / np.float32(scale))
        assert np.array_equal(codes, ref), "row codes differ from torch's encoding of v / scale"
        i = int(np.argmax(np.abs(row)))
        assert codes[i] & 0x7F == 0x7E, "the row's largest value must map to +-448"
        deq = _e4m3_decode_torch(codes) * scale
        assert np.all(np.abs(deq - row) <= np.abs(row) * 2.0 ** -4 + scale * 2.0 ** -10)
    codes, scale = o.quantize_row_e4m3(np.zeros(5, np.float32))
    assert scale == 1.0 and not codes.any()


def _fp8_layer(rng, T, H, I, E, S):
    x = _rand_bits(rng, (T, H), 1.0)
    wr = _rand_bits(rng, (E, H), 0.3)
    mk = lambda shape: _e4m3_torch(rng.standard_normal(shape).astype(np.float32))
    w13s = [mk((2 * I, H)) for _ in range(E)]
    w2s = [mk((H, I)) for _ in range(E)]
    s13 = rng.uniform(0.02, 0.05, E).astype(np.float32)
    s2 = rng.uniform(0.02, 0.05, E).astype(np.float32)
    sw = (mk((2 * I, H)), mk((H, I)), np.float32(0.03), np.float32(0.04)) if S else None
    return x, wr, w13s, w2s, s13, s2, sw


def _dense_fp8(x, ids, w, w13s, w2s, s13, s2, sw):
    """Dense brute force of the FP8 layer: every expert on every token, torch's
    E4M3 conversion for every quantization, numpy fp64 matmuls, a rounded
    once to binary32 before its quantization (strict mode)."""
    X32 = _decode(x).astype(np.float32)
    T, H = X32.shape
    E = len(w13s)
    xs = np.abs(X32).max(axis=1) / np.float32(448.0)
    xs[xs == 0] = 1
    XQ = _e4m3_decode_torch(_e4m3_torch(X32 / xs[:, None])) * xs.astype(np.float64)[:, None]
    G = np.zeros((T, E))
    for t in range(T):
        for j in range(ids.shape[1]):
            G[t, ids[t, j]] += w[t, j]

    def ffn(W13c, W2c, sc13, sc2):
        W13 = _e4m3_decode_torch(W13c) * np.float64(sc13)
        W2 = _e4m3_decode_torch(W2c) * np.float64(sc2)
        I = W13.shape[0] // 2
        A = (_silu(XQ @ W13[:I].T) * (XQ @ W13[I:].T)).astype(np.float32)
        sa = np.abs(A).max(axis=1) / np.float32(448.0)
        sa[sa == 0] = 1
        AQ = _e4m3_decode_torch(_e4m3_torch(A / sa[:, None])) * sa.astype(np.float64)[:, None]
        return AQ @ W2.T

    out = np.zeros((T, H))
    for e in range(E):
        out += G[:, e:e + 1] * ffn(w13s[e], w2s[e], s13[e], s2[e])
    if sw is not None:
        out += ffn(*sw)
    return out


def pin_fp8_dense(o):
    rng = np.random.default_rng(15)
    for (T, H, I, E, k, S) in [(20, 32, 16, 5, 2, 1), (12, 64, 32, 3, 3, 0)]:
        x, wr, w13s, w2s, s13, s2, sw = _fp8_layer(rng, T, H, I, E, S)
        r = o.route(x, wr, None, k)
        kw = {} if sw is None else dict(shared_w13=sw[0], shared_w2=sw[1], shared_s13=sw[2], shared_s2=sw[3])
        got = o.moe_tokens_fp8(x, np.arange(T), r["ids"], r["w"], w13s, w2s, s13, s2, mirrored=False, **kw)
        ref = _dense_fp8(x, r["ids"], r["w"], w13s, w2s, s13, s2, sw)
        scale = np.sqrt((ref ** 2).mean())
        assert np.max(np.abs(got - ref)) <= 1e-9 * max(1.0, scale), "FP8 layer != dense brute force"
        # mirrored mode: bf16-valued outputs close to strict
        m = o.moe_tokens_fp8(x, np.arange(T), r["ids"], r["w"], w13s, w2s, s13, s2, mirrored=True, **kw)
        assert np.array_equal(_decode(_bits_from_f32(m.astype(np.float32))), m)
        assert np.max(np.abs(m - got)) <= 0.1 * scale


ALL_PINS += [pin_e4m3, pin_quantize_rows, pin_fp8_dense]


# ---------------------------------------------------------------- NVFP4 --
# E2M1 magnitudes of codes 0..7 by the format's definition (exponent field 0:
# 0.5 * m; otherwise 2^(e-1) * (1 + m/2)); bit 3 is the sign.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_nearest(v: float) -> int:
    """Brute force over the 8 magnitudes: nearest, ties to the even code
    (mantissa bit 0), saturating at 6, sign kept."""
    a = abs(v)
    sign = 8 if math.copysign(1.0, v) < 0 else 0
    if a >= 6.0:
        return sign | 7
    return sign | min(range(8), key=lambda c: (abs(a - E2M1_MAGNITUDES[c]), c & 1))


def _nvfp4_decode(codes, sf):
    """Dequantized values (without the row scale) of one-code-per-byte E2M1
    codes and their E4M3 block scales, blocks of 16 along the last axis."""
    codes = np.asarray(codes)
    mag = np.array(E2M1_MAGNITUDES)[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    scale = np.repeat(_e4m3_decode_torch(np.asarray(sf)), 16, axis=-1)
    return mag * scale


def pin_e2m1(o):
    for c in range(16):
        want = E2M1_MAGNITUDES[c & 7] * (-1.0 if c & 8 else 1.0)
        got = o.e2m1_decode(c)
        assert got == want and math.copysign(1.0, got) == (-1.0 if c & 8 else 1.0), f"E2M1 decode of {c}"
    grid = np.concatenate([np.arange(-8.0, 8.0, 1.0 / 64), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, 6.5, 1e9]])
    for v in grid:
        assert o.e2m1_encode(float(v)) == _e2m1_nearest(float(v)), f"E2M1 encoding of {v}"


def pin_quantize_rows_nvfp4(o):
    rng = np.random.default_rng(16)
    # 1) rows of exactly representable values come back with their own codes:
    #    block b holds E2M1 magnitudes times 2^e_b with one element at 6 * 2^e_b
    for n, spread in ((16, 0), (64, 3), (2048, 6)):
        nb = n // 16
        e = rng.integers(-spread, 1, size=nb) if spread else np.zeros(nb, dtype=int)
        codes = rng.integers(0, 16, size=n).astype(np.uint8)
        codes[np.arange(nb) * 16 + rng.integers(0, 16, size=nb)] = 7
        vals = (np.array(E2M1_MAGNITUDES)[codes & 7] * np.where(codes & 8, -1.0, 1.0)
                * np.repeat(2.0 ** e, 16) * 3.0).astype(np.float32)
        got, sf, s = o.quantize_row_nvfp4(vals)
        same = (got & 7) == (codes & 7)
        nz = (codes & 7) != 0
        assert same.all() and ((got[nz] & 8) == (codes[nz] & 8)).all(), "representable row did not round-trip"
        assert np.allclose(_nvfp4_decode(got, sf) * s, vals, rtol=1e-6, atol=0)
        assert (sf[e == 0] == 0x7E).all(), "blocks holding the row maximum take scale 448"
    # 2) scaling a row by 2^j changes only the row scale
    for n in (32, 512):
        row = (rng.standard_normal(n) * 3.0).astype(np.float32)
        c0, sf0, s0 = o.quantize_row_nvfp4(row)
        for j in (-7, 5):
            c1, sf1, s1 = o.quantize_row_nvfp4(row * np.float32(2.0 ** j))
            assert np.array_equal(c0, c1) and np.array_equal(sf0, sf1) and s1 == s0 * 2.0 ** j
    # 3) error bound: each value is within one E4M3-scaled step of its code
    for n in (16, 256, 2048):
        row = (rng.standard_normal(n) * rng.uniform(0.01, 50)).astype(np.float32)
        row[rng.integers(0, n, size=n // 32)] *= 20            # outliers
        c, sf, s = o.quantize_row_nvfp4(row)
        deq = _nvfp4_decode(c, sf) * s
        eff = np.repeat(_e4m3_decode_torch(sf), 16) * s
        assert np.all(np.abs(deq - row) <= eff * 1.0 + 1e-30), "error above the coarsest half step"
        i = int(np.argmax(np.abs(row)))
        assert c[i] & 7 == 7 and sf[i // 16] == 0x7E, "the row maximum must map to +-6 with scale 448"
        bmax = np.abs(row).reshape(-1, 16).max(axis=1)
        assert np.all(np.abs(_e4m3_decode_torch(sf) * 6 * s - bmax) <= bmax * 2.0 ** -3), "block scale off"
    # 4) zero row, zero block
    c, sf, s = o.quantize_row_nvfp4(np.zeros(32, np.float32))
    assert s == 1.0 and not c.any() and not sf.any()
    row = rng.standard_normal(48).astype(np.float32)
    row[16:32] = 0
    c, sf, s = o.quantize_row_nvfp4(row)
    assert sf[1] == 0 and not c[16:32].any()


def _nvfp4_layer(rng, T, H, I, E, S):
    x = _rand_bits(rng, (T, H), 1.0)
    wr = _rand_bits(rng, (E, H), 0.3)
    code = lambda shape: rng.integers(0, 16, size=shape).astype(np.uint8)
    sfc = lambda shape: rng.integers(0x30, 0x48, size=shape).astype(np.uint8)   # E4M3 0.5 .. 4.0
    mk = lambda: (code((2 * I, H)), sfc((2 * I, H // 16)), np.float32(rng.uniform(0.01, 0.02)),
                  code((H, I)), sfc((H, I // 16)), np.float32(rng.uniform(0.01, 0.02)))
    experts = [mk() for _ in range(E)]
    return x, wr, experts, (mk() if S else None)


def _dense_nvfp4(o, x, ids, w, experts, shared):
    """Dense brute force of the NVFP4 layer: every expert on every token,
    weights dequantized with numpy, fp64 matmuls; activation rows quantized
    with the oracle's row quantizer (pinned above), a rounded once to binary32
    (strict mode)."""
    X32 = _decode(x).astype(np.float32)
    T, H = X32.shape
    E = len(experts)

    def quant_rows(A32):
        out = np.zeros(A32.shape)
        for t in range(A32.shape[0]):
            c, sf, s = o.quantize_row_nvfp4(A32[t])
            out[t] = _nvfp4_decode(c, sf) * s
        return out

    XQ = quant_rows(X32)
    G = np.zeros((T, E))
    for t in range(T):
        for j in range(ids.shape[1]):
            G[t, ids[t, j]] += w[t, j]

    def ffn(c13, sf13, s13, c2, sf2, s2):
        W13 = _nvfp4_decode(c13, sf13) * np.float64(s13)
        W2 = _nvfp4_decode(c2, sf2) * np.float64(s2)
        I = W13.shape[0] // 2
        A = (_silu(XQ @ W13[:I].T) * (XQ @ W13[I:].T)).astype(np.float32)
        return quant_rows(A) @ W2.T

    out = np.zeros((T, H))
    for e in range(E):
        out += G[:, e:e + 1] * ffn(*experts[e])
    if shared is not None:
        out += ffn(*shared)
    return out


def pin_nvfp4_dense(o):
    rng = np.random.default_rng(17)
    for (T, H, I, E, k, S) in [(10, 64, 32, 5, 2, 1), (6, 32, 48, 3, 3, 0)]:
        x, wr, experts, shared = _nvfp4_layer(rng, T, H, I, E, S)
        r = o.route(x, wr, None, k)
        args = ([e[0] for e in experts], [e[1] for e in experts], [e[2] for e in experts],
                [e[3] for e in experts], [e[4] for e in experts], [e[5] for e in experts])
        got = o.moe_tokens_nvfp4(x, np.arange(T), r["ids"], r["w"], *args, shared=shared, mirrored=False)
        ref = _dense_nvfp4(o, x, r["ids"], r["w"], experts, shared)
        scale = np.sqrt((ref ** 2).mean())
        assert np.max(np.abs(got - ref)) <= 1e-9 * max(1.0, scale), "NVFP4 layer != dense brute force"
        m = o.moe_tokens_nvfp4(x, np.arange(T), r["ids"], r["w"], *args, shared=shared, mirrored=True)
        assert np.array_equal(_decode(_bits_from_f32(m.astype(np.float32))), m)
        assert np.sqrt(((m - got) ** 2).mean()) <= 0.1 * scale


ALL_PINS += [pin_e2m1, pin_quantize_rows_nvfp4, pin_nvfp4_dense]


def pin_nvfp4_linear(o):
    """The NVFP4 linear layer on given codes against numpy: the rows and the
    weights dequantized with the format tables, an fp64 matmul times the row
    and tensor scales (epilogue 0), and SiLU(gate) * up of the two halves
    (epilogue 1); mirrored mode is torch's bf16 rounding of that."""
    rng = np.random.default_rng(18)
    for (n, K, N) in [(7, 64, 5), (3, 256, 16)]:
        codes = rng.integers(0, 16, size=(n, K)).astype(np.uint8)
        sf = rng.integers(0x28, 0x50, size=(n, K // 16)).astype(np.uint8)
        rs = rng.uniform(0.001, 3.0, size=n).astype(np.float32)
        for epi in (0, 1):
            rows = 2 * N if epi else N
            w = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
            wsf = rng.integers(0x28, 0x50, size=(rows, K // 16)).astype(np.uint8)
            ws = np.float32(rng.uniform(0.005, 0.02))
            A = _nvfp4_decode(codes, sf) * rs[:, None].astype(np.float64)
            W = _nvfp4_decode(w, wsf) * np.float64(ws)
            if epi == 0:
                ref = A @ W.T
            else:
                g, u = A @ W[:N].T, A @ W[N:].T
                ref = _silu(g) * u
            got = o.nvfp4_linear(codes, sf, rs, w, wsf, ws, epilogue=epi, mirrored=False)
            scale = max(1.0, np.abs(ref).max())
            assert np.max(np.abs(got - ref)) <= 1e-12 * scale, f"NVFP4 linear (epilogue {epi}) != numpy"
            # mirrored: bf16 values within half a bf16 step (at most 2^-8 relative) of the exact result
            m = o.nvfp4_linear(codes, sf, rs, w, wsf, ws, epilogue=epi, mirrored=True)
            assert np.array_equal(_decode(_bits_from_f32(m.astype(np.float32))), m)
            assert np.all(np.abs(m - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)

ALL_PINS += [pin_nvfp4_linear]


def pin_e4m3_linear(o):
    """The E4M3 linear layer on given codes against numpy: rows and weights
    decoded by torch's float8_e4m3fn, an fp64 matmul times the row and
    tensor scales (epilogue 0), SiLU(gate) * up of the two halves (1)."""
    rng = np.random.default_rng(19)
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)   # no NaN codes
    for (n, K, N) in [(6, 32, 5), (3, 128, 12)]:
        codes = rng.choice(finite, size=(n, K))
        rs = rng.uniform(0.001, 3.0, size=n).astype(np.float32)
        for epi in (0, 1):
            rows = 2 * N if epi else N
            w = rng.choice(finite, size=(rows, K))
            ws = np.float32(rng.uniform(0.005, 0.02))
            A = _e4m3_decode_torch(codes) * rs[:, None].astype(np.float64)
            W = _e4m3_decode_torch(w) * np.float64(ws)
            with np.errstate(over="ignore"):      # exp(-g) overflows to inf for large negative g: SiLU -> 0
                ref = A @ W.T if epi == 0 else _silu(A @ W[:N].T) * (A @ W[N:].T)
            got = o.e4m3_linear(codes, rs, w, ws, epilogue=epi, mirrored=False)
            assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.abs(ref).max()), f"E4M3 linear {epi} != numpy"
            m = o.e4m3_linear(codes, rs, w, ws, epilogue=epi, mirrored=True)
            assert np.array_equal(_decode(_bits_from_f32(m.astype(np.float32))), m)
            assert np.all(np.abs(m - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)


ALL_PINS += [pin_e4m3_linear]
