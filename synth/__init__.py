"""Seeded synthetic inputs for the output head (numpy only).

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark. It holds input generation only: random draws, rounding of those
draws into the storage formats (bf16 / fp16 / int8) and the placement of
planted ties. It computes nothing of the head itself (no dot products, no
argmax, no softmax), so the oracle and the CUDA path stay independent.

Every array is returned as raw storage: bf16 and fp16 as ``uint16`` bit
patterns, int8 as ``int8``. Row-major, K (= d) contiguous: ``W`` is [V, d]
(the layout of a linear layer's weight), ``h`` is [B, d].

The shapes and distributions follow the workloads of the source pages:
TinyLlama-1.1B's head (d=2048, V=32000) for the greedy-decoding study in
"Greedy Decoding Has a Precision Clause"; Qwen2.5-class heads for the
speculative-verify and trainer-scoring workloads of "TandemLLM docs,
12 Exactness" and "batch-logprob-gap"; a Llama-3-class vocabulary for the
integer head of "Eliminating Nondeterminism in LLM Inference with
Integer-Only Arithmetic". Those pages measure on trained checkpoints and
public prompt sets; these draws stand in for their shapes only.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_from_f32", "f16_bits_from_f32", "normal_bf16", "uniform_int8",
    "pr1", "sweep", "spec_verify", "logprob", "int8_head", "small_float",
    "small_int8", "plant_drafts", "float_rows", "SEED_W", "SEED_H", "SEED_X",
]

SEED_W, SEED_H, SEED_X = 1000, 2000, 3000


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); bit patterns.

    Inputs are finite draws, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def f16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE binary16 (numpy's cast rounds to nearest even)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal_f32(rng: np.random.Generator, shape, sigma: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return x


def normal_bf16(seed: int, shape, sigma: float = 1.0) -> np.ndarray:
    return bf16_bits_from_f32(_normal_f32(_rng(seed), shape, sigma))


def uniform_int8(seed: int, shape, lo: int = -127, hi: int = 127) -> np.ndarray:
    return _rng(seed).integers(lo, hi + 1, size=shape, dtype=np.int8)


# --------------------------------------------------------------------------
# The five workloads. ``cfg`` numbers the workload (1..5); seeds are
# W = 1000+cfg, h = 2000+cfg, extra draws = 3000+cfg.
# --------------------------------------------------------------------------

def pr1(n_rows: int = 16, V: int = 32000, d: int = 2048):
    """Greedy decode of one row at a time (TinyLlama-1.1B head shape).

    W ~ N(0, 0.02) in bf16, h ~ N(0, 1) in bf16; each row is a B=1 call.
    """
    W = normal_bf16(SEED_W + 1, (V, d), 0.02)
    h = normal_bf16(SEED_H + 1, (n_rows, d), 1.0)
    return {"W": W, "h": h, "V": V, "d": d, "dtype": "bf16"}


def _next_bf16_bits(bits: np.uint16, up: bool) -> np.uint16:
    """Neighbouring value, one ulp larger (up) or smaller in value, of a
    16-bit sign-magnitude format (bf16 or fp16, finite non-extreme values)."""
    b = int(bits)
    neg = bool(b & 0x8000)
    mag = b & 0x7FFF
    if up != neg:   # magnitude grows
        mag += 1
    else:
        if mag == 0:
            return np.uint16(0x0001 if up else 0x8001)
        mag -= 1
    return np.uint16((b & 0x8000) | mag)


# Pair layout for the planted near ties: (a, b) rows of W.
#   inside one 128-row tile, both orders; neighbouring tiles; far apart in V.
TIE_PAIRS = ((10, 77), (300, 261), (1023, 1024), (1151, 1090),
             (5, 31990), (31000, 700), (12345, 12346), (20000, 19872))
EXACT_TIE_PAIRS = (6, 7)   # indices into TIE_PAIRS that get an exact tie


def sweep(V: int = 32000, d: int = 2048, n_plain: int = 56, c: float = 50.0):
    """The batch-invariance sweep: the PR1 head with 8 planted near-tie pairs.

    Reading of the construction (the workload only says "two W rows equal
    except 1-3 elements shifted by one bf16 ulp, h chosen so the top-2 gap is
    at most one ulp"): row b is a copy of row a with 1-3 elements moved by one
    bf16 ulp; the hidden row is bf16(c * W[a] / |W[a]| + small noise), which
    makes rows a and b the two best by a wide margin over the rest, with a gap
    far below one bf16 ulp of the winning logit. For two pairs the two moved
    elements go in opposite directions at positions where h holds the same
    value and W the same binade, so the two logits tie exactly.
    Rows 0..7 of h are the tie rows, rows 8..63 are plain N(0, 1) rows.
    """
    assert V > max(max(p) for p in TIE_PAIRS)
    W = normal_bf16(SEED_W + 1, (V, d), 0.02)        # same head as pr1
    rng = _rng(SEED_X + 2)
    Wf = (W.astype(np.uint32) << 16).view(np.float32)
    h_rows = []
    for k, (a, b) in enumerate(TIE_PAIRS):
        wa = Wf[a].astype(np.float32)
        base = np.float32(c) * wa / np.float32(np.linalg.norm(wa))
        noise = _normal_f32(rng, (d,), 0.02)
        hk = bf16_bits_from_f32(base + noise)
        if k in EXACT_TIE_PAIRS:
            # two positions i, j with h[i] == h[j] and W[a][i] == W[a][j] == w
            # (w with a non-zero mantissa, so one ulp up and one ulp down are
            # the same step): +ulp*h[i] - ulp*h[j] cancels exactly.
            cand = [int(x) for x in rng.permutation(d) if (int(W[a][x]) & 0x7F) != 0]
            i, j = cand[0], cand[1]
            hk[j] = hk[i]
            W[a][j] = W[a][i]
            row = W[a].copy()
            row[i] = _next_bf16_bits(row[i], True)
            row[j] = _next_bf16_bits(row[j], False)
        else:
            row = W[a].copy()
            n_moved = 1 + (k % 3)
            pos = rng.choice(d, size=n_moved, replace=False)
            for p in pos:
                row[p] = _next_bf16_bits(row[p], bool(rng.integers(0, 2)))
        W[b] = row
        h_rows.append(hk)
    plain = normal_bf16(SEED_H + 2, (n_plain, d), 1.0)
    h = np.concatenate([np.stack(h_rows), plain], axis=0)
    return {"W": W, "h": h, "V": V, "d": d, "dtype": "bf16",
            "tie_pairs": TIE_PAIRS, "exact_tie_pairs": EXACT_TIE_PAIRS}


def spec_verify(V: int = 152064, d: int = 3584, B: int = 256):
    """Speculative-verify block: 16 requests x 16 draft positions = 256 rows.

    W ~ N(0, 0.015) bf16; h = bf16(s_n * g_n), g ~ N(0, 1), s_n ~ U[0.5, 2].
    """
    W = normal_bf16(SEED_W + 3, (V, d), 0.015)
    rng = _rng(SEED_H + 3)
    g = _normal_f32(rng, (B, d), 1.0)
    s = rng.uniform(0.5, 2.0, size=(B, 1)).astype(np.float32)
    h = bf16_bits_from_f32(g * s)
    return {"W": W, "h": h, "V": V, "d": d, "dtype": "bf16"}


def logprob(V: int = 151936, d: int = 1536, n_seq: int = 8, seq_len: int = 1024,
            fmt: str = "bf16"):
    """Trainer-side scoring: 8 sequences x 1024 tokens, uniform target ids.

    The fp16 variant rounds the same float32 draws to fp16 instead of bf16.
    """
    rw = _rng(SEED_W + 4)
    rh = _rng(SEED_H + 4)
    Wf = _normal_f32(rw, (V, d), 0.02)
    hf = _normal_f32(rh, (n_seq * seq_len, d), 1.0)
    conv = bf16_bits_from_f32 if fmt == "bf16" else f16_bits_from_f32
    W = conv(Wf)
    del Wf
    h = conv(hf)
    targets = _rng(SEED_X + 4).integers(0, V, size=n_seq * seq_len).astype(np.int32)
    return {"W": W, "h": h, "targets": targets, "V": V, "d": d, "dtype": fmt,
            "n_seq": n_seq, "seq_len": seq_len}


def int8_head(V: int = 128256, d: int = 4096, B: int = 512, n_dup: int = 8):
    """Integer-only head: int8 W and h uniform in [-127, 127].

    ``n_dup`` W rows are copies of other rows (exact integer ties), so that the
    lowest-index rule is exercised; pairs straddle tiles and sit far apart.
    """
    W = uniform_int8(SEED_W + 5, (V, d))
    rng = _rng(SEED_X + 5)
    pairs = []
    for _ in range(n_dup):
        a, b = (int(x) for x in rng.choice(V, size=2, replace=False))
        W[b] = W[a]
        pairs.append((a, b))
    h = uniform_int8(SEED_H + 5, (B, d))
    # rows that point straight at a duplicated W row make the tie the winner
    for k, (a, _) in enumerate(pairs[: min(n_dup, B)]):
        h[k] = W[a]
    return {"W": W, "h": h, "V": V, "d": d, "dtype": "int8", "dup_pairs": pairs}


def small_float(seed: int, V: int, d: int, B: int, fmt: str = "bf16",
                sigma_w: float = 0.02, sigma_h: float = 1.0, n_ties: int = 0,
                n_near: int = 0):
    """Small float case for parity tests: ragged V and d, optional exact ties
    and near ties.

    Exact ties copy a W row; hidden rows 0..n_ties-1 are then drawn close to
    the copied row so the tie is the winner. Near ties (hidden rows n_ties ..
    n_ties+n_near-1) copy a W row with one or two elements moved by one step
    of the storage format, so the two best logits differ by far less than a
    16-bit step of their value.
    """
    rng = _rng(seed)
    Wf = _normal_f32(rng, (V, d), sigma_w)
    hf = _normal_f32(rng, (B, d), sigma_h)
    conv = bf16_bits_from_f32 if fmt == "bf16" else f16_bits_from_f32
    W = conv(Wf)
    h = conv(hf)
    for k in range(min(n_ties, B) if V >= 2 else 0):
        a, b = (int(x) for x in rng.choice(V, size=2, replace=False))
        W[b] = W[a]
        wa = (W[a].astype(np.uint32) << 16).view(np.float32) if fmt == "bf16" \
            else W[a].view(np.float16).astype(np.float32)
        h[k] = conv(np.float32(40.0) * wa / np.float32(np.linalg.norm(wa) + 1e-30)
                    + _normal_f32(rng, (d,), 0.01))
    for k in range(n_ties, min(n_ties + n_near, B) if V >= 2 else 0):
        a, b = (int(x) for x in rng.choice(V, size=2, replace=False))
        row = W[a].copy()
        for p in rng.choice(d, size=min(1 + (k % 2), d), replace=False):
            row[p] = _next_bf16_bits(row[p], bool(rng.integers(0, 2)))
        W[b] = row
        wa = (W[a].astype(np.uint32) << 16).view(np.float32) if fmt == "bf16" \
            else W[a].view(np.float16).astype(np.float32)
        h[k] = conv(np.float32(40.0) * wa / np.float32(np.linalg.norm(wa) + 1e-30)
                    + _normal_f32(rng, (d,), 0.01))
    targets = rng.integers(0, V, size=B).astype(np.int32)
    return {"W": W, "h": h, "targets": targets, "V": V, "d": d, "dtype": fmt}


def small_int8(seed: int, V: int, d: int, B: int, n_ties: int = 0,
               lo: int = -127, hi: int = 127):
    rng = _rng(seed)
    W = rng.integers(lo, hi + 1, size=(V, d), dtype=np.int8)
    h = rng.integers(lo, hi + 1, size=(B, d), dtype=np.int8)
    for k in range(min(n_ties, B) if V >= 2 else 0):
        a, b = (int(x) for x in rng.choice(V, size=2, replace=False))
        W[b] = W[a]
        h[k] = W[a]
    return {"W": W, "h": h, "V": V, "d": d, "dtype": "int8"}


def plant_drafts(tokens: np.ndarray, V: int, seed: int):
    """Drafted tokens for a speculative-verify block with planted agreement.

    ``tokens`` [R, P] are reference tokens supplied by the caller. Request r
    copies its first ``cut[r]`` tokens (cut ~ U{0 .. P}, so some requests
    agree everywhere), replaces position ``cut[r]`` by a different id and
    draws the rest uniformly. Returns (drafts int32 [R, P], cut int64 [R]).
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    R, P = tokens.shape
    rng = _rng(seed)
    cut = rng.integers(0, P + 1, size=R)
    drafts = tokens.copy()
    for r in range(R):
        c = int(cut[r])
        if c < P:
            drafts[r, c] = (tokens[r, c] + 1 + rng.integers(0, max(V - 1, 1))) % V
            drafts[r, c + 1:] = rng.integers(0, V, size=P - c - 1)
    return drafts.astype(np.int32), cut


def float_rows(seed: int, B: int, d: int, fmt: str, special: bool = True):
    """Float hidden rows for the integer front end, as raw storage (uint16
    for bf16 / fp16, uint32 for fp32). Rows are N(0, 1) times a per-row scale
    2^U{-20..20}; with ``special`` the first rows are an all-zero row, a row
    with one non-zero entry, a row of subnormals and a row near the format's
    largest values (when B allows)."""
    rng = _rng(seed)
    x = _normal_f32(rng, (B, d), 1.0) * np.exp2(rng.integers(-20, 21, size=(B, 1))).astype(np.float32)
    if special:
        tiny = {"bf16": 2.0 ** -130, "fp16": 2.0 ** -20, "fp32": 2.0 ** -140}[fmt]
        big = {"bf16": 1e38, "fp16": 6e4, "fp32": 3e38}[fmt]
        rows = [np.zeros(d, np.float32)]
        one = np.zeros(d, np.float32)
        one[rng.integers(0, d)] = -3.0
        rows.append(one)
        rows.append((rng.integers(-4, 5, size=d) * tiny).astype(np.float32))
        rows.append(np.clip(_normal_f32(rng, (d,), 0.4), -1, 1).astype(np.float32) * np.float32(big))
        for k, r in enumerate(rows[:B]):
            x[k] = r
    if fmt == "bf16":
        return bf16_bits_from_f32(x)
    if fmt == "fp16":
        return f16_bits_from_f32(np.clip(x, -65504, 65504))
    return x.view(np.uint32).copy()
