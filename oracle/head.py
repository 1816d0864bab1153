"""CPU oracle of the output head -- TEST INFRASTRUCTURE ONLY (see package doc).

Sources, by page title:

* [Precision] "Greedy Decoding Has a Precision Clause" -- section "Token-ranking
  margins explain why numerical error sometimes matters": the lm_head maps the
  final hidden representation to vocabulary scores (logits); greedy decoding
  takes the highest score; the top-two logit margin decides how easily a
  perturbation flips the choice.
* [DetLLM] "Eliminating Nondeterminism in LLM Inference with Integer-Only
  Arithmetic" -- section "DetLLM" (int8 x int8 -> int32 matmul; argmax breaks
  ties toward the lowest token id) and section "What if we don't use floats at
  all?" (integer sums are order-free while they cannot overflow, and the
  overflow can be bounded in advance).
* [Exactness] "TandemLLM docs, 12 Exactness" -- section 12.2 "The exception:
  near ties": the head returns fp32 logits; the gap between the two best
  logits is reported in bf16 units in the last place (ulps); observed gaps are
  fractions of an ulp, so the gap is a real number, not a count.
* [Decoding] "Inference and Decoding" -- section 3 "The sampling methods",
  Temperature: p_i = exp(z_i / tau) / sum_j exp(z_j / tau); tau = 1 here.
* [LogprobGap] "batch-logprob-gap" -- the trainer's per-token log-probability
  log p(target) and the ratio exp(logp_new - logp_old).
* [Precision] section "Correct the vulnerable token decisions, not every
  calculation": ordinary inference is left as it is unless the top-two margin
  of its logits is below a threshold tau (0.001 in the page's experiments);
  at such a step the output projection is recomputed in FP32 and the token is
  taken from that. The ordinary head is a 16-bit one, so its logits are the
  16-bit roundings of the products' sums.
* [Exactness] section 12.5 (Sampling): a request with a seed draws
  the token at index t as the argmax of log p_t + G_t, G_t Gumbel noise from
  a generator seeded by (seed, t) -- an exact sample from p_t that does not
  depend on what else was computed. [Decoding] section 3: p = softmax(z/T).
* [DetLLM] section "DetLLM": every tensor carries a dyadic scale (an integer
  multiplier and a shift, one fixed rounding rule); each token's activations
  are quantized from that token's own values, so its bits cannot depend on
  the rest of the batch.
* [Decoding] section 6 (Speculative decoding): the target scores all drafted
  positions in one forward pass and keeps the drafted tokens while they agree
  with it; [Exactness] 12.1: greedy speculative output equals plain greedy
  decoding, so at temperature 0 "agree" means "equals the greedy token".

Readings where the pages are silent (each also listed with the design notes):

* the logit is the raw product h . w, no bias, no temperature, no rounding of
  the logit to bf16 ([Exactness] 12.2: the head returns fp32 logits);
* "second value" is the runner-up of the multiset of logits, so an exact tie
  gives a gap of zero;
* the ulp is the bf16 ulp of the winning logit m:
  ulp(m) = 2^(max(floor(log2|m|), -126) - 7), i.e. bf16's 8-bit significand
  at m's binade, never below bf16's smallest normal binade;
* with a single vocabulary entry there is no runner-up: s = -inf, gap = +inf
  (float heads) and gap = INT32_MAX (integer head);
* the integer head's gap is the exact integer m - s (a bf16 ulp has no meaning
  for int32 logits);
* a target id outside [0, V) has no log-probability: NaN;
* margin gate: the ordinary 16-bit head's logits are the exact logits rounded
  once, to nearest with ties to even, into the head's storage format (bf16 or
  fp16); its token is the lowest index of their maximum; the margin is the
  difference of the two largest rounded values of the multiset (zero on a
  tie), rounded once to float32; the gate fires when margin < tau (tau and
  the comparison in float32); a fired row takes the FP32 recompute over the
  full vocabulary, i.e. the argmax of the unrounded logits;
* seeded sampling: the pages name no generator. Philox4x32-10 (Salmon et al.,
  "Parallel random numbers: as easy as 1, 2, 3", SC'11) keyed by the 64-bit
  seed (low word first); entry v of position t takes word (v mod 4) of the
  block with counter (v div 4, t low word, t high word, 0); a word x maps to
  the uniform U = (2 floor(x / 2^9) + 1) 2^-24 in (0, 1), exact in float32;
  G = -log(-log U). log p_t + G differs from z/T + G by a constant per row,
  so the sample is the argmax of z/T + G (lowest index on a tie);
* integer front end: a float row x (bf16, fp16 or fp32 values, exact
  dyadic rationals) becomes int8 q = RNE(x * M / 2^S) with amax = max |x|,
  E = floor(log2 amax), S = E + 8 and M = floor(127 * 2^S / amax) (a 15-bit
  multiplier in [16256, 32512]); RNE rounds to nearest, ties to even; the
  largest element maps to +-127 and no value leaves [-127, 127]; an all-zero
  row gives q = 0, M = 0, S = 0. x ~ q * 2^S / M.
"""
from __future__ import annotations

import numpy as np

INT32_MAX = 2**31 - 1


# --------------------------------------------------------------------------
# Exact decoding of the stored formats
# --------------------------------------------------------------------------

def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64, exactly (bf16 is the top half of fp32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def decode_fp16(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64, exactly (subnormals included)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def decode_int8(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.int8).astype(np.int64)


def decode_fp32(bits: np.ndarray) -> np.ndarray:
    """IEEE binary32 bit patterns (uint32) -> float64, exactly."""
    return np.asarray(bits, dtype=np.uint32).view(np.float32).astype(np.float64)


def decode(arr: np.ndarray, fmt: str) -> np.ndarray:
    if fmt == "fp32":
        return decode_fp32(arr)
    if fmt == "bf16":
        return decode_bf16(arr)
    if fmt == "fp16":
        return decode_fp16(arr)
    if fmt == "int8":
        return decode_int8(arr)
    raise ValueError(f"unknown format {fmt!r}")


# --------------------------------------------------------------------------
# Logits
# --------------------------------------------------------------------------

def logits_float(W: np.ndarray, h: np.ndarray):
    """Float head logits z[n, v] = sum_k h[n, k] * W[v, k]   ([Precision]).

    ``W`` [V, d] and ``h`` [B, d] are float64 (exactly decoded inputs). Every
    product of two bf16/fp16 values is exact in float64; the float64 sum adds
    at most d * 2^-53 * sum|w h| of error, negligible against the 1e-6 * sum|w h|
    tolerance the GPU is held to.

    Returns (z, A) where A[n, v] = sum_k |h[n, k] * W[v, k]| is the error base
    of the per-entry tolerance.
    """
    z = h @ W.T
    A = np.abs(h) @ np.abs(W).T
    return z, A


def logits_int(W: np.ndarray, h: np.ndarray) -> np.ndarray:
    """Integer head logits z[n, v] = sum_k h[n, k] * W[v, k], exactly ([DetLLM]).

    int64 accumulation: |z| <= d * 128^2, far below 2^63, so the int64 sum
    is exact in any order.
    """
    return np.asarray(h, dtype=np.int64) @ np.asarray(W, dtype=np.int64).T


def logits_int_f64(W: np.ndarray, h: np.ndarray) -> np.ndarray:
    """The same exact integer logits through a float64 matrix product ([DetLLM]).

    Every product of two int8 values is an integer of magnitude <= 2^14, and
    every partial sum of d of them, in any order or grouping, is an integer of
    magnitude <= d * 2^14 < 2^53 (d < 2^39): each float64 addition (or fused
    multiply-add) is then exact, so the result is the exact integer whatever
    order the matrix product takes -- the float64 product is used only for
    its speed on large row counts.
    """
    d = np.asarray(W).shape[1]
    if d * 128 * 128 >= 2**53:
        raise ValueError("partial sums could exceed 2^53")
    z = np.asarray(h, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T
    return z.astype(np.int64)


def bigint_dot(w_row, h_row) -> int:
    """One logit by Python big-integer arithmetic (no overflow possible)."""
    return sum(int(a) * int(b) for a, b in zip(w_row.tolist(), h_row.tolist()))


# --------------------------------------------------------------------------
# Token decision: argmax, runner-up, gap in bf16 ulps
# --------------------------------------------------------------------------

def ulp_bf16(m) -> np.ndarray:
    """bf16 unit in the last place at the binade of m ([Exactness] 12.2).

    2^(E - 7) with E = floor(log2 |m|) clamped below at -126 (bf16's smallest
    normal exponent; m = 0 falls there too).
    """
    m = np.asarray(m, dtype=np.float64)
    _, e = np.frexp(np.abs(m))          # |m| = f * 2^e, f in [0.5, 1)
    E = np.where(m == 0, -126, np.maximum(e - 1, -126))
    return np.ldexp(1.0, E - 7)


def top2(z: np.ndarray):
    """Greedy winner and runner-up value, row by row ([DetLLM], [Precision]).

    token = the lowest index attaining the row maximum (numpy's argmax returns
    the first occurrence); m = the maximum; s = the second element of the row
    sorted in descending order (equal to m on an exact tie; -inf if V = 1).
    """
    z = np.asarray(z)
    token = np.argmax(z, axis=1).astype(np.int64)
    m = z[np.arange(z.shape[0]), token]
    if z.shape[1] >= 2:
        s = np.sort(z, axis=1)[:, -2]
    else:
        s = np.full(z.shape[0], -np.inf if z.dtype.kind == "f" else None)
    return token, m, s


def greedy(z: np.ndarray):
    """Float head decision: (token, gap in bf16 ulps of the winner, m, s)."""
    token, m, s = top2(np.asarray(z, dtype=np.float64))
    with np.errstate(invalid="ignore"):
        gap = (m - s) / ulp_bf16(m)
    return token, gap, m, s


def greedy_int(z: np.ndarray):
    """Integer head decision: (token, exact gap m - s, m, s) ([DetLLM])."""
    z = np.asarray(z, dtype=np.int64)
    token = np.argmax(z, axis=1).astype(np.int64)
    m = z[np.arange(z.shape[0]), token]
    if z.shape[1] >= 2:
        s = np.sort(z, axis=1)[:, -2]
        gap = m - s
    else:
        s = np.full(z.shape[0], np.iinfo(np.int64).min)
        gap = np.full(z.shape[0], INT32_MAX, dtype=np.int64)
    return token, gap, m, s


def gap_from_top2_f32(m32: np.ndarray, s32: np.ndarray) -> np.ndarray:
    """The float32 gap the head reports for its own float32 top-2 values.

    (m - s) / ulp_bf16(m) evaluated exactly (float64 difference of two float32
    values, scaling by a power of two) and rounded once to float32.
    """
    m = np.asarray(m32, dtype=np.float32).astype(np.float64)
    s = np.asarray(s32, dtype=np.float32).astype(np.float64)
    with np.errstate(invalid="ignore"):
        return ((m - s) / ulp_bf16(m)).astype(np.float32)


# --------------------------------------------------------------------------
# Log-sum-exp and the target log-probability
# --------------------------------------------------------------------------

def logsumexp(z: np.ndarray) -> np.ndarray:
    """log sum_v exp(z[n, v]) at temperature 1 ([Decoding] section 3).

    Shifted by the row maximum M so that no exp overflows:
    lse = M + log(sum_v exp(z_v - M)).
    """
    z = np.asarray(z, dtype=np.float64)
    M = np.max(z, axis=1)
    return M + np.log(np.sum(np.exp(z - M[:, None]), axis=1))


def logprob(z: np.ndarray, targets: np.ndarray) -> np.ndarray:
    """log p(target) = z[n, target_n] - logsumexp(z[n])   ([LogprobGap]).

    Targets outside [0, V) give NaN.
    """
    z = np.asarray(z, dtype=np.float64)
    t = np.asarray(targets, dtype=np.int64)
    B, V = z.shape
    ok = (t >= 0) & (t < V)
    zt = np.where(ok, z[np.arange(B), np.where(ok, t, 0)], np.nan)
    return zt - logsumexp(z)


# --------------------------------------------------------------------------
# Whole-head entry points (what one library call computes)
# --------------------------------------------------------------------------

def head_greedy(W_raw: np.ndarray, h_raw: np.ndarray, fmt: str) -> dict:
    """Greedy call: logits, token and top-2 gap for every hidden row."""
    if fmt == "int8":
        z = logits_int(decode_int8(W_raw), decode_int8(h_raw))
        token, gap, m, s = greedy_int(z)
        return {"logits": z, "token": token, "gap": gap, "m": m, "s": s}
    z, A = logits_float(decode(W_raw, fmt), decode(h_raw, fmt))
    token, gap, m, s = greedy(z)
    return {"logits": z, "A": A, "token": token, "gap": gap, "m": m, "s": s}


def head_logprob(W_raw: np.ndarray, h_raw: np.ndarray, targets: np.ndarray,
                 fmt: str) -> dict:
    """Log-prob call: logp of each row's target, with lse and the logits."""
    if fmt not in ("bf16", "fp16"):
        raise ValueError("the log-probability is defined for the float heads")
    z, A = logits_float(decode(W_raw, fmt), decode(h_raw, fmt))
    lse = logsumexp(z)
    lp = logprob(z, targets)
    return {"logits": z, "A": A, "lse": lse, "logp": lp}


# --------------------------------------------------------------------------
# Greedy speculative-verify acceptance
# --------------------------------------------------------------------------

def verify_accept(tokens: np.ndarray, drafts: np.ndarray) -> np.ndarray:
    """Accepted draft length per request ([Decoding] section 6, [Exactness] 12.1).

    tokens [R, P]: the target's greedy token at each of a request's P verified
    positions; drafts [R, P]: the token the drafter proposed for each
    position. Accepted = the number of leading positions whose draft equals
    the target's token (0 .. P); the caller keeps those drafts and takes the
    target's token at the first mismatch.
    """
    tokens = np.asarray(tokens)
    drafts = np.asarray(drafts)
    R, P = tokens.shape
    out = np.empty(R, dtype=np.int64)
    for r in range(R):
        a = 0
        while a < P and drafts[r, a] == tokens[r, a]:
            a += 1
        out[r] = a
    return out



# --------------------------------------------------------------------------
# Margin-gated FP32 recompute
# --------------------------------------------------------------------------

# (significand bits after the point, smallest normal exponent, largest finite)
_FORMATS = {
    "bf16": (7, -126, (2.0 - 2.0 ** -7) * 2.0 ** 127),
    "fp16": (10, -14, 65504.0),
}


def round_to_format(x, fmt: str) -> np.ndarray:
    """Round float64 values once to the nearest value of bf16 or fp16, ties to
    even (IEEE 754 roundTiesToEven), returned as float64.

    In the binade [2^E, 2^(E+1)) (E clamped below at the smallest normal
    exponent, which also covers the subnormals) the format's numbers are the
    multiples of q = 2^(E - p); |x| / q is exact, np.rint rounds it half to
    even, and a result above the largest finite value overflows to infinity.
    """
    p, emin, vmax = _FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, e = np.frexp(ax)
    E = np.maximum(e - 1, emin)
    q = np.ldexp(1.0, E - p)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.rint(ax / q) * q
    r = np.where(r > vmax, np.inf, r)
    return np.copysign(r, x)


def gated_greedy(z: np.ndarray, tau: float, fmt: str) -> dict:
    """Margin-gated decision ([Precision], "Correct the vulnerable token
    decisions"), row by row.

    z [B, V]: the unrounded logits (exact, or the head's own float32 values).
    base = lowest index of the maximum of the rounded logits (the ordinary
    16-bit head's greedy token); margin = float32(M16 - S16) with M16, S16
    the two largest rounded values of the multiset; fired = margin < tau in
    float32; token = argmax of the unrounded logits (lowest index) where
    fired, else base.
    """
    z = np.asarray(z, dtype=np.float64)
    z16 = round_to_format(z, fmt)
    base = np.argmax(z16, axis=1).astype(np.int64)
    M16 = z16[np.arange(z.shape[0]), base]
    if z.shape[1] >= 2:
        S16 = np.sort(z16, axis=1)[:, -2]
    else:
        S16 = np.full(z.shape[0], -np.inf)
    with np.errstate(invalid="ignore"):
        margin = (M16 - S16).astype(np.float32)
    fired = margin < np.float32(tau)
    full = np.argmax(z, axis=1).astype(np.int64)
    token = np.where(fired, full, base)
    return {"token": token, "base": base, "margin": margin, "fired": fired}


# --------------------------------------------------------------------------
# Seeded Gumbel-max sampling
# --------------------------------------------------------------------------

_M32 = np.uint64(0xFFFFFFFF)
PHILOX_M = (np.uint64(0xD2511F53), np.uint64(0xCD9E8D57))
PHILOX_W = (np.uint64(0x9E3779B9), np.uint64(0xBB67AE85))


def philox4x32_10(counter, key) -> np.ndarray:
    """Philox4x32 with 10 rounds (Salmon et al., SC'11), vectorised.

    counter [..., 4] and key [..., 2] of 32-bit words (any integer dtype);
    returns [..., 4] uint32. One round: the products M0 * c0 and M1 * c2
    (64-bit, exact in uint64) give the new block (hi(M1 c2) ^ c1 ^ k0,
    lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key then advances by the
    Weyl increments (mod 2^32).
    """
    c = np.asarray(counter, dtype=np.uint64) & _M32
    k = np.asarray(key, dtype=np.uint64) & _M32
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0, k1 = k[..., 0], k[..., 1]
    for _ in range(10):
        p0 = PHILOX_M[0] * c0
        p1 = PHILOX_M[1] * c2
        c0, c1, c2, c3 = ((p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & _M32,
                          (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & _M32)
        k0 = (k0 + PHILOX_W[0]) & _M32
        k1 = (k1 + PHILOX_W[1]) & _M32
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniform_from_word(x) -> np.ndarray:
    """U = (2 * (x >> 9) + 1) * 2^-24: 2^23 equally spaced values in (0, 1),
    each exact in float32 (and float64)."""
    x = np.asarray(x, dtype=np.uint64)
    return ((x >> np.uint64(9)) * np.uint64(2) + np.uint64(1)).astype(np.float64) * 2.0 ** -24


def _u64_list(xs) -> list:
    """64-bit keys as Python integers in [0, 2^64), element by element (a
    list mixing values above and below 2^63 must not pass through a float
    array; negative int64 values are read as their two's-complement bits)."""
    if isinstance(xs, np.ndarray):
        xs = xs.reshape(-1).tolist()
    return [int(x) % (1 << 64) for x in xs]


def gumbel_rows(seeds, positions, V: int) -> np.ndarray:
    """G[n, v] = -log(-log U) for the (seed_n, position_n) of each row."""
    seeds = _u64_list(seeds)
    pos = _u64_list(positions)
    B = len(seeds)
    v = np.arange(V, dtype=np.uint64)[None, :].repeat(B, axis=0)
    t_lo = np.array([t & 0xFFFFFFFF for t in pos], dtype=np.uint64)[:, None].repeat(V, axis=1)
    t_hi = np.array([(t >> 32) & 0xFFFFFFFF for t in pos], dtype=np.uint64)[:, None].repeat(V, axis=1)
    counter = np.stack([v >> np.uint64(2), t_lo, t_hi, np.zeros_like(v)], axis=-1)
    k_lo = np.array([x & 0xFFFFFFFF for x in seeds], dtype=np.uint64)[:, None].repeat(V, axis=1)
    k_hi = np.array([(x >> 32) & 0xFFFFFFFF for x in seeds], dtype=np.uint64)[:, None].repeat(V, axis=1)
    words = philox4x32_10(counter, np.stack([k_lo, k_hi], axis=-1))
    x = np.take_along_axis(words, (v & np.uint64(3)).astype(np.int64)[..., None], axis=-1)[..., 0]
    return -np.log(-np.log(uniform_from_word(x)))


def gumbel_noise(seed: int, t: int, V: int) -> np.ndarray:
    """G_v = -log(-log U_v), v = 0 .. V-1, for one (seed, position)."""
    return gumbel_rows([seed], [t], V)[0]


def sample(z: np.ndarray, temperature: float, seeds, positions) -> dict:
    """Seeded Gumbel-max sample per row ([Exactness] 12.5, [Decoding] 3).

    score[n, v] = z[n, v] / T + G(seed_n, t_n)_v in float64; token = lowest
    index of the maximum score; also the best and runner-up scores (the
    runner-up of the multiset), whose difference says how near the draw was
    to going the other way.
    """
    z = np.asarray(z, dtype=np.float64)
    score = z / float(temperature) + gumbel_rows(seeds, positions, z.shape[1])
    token, m, s = top2(score)
    return {"token": token, "m": m, "s": s, "score": score}


# --------------------------------------------------------------------------
# Integer front end: per-token requantization to int8 with a dyadic scale
# --------------------------------------------------------------------------

def quantize_rows(x: np.ndarray):
    """Per-row int8 quantization with a dyadic multiplier ([DetLLM]).

    x [B, d] float64 holding exactly decoded bf16 / fp16 / fp32 values.
    Returns (q int8 [B, d], M int64 [B], S int64 [B]) with, per row,
    amax = max |x|, E = floor(log2 amax), S = E + 8,
    M = floor(127 * 2^S / amax) in exact rational arithmetic, and
    q = round-half-even(x * M * 2^-S). x * M has at most 24 + 15 significant
    bits and the scaling is a power of two, so the float64 product is exact
    and np.rint rounds it once, ties to even.
    """
    from fractions import Fraction
    x = np.asarray(x, dtype=np.float64)
    B, d = x.shape
    q = np.zeros((B, d), dtype=np.int8)
    M = np.zeros(B, dtype=np.int64)
    S = np.zeros(B, dtype=np.int64)
    for n in range(B):
        amax = float(np.max(np.abs(x[n]))) if d > 0 else 0.0
        if amax == 0.0:
            continue
        E = int(np.frexp(amax)[1]) - 1                  # amax in [2^E, 2^(E+1))
        s = E + 8
        m = (Fraction(127) * Fraction(2) ** s) // Fraction(amax)
        M[n], S[n] = int(m), s
        q[n] = np.rint(x[n] * float(m) * 2.0 ** (-s)).astype(np.int8)
    return q, M, S
