"""Pins for the CPU oracle: checks that do not re-use the oracle's formulas.

Each ``pin_*`` takes an oracle object (the ``oracle`` package, or a copy with
a planted mistake) and raises AssertionError when the oracle disagrees with
what the pages or the mathematics fix. The pins use independent routes:

* hand-worked values (``golden/tiny_head_d8_v16.txt``) and values printed on
  the pages (``golden/page_examples.txt``);
* brute force with exact rationals (``fractions.Fraction``) and Python big
  integers, with inputs decoded through ``struct`` instead of numpy views;
* 60-digit ``mpmath`` log-sum-exp and scipy's ``logsumexp`` as an outside
  library routine;
* closed forms (uniform logits, one dominant logit, the int32 bound) and
  invariants (row permutation, duplicated rows, logp <= 0, lse >= max,
  probabilities summing to one, the token-flip criterion).
"""
from __future__ import annotations

import math
import os
import struct
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# fixture readers and independent helpers
# --------------------------------------------------------------------------

def read_tiny():
    W, h, z, tok, gap = {}, {}, {}, {}, {}
    with open(os.path.join(GOLDEN, "tiny_head_d8_v16.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":", 1)
            kind, idx = key.split()
            idx = int(idx)
            nums = [Fraction(x) for x in vals.split()]
            {"W": W, "h": h, "z": z, "token": tok, "gap": gap}[kind][idx] = nums
    Wm = [W[i] for i in range(len(W))]
    hm = [h[i] for i in range(len(h))]
    zm = [z[i] for i in range(len(z))]
    return Wm, hm, zm, [int(tok[i][0]) for i in range(len(tok))], \
        [gap[i][0] for i in range(len(gap))]


def read_page_examples():
    out = {}
    with open(os.path.join(GOLDEN, "page_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = float(v)
    return out


def bf16_bits_of(x: Fraction) -> int:
    """bf16 bit pattern of a value that is exact in bf16 (via struct)."""
    b = struct.unpack(">I", struct.pack(">f", float(x)))[0]
    assert b & 0xFFFF == 0, f"{x} is not exact in bf16"
    return b >> 16


def exact_bf16(bits: int) -> Fraction:
    return Fraction(struct.unpack(">f", struct.pack(">I", int(bits) << 16))[0])


def exact_fp16(bits: int) -> Fraction:
    return Fraction(struct.unpack("<e", struct.pack("<H", int(bits)))[0])


def exact_ulp_bf16(m: Fraction) -> Fraction:
    """bf16 ulp at m's binade by exact search over powers of two."""
    a = abs(m)
    if a == 0:
        E = -126
    else:
        E = 0
        while Fraction(2) ** E > a:
            E -= 1
        while Fraction(2) ** (E + 1) <= a:
            E += 1
        E = max(E, -126)
    return Fraction(2) ** (E - 7)


def loop_argmax_lowest(row):
    best = 0
    for v in range(1, len(row)):
        if row[v] > row[best]:
            best = v
    return best


def _rand_bf16_bits(rng, shape, scale):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    u = x.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------
# pins
# --------------------------------------------------------------------------

def pin_tiny_golden(o):
    """Hand-worked d=8, V=16 case: logits, tokens, gaps, ln 16."""
    Wf, hf, zf, toks, gaps = read_tiny()
    W_bits = np.array([[bf16_bits_of(x) for x in r] for r in Wf], np.uint16)
    h_bits = np.array([[bf16_bits_of(x) for x in r] for r in hf], np.uint16)
    out = o.head_greedy(W_bits, h_bits, "bf16")
    z = out["logits"]
    assert z.shape == (len(hf), len(Wf)), z.shape
    for n in range(len(hf)):
        for v in range(len(Wf)):
            assert Fraction(float(z[n, v])) == zf[n][v], (n, v, z[n, v], zf[n][v])
        assert int(out["token"][n]) == toks[n], (n, out["token"][n], toks[n])
        assert Fraction(float(out["gap"][n])) == gaps[n], (n, out["gap"][n], gaps[n])
    lp = o.head_logprob(W_bits, h_bits, np.arange(len(hf), dtype=np.int32), "bf16")
    # h1 has all-zero logits: lse = ln 16, logp = -ln 16 (closed form)
    assert abs(lp["lse"][1] - math.log(16)) <= 1e-15
    assert abs(lp["logp"][1] + math.log(16)) <= 1e-15


def pin_bruteforce_float(o):
    """Random tiny bf16 and fp16 heads against exact rational dot products."""
    rng = np.random.default_rng(7)
    for fmt in ("bf16", "fp16"):
        V, d, B = 16, 8, 5
        if fmt == "bf16":
            Wb = _rand_bf16_bits(rng, (V, d), 0.5)
            hb = _rand_bf16_bits(rng, (B, d), 2.0)
            dec = exact_bf16
        else:
            Wb = (rng.standard_normal((V, d)) * 0.5).astype(np.float16).view(np.uint16)
            hb = (rng.standard_normal((B, d)) * 2.0).astype(np.float16).view(np.uint16)
            dec = exact_fp16
        Wq = [[dec(Wb[v, k]) for k in range(d)] for v in range(V)]
        hq = [[dec(hb[n, k]) for k in range(d)] for n in range(B)]
        out = o.head_greedy(Wb, hb, fmt)
        z = out["logits"]
        assert z.shape == (B, V)
        for n in range(B):
            ex = [sum(hq[n][k] * Wq[v][k] for k in range(d)) for v in range(V)]
            Aex = [sum(abs(hq[n][k] * Wq[v][k]) for k in range(d)) for v in range(V)]
            for v in range(V):
                # float64 sum of exact products: error <= d * 2^-53 * A
                assert abs(Fraction(float(z[n, v])) - ex[v]) <= \
                    d * Fraction(1, 2**53) * Aex[v], (fmt, n, v)
                assert abs(Fraction(float(out["A"][n, v])) - Aex[v]) <= \
                    d * Fraction(1, 2**53) * Aex[v]
            t = loop_argmax_lowest(ex)
            assert int(out["token"][n]) == t, (fmt, n)
            srt = sorted(ex, reverse=True)
            g = (srt[0] - srt[1]) / exact_ulp_bf16(srt[0])
            assert abs(Fraction(float(out["gap"][n])) - g) <= abs(g) * Fraction(1, 2**40) + \
                Fraction(1, 2**40), (fmt, n, float(out["gap"][n]), float(g))


def pin_logsumexp_mpmath(o):
    """log-sum-exp and logp against 60-digit mpmath and scipy's routine."""
    import mpmath
    from scipy.special import logsumexp as scipy_lse
    mpmath.mp.dps = 60
    rng = np.random.default_rng(11)
    V, d, B = 16, 8, 4
    Wb = _rand_bf16_bits(rng, (V, d), 1.0)
    hb = _rand_bf16_bits(rng, (B, d), 3.0)
    t = rng.integers(0, V, size=B).astype(np.int32)
    out = o.head_logprob(Wb, hb, t, "bf16")
    assert out["lse"].shape == (B,) and out["logp"].shape == (B,)
    Wq = [[exact_bf16(Wb[v, k]) for k in range(d)] for v in range(V)]
    hq = [[exact_bf16(hb[n, k]) for k in range(d)] for n in range(B)]
    for n in range(B):
        ex = [sum(hq[n][k] * Wq[v][k] for k in range(d)) for v in range(V)]
        lse = mpmath.log(mpmath.fsum(mpmath.exp(mpmath.mpf(x.numerator) / x.denominator)
                                     for x in ex))
        lp = mpmath.mpf(ex[t[n]].numerator) / ex[t[n]].denominator - lse
        assert abs(out["lse"][n] - float(lse)) <= 1e-13 * max(1.0, abs(float(lse)))
        assert abs(out["logp"][n] - float(lp)) <= 1e-13 * max(1.0, abs(float(lse)))
        zz = np.array([float(x) for x in ex])
        assert abs(out["lse"][n] - scipy_lse(zz)) <= 1e-12 * max(1.0, abs(float(lse)))


def pin_closed_forms(o):
    """Uniform logits, a dominant logit, tiny winners, out-of-range targets."""
    V = 16
    # uniform logits c: lse = c + ln V, logp = -ln V for every target
    z = np.full((3, V), [[-3.0], [0.0], [7.5]])
    lse = o.logsumexp(z)
    assert np.allclose(lse, np.array([-3.0, 0.0, 7.5]) + math.log(V), rtol=0, atol=1e-14)
    lp = o.logprob(z, np.array([0, 5, 15]))
    assert np.allclose(lp, -math.log(V), rtol=0, atol=1e-14)
    # one dominant logit L: lse = L (to double precision), no overflow at L = 1000
    z = np.zeros((1, V))
    z[0, 9] = 1000.0
    assert o.logsumexp(z)[0] == 1000.0
    assert o.logprob(z, np.array([9]))[0] == 0.0
    assert o.logprob(z, np.array([3]))[0] == -1000.0
    # large negative logits: lse stays finite
    assert np.isfinite(o.logsumexp(np.full((1, V), -1000.0)))[0]
    # out-of-range target -> NaN
    assert np.isnan(o.logprob(np.zeros((2, V)), np.array([-1, V]))).all()
    # the ulp's lower clamp: m = 2^-127, s = 0 -> ulp 2^-133, gap 64
    z = np.zeros((1, 4))
    z[0, 2] = 2.0 ** -127
    tok, gap, m, s = o.greedy(z)
    assert tok[0] == 2 and gap[0] == 64.0
    # negative winner: m = -1, s = -1 - 2^-7; ulp(-1) = 2^-7 -> gap 1
    z = np.array([[-4.0, -1.0 - 2.0 ** -7, -1.0, -2.0]])
    tok, gap, m, s = o.greedy(z)
    assert tok[0] == 2 and gap[0] == 1.0
    # V = 1: no runner-up
    tok, gap, m, s = o.greedy(np.array([[0.25]]))
    assert tok[0] == 0 and gap[0] == np.inf
    # ulp on both sides of a binade edge
    assert o.ulp_bf16(np.array([1.0]))[0] == 2.0 ** -7
    assert o.ulp_bf16(np.array([0.99609375]))[0] == 2.0 ** -8
    assert o.ulp_bf16(np.array([-3.5]))[0] == 2.0 ** -6


def pin_page_examples(o):
    """Values printed on the pages: ties, the step-0 cushion, fp limits."""
    pe = read_page_examples()
    # float non-associativity (harness arithmetic is IEEE double)
    assert (0.1 + 1e20) - 1e20 == pe["nonassoc_left"]
    assert 0.1 + (1e20 - 1e20) == pe["nonassoc_right"]
    # 2^24 + 1 rounds to 2^24 in fp32
    lim = np.float32(pe["fp32_int_limit"])
    assert lim + np.float32(1) == lim and lim - np.float32(1) != lim
    # step 457: a 0.03 lead wins; an exact tie goes to the lower id (" is")
    id_is, id_introduces = 3, 11
    z = np.zeros((2, 16))
    z[0, id_introduces] = 5.0 + pe["step457_lead"]
    z[0, id_is] = 5.0
    z[1, id_introduces] = 5.0
    z[1, id_is] = 5.0
    tok, gap, _, _ = o.greedy(z)
    assert tok[0] == id_introduces and tok[1] == id_is and gap[1] == 0.0
    # step 0: shifts of at most 0.094 cannot move a winner with a 2.66 gap
    rng = np.random.default_rng(3)
    base = rng.uniform(-5, 5, size=(200, 64))
    w = rng.integers(0, 64, size=200)
    base[np.arange(200), w] = base.max(axis=1) + pe["step0_top2_gap"]
    shift = rng.uniform(-pe["step0_max_shift"], pe["step0_max_shift"], size=base.shape)
    t0, _, _, _ = o.greedy(base)
    t1, _, _, _ = o.greedy(base + shift)
    assert (t0 == w).all() and (t1 == w).all()
    # near-tie gaps are fractions of an ulp: in the binade [1, 2) the bf16 ulp
    # is 2^-7, so logits 1.5 and 1.5 - g * 2^-7 are g ulp apart
    for g in (pe["near_tie_gap_min_ulp"], pe["near_tie_gap_max_ulp"]):
        z = np.array([[1.5 - g * 2.0 ** -7, 1.5, -2.0]])
        tok, gap, m, s = o.greedy(z)
        assert tok[0] == 1
        assert abs(gap[0] - g) <= 1e-12 and gap[0] < pe["one_ulp_rule"]


def pin_int_head(o):
    """Integer head: closed-form bound, big-integer dots, int ties."""
    d = 4096
    W = np.full((3, d), 127, np.int8)
    W[1] = -127
    W[2, :] = -128
    h = np.full((2, d), 127, np.int8)
    h[1] = -128
    out = o.head_greedy(W, h, "int8")
    z = out["logits"]
    assert z.shape == (2, 3)
    # d * 127^2 = 66,064,384 < 2^31: the int32 accumulator cannot overflow
    assert int(z[0, 0]) == 66_064_384 == d * 127 * 127 < 2**31
    assert int(z[0, 1]) == -66_064_384
    assert int(z[1, 2]) == d * 128 * 128 == 2**26
    rng = np.random.default_rng(5)
    V, d, B = 40, 24, 6
    W = rng.integers(-128, 128, size=(V, d), dtype=np.int8)
    W[33] = W[7]                      # exact tie: rows 7 and 33
    h = rng.integers(-128, 128, size=(B, d), dtype=np.int8)
    h[0] = W[7]
    out = o.head_greedy(W, h, "int8")
    for n in range(B):
        ex = [sum(int(a) * int(b) for a, b in zip(W[v].tolist(), h[n].tolist()))
              for v in range(V)]
        assert [int(x) for x in out["logits"][n]] == ex, n
        t = loop_argmax_lowest(ex)
        assert int(out["token"][n]) == t
        srt = sorted(ex, reverse=True)
        assert int(out["gap"][n]) == srt[0] - srt[1]
    assert int(out["token"][0]) == 7 and int(out["gap"][0]) == 0
    assert o.bigint_dot(W[3], h[2]) == sum(int(a) * int(b) for a, b in
                                            zip(W[3].tolist(), h[2].tolist()))
    # the float64 product gives the same integers: random rows, and the
    # extremes (sums of 16384 products of +-128, |z| = 2^28, where a float32
    # sum would have rounded)
    for z64 in (o.logits_int_f64(W, h),):
        assert z64.dtype == np.int64
        for n in range(B):
            ex = [sum(int(a) * int(b) for a, b in zip(W[v].tolist(), h[n].tolist()))
                  for v in range(V)]
            assert [int(x) for x in z64[n]] == ex, n
    d = 16384
    We = np.full((2, d), -128, np.int8)
    We[1] = 127
    he = np.full((2, d), -128, np.int8)
    he[1] = 127
    he[1, -1] = -128
    ze = o.logits_int_f64(We, he)
    for n in range(2):
        for v in range(2):
            assert int(ze[n, v]) == o.bigint_dot(We[v], he[n])
    assert int(ze[0, 0]) == 2**28
    # 127^2 (d - 1) - 127 * 128 = 264,225,151: odd and above 2^24, so no
    # float32 holds it
    assert int(ze[1, 1]) == 127 * 127 * (d - 1) - 127 * 128 == 264_225_151


def pin_invariants(o):
    """Row permutation, duplicated rows, logp <= 0, lse >= max, sum p = 1, flips."""
    rng = np.random.default_rng(21)
    V, d, B = 37, 16, 9
    Wb = _rand_bf16_bits(rng, (V, d), 0.3)
    hb = _rand_bf16_bits(rng, (B, d), 1.0)
    hb[4] = hb[1]                                  # duplicated row
    t = rng.integers(0, V, size=B).astype(np.int32)
    g = o.head_greedy(Wb, hb, "bf16")
    lp = o.head_logprob(Wb, hb, t, "bf16")
    perm = rng.permutation(B)
    gp = o.head_greedy(Wb, hb[perm], "bf16")
    lpp = o.head_logprob(Wb, hb[perm], t[perm], "bf16")
    assert (gp["token"] == g["token"][perm]).all()
    assert (gp["gap"] == g["gap"][perm]).all()
    assert (lpp["logp"] == lp["logp"][perm]).all()
    assert g["token"][4] == g["token"][1] and g["gap"][4] == g["gap"][1]
    assert (lp["logp"] <= 0).all()
    assert (lp["lse"] >= g["logits"].max(axis=1)).all()
    # sum over all targets of p = 1
    allt = o.logprob(np.repeat(lp["logits"][:1], V, axis=0), np.arange(V))
    assert abs(np.exp(allt).sum() - 1.0) <= 1e-12
    assert (g["gap"] >= 0).all()
    # gap == 0 exactly when the maximum is attained twice
    z = g["logits"]
    ties = (z == z.max(axis=1, keepdims=True)).sum(axis=1) >= 2
    assert ((g["gap"] == 0) == ties).all()
    # token-flip criterion ("Greedy Decoding Has a Precision Clause", section
    # "Token-ranking margins ..."): with winner v1 and perturbation D, the
    # winner changes iff some v != v1 has D(v) - D(v1) >= z(v1) - z(v), with
    # equality enough only for v < v1 (an exact tie goes to the lower id).
    # Dyadic values keep every sum exact.
    for _ in range(300):
        z = rng.integers(-64, 64, size=(1, 12)) / 8.0
        D = rng.integers(-8, 9, size=(1, 12)) / 8.0
        v1 = int(o.greedy(z)[0][0])
        changed = int(o.greedy(z + D)[0][0]) != v1
        pred = False
        for v in range(12):
            if v == v1:
                continue
            lhs = D[0, v] - D[0, v1]
            rhs = z[0, v1] - z[0, v]
            if lhs > rhs or (lhs == rhs and v < v1):
                pred = True
        assert changed == pred


def pin_gap_from_top2(o):
    """The float32 gap the library must report for its own top-2 values."""
    m = np.array([1.0, 4.03125, 0.5, -1.0, 3.0], np.float32)
    s = np.array([0.99609375, 4.0, 0.5, -1.0078125, -3.0], np.float32)
    g = o.gap_from_top2_f32(m, s)
    assert g.dtype == np.float32
    assert g.tolist() == [0.5, 1.0, 0.0, 1.0, 6.0 / 2.0 ** -6]


def pin_verify_accept(o):
    """Accepted draft length: hand-worked cases and the defining property."""
    toks = np.array([[5, 7, 9, 11],      # drafts all agree -> 4
                     [5, 7, 9, 11],      # first position disagrees -> 0
                     [5, 7, 9, 11],      # third disagrees -> 2
                     [1, 1, 1, 1]])      # agrees, then disagrees, then agrees -> 1
    drafts = np.array([[5, 7, 9, 11],
                       [6, 7, 9, 11],
                       [5, 7, 8, 11],
                       [1, 2, 1, 1]])
    assert o.verify_accept(toks, drafts).tolist() == [4, 0, 2, 1]
    rng = np.random.default_rng(9)
    t = rng.integers(0, 3, size=(200, 16))
    d = np.where(rng.random((200, 16)) < 0.8, t, rng.integers(0, 3, size=(200, 16)))
    a = o.verify_accept(t, d)
    for r in range(200):
        assert (d[r, :a[r]] == t[r, :a[r]]).all()
        assert a[r] == 16 or d[r, a[r]] != t[r, a[r]]


# ---- rounding into the 16-bit formats, by exact search over bit patterns

def _format_table(fmt):
    """All non-negative finite values of the format, ascending, with their
    bit patterns (decoded through struct, not numpy)."""
    if fmt == "bf16":
        bits = range(0x0000, 0x7F80)
        vals = [struct.unpack(">f", struct.pack(">I", b << 16))[0] for b in bits]
    else:
        bits = range(0x0000, 0x7C00)
        vals = [struct.unpack("<e", struct.pack("<H", b))[0] for b in bits]
    return list(vals), list(bits)


_TABLES = {}


def exact_round(x: float, fmt: str) -> float:
    """Nearest value of the format by exact rational comparison; on a tie the
    one whose bit pattern is even; beyond the largest finite value by half a
    step or more (ties included, as the step above is even), infinity."""
    import bisect
    if fmt not in _TABLES:
        _TABLES[fmt] = _format_table(fmt)
    vals, bits = _TABLES[fmt]
    ax = Fraction(abs(x))
    vmax = Fraction(vals[-1])
    step = vmax - Fraction(vals[-2])
    if ax >= vmax + step / 2:
        return math.copysign(math.inf, x)
    k = bisect.bisect_left(vals, float(ax))
    if k < len(vals) and Fraction(vals[k]) == ax:
        r = vals[k]
    else:
        lo, hi = vals[k - 1], vals[k]
        dl, dh = ax - Fraction(lo), Fraction(hi) - ax
        if dl < dh:
            r = lo
        elif dh < dl:
            r = hi
        else:
            r = lo if bits[k - 1] % 2 == 0 else hi
    return math.copysign(r, x)


def pin_round_to_format(o):
    """Rounding into bf16 / fp16: hand-picked midpoints, subnormals and
    overflow, brute force on random float64 values, and the library
    conversions (torch float32 -> bfloat16, numpy float32 -> float16) on
    random float32 values."""
    hand = {
        "bf16": [(1 + 2 ** -8, 1.0), (1 + 3 * 2 ** -8, 1 + 2 ** -6), (-(1 + 2 ** -8), -1.0),
                 (2 ** -134, 0.0), (1.5 * 2 ** -133, 2 ** -132), ((2 - 2 ** -8) * 2 ** 127, math.inf),
                 ((2 - 2 ** -7) * 2 ** 127, (2 - 2 ** -7) * 2 ** 127), (3.0 + 2 ** -8, 3.0)],
        "fp16": [(65520.0, math.inf), (65519.0, 65504.0), (2 ** -25, 0.0),
                 (1.5 * 2 ** -24, 2 ** -23), (2.5 * 2 ** -24, 2 ** -23), (2 + 2 ** -10, 2.0),
                 (2 + 3 * 2 ** -10, 2 + 2 ** -8)],
    }
    for fmt, cases in hand.items():
        got = o.round_to_format(np.array([c[0] for c in cases]), fmt)
        assert got.tolist() == [c[1] for c in cases], (fmt, got)
    rng = np.random.default_rng(21)
    for fmt, scale in (("bf16", 8.0), ("fp16", 8.0)):
        x = rng.normal(0, scale, 300) * np.exp2(rng.integers(-20, 20, 300))
        x = np.concatenate([x, rng.normal(0, 1e-6, 40)])
        got = o.round_to_format(x, fmt)
        want = [exact_round(float(v), fmt) for v in x]
        assert got.tolist() == want, fmt
    x32 = (rng.normal(0, 4, 4000) * np.exp2(rng.integers(-30, 30, 4000))).astype(np.float32)
    import torch
    lib_bf16 = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert (o.round_to_format(x32.astype(np.float64), "bf16") == lib_bf16).all()
    with np.errstate(over="ignore"):
        lib_fp16 = x32.astype(np.float16).astype(np.float64)
    assert (o.round_to_format(x32.astype(np.float64), "fp16") == lib_fp16).all()


def _loop_gated(row, tau, fmt):
    """Gated decision of one row by Python loops over exactly rounded values."""
    r16 = [exact_round(float(v), fmt) for v in row]
    base, M = 0, r16[0]
    for v in range(1, len(row)):
        if r16[v] > M:
            base, M = v, r16[v]
    rest = sorted(r16, reverse=True)
    S = rest[1] if len(rest) > 1 else -math.inf
    margin = np.float32(M - S) if S != -math.inf else np.float32(math.inf)
    fired = bool(margin < np.float32(tau))
    full = loop_argmax_lowest(list(row))
    return (full if fired else base), base, float(margin), fired


def pin_gated_greedy(o):
    """Margin gate: hand-worked rows, brute force on small rows, and the
    consequence of monotone rounding (with tau > 0 the gated token is the
    argmax of the unrounded logits)."""
    cases = [  # (row, tau, fmt) -> (token, base, margin, fired)
        ([2.0, 2.0 + 2 ** -10, 1.0], 0.001, "bf16", (1, 0, 0.0, True)),
        ([1.0, 3.0, 3.0 - 2 ** -6], 0.001, "bf16", (1, 1, 2 ** -6, False)),
        ([5.0, 5.0], 0.001, "bf16", (0, 0, 0.0, True)),
        ([2.0, 2.0 + 2 ** -10, 1.0], 0.0, "bf16", (0, 0, 0.0, False)),
        ([1.0, 3.0, 3.0 - 2 ** -6], 0.02, "bf16", (1, 1, 2 ** -6, True)),
        ([3.0 + 2 ** -8, 3.0], 0.001, "bf16", (0, 0, 0.0, True)),
        ([2.0, 2.0 + 2 ** -8], 0.001, "bf16", (1, 0, 0.0, True)),
        ([2.0, 2.0 + 2 ** -8], 0.001, "fp16", (1, 1, 2 ** -8, False)),
        ([2.0, 2.0 + 2 ** -12, -7.0], 0.001, "fp16", (1, 0, 0.0, True)),
        ([-4.0, -4.0 - 2 ** -5, -4.0 + 2 ** -8], 0.001, "bf16", (2, 0, 0.0, True)),
        ([-4.0, -4.0 - 2 ** -5, -4.0 + 2 ** -6], 0.001, "bf16", (2, 2, 2 ** -6, False)),
    ]
    for row, tau, fmt, (tok, base, margin, fired) in cases:
        g = o.gated_greedy(np.array([row]), tau, fmt)
        got = (int(g["token"][0]), int(g["base"][0]), float(g["margin"][0]), bool(g["fired"][0]))
        assert got == (tok, base, margin, fired), (row, tau, fmt, got)
    g = o.gated_greedy(np.array([[7.0]]), 0.001, "bf16")
    assert int(g["token"][0]) == 0 and g["margin"][0] == np.inf and not g["fired"][0]
    rng = np.random.default_rng(22)
    for fmt in ("bf16", "fp16"):
        z = rng.integers(-40, 40, size=(150, 5)) / 16.0 + rng.normal(0, 0.004, (150, 5))
        for tau in (0.001, 0.0, 0.05):
            g = o.gated_greedy(z, tau, fmt)
            for n in range(z.shape[0]):
                want = _loop_gated(z[n], tau, fmt)
                got = (int(g["token"][n]), int(g["base"][n]), float(g["margin"][n]),
                       bool(g["fired"][n]))
                assert got == want, (fmt, tau, z[n], got, want)
            if tau > 0:
                assert (g["token"] == np.array([loop_argmax_lowest(list(r)) for r in z])).all()


# ---- seeded sampling

def read_philox_kat():
    out = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            w = [int(x, 16) for x in line.split()]
            out.append((w[0:4], w[4:6], w[6:10]))
    return out


def _philox_py(c, k):
    """Philox4x32-10 on Python integers (a second route, checked by the same
    published vectors as the oracle's)."""
    M0, M1, W0, W1, MASK = 0xD2511F53, 0xCD9E8D57, 0x9E3779B9, 0xBB67AE85, 0xFFFFFFFF
    c = list(c)
    k0, k1 = k
    for _ in range(10):
        p0, p1 = M0 * c[0], M1 * c[2]
        c = [(p1 >> 32) ^ c[1] ^ k0, p1 & MASK, (p0 >> 32) ^ c[3] ^ k1, p0 & MASK]
        k0, k1 = (k0 + W0) & MASK, (k1 + W1) & MASK
    return c


def pin_philox_kat(o):
    """The generator against the published known-answer vectors."""
    for c, k, r in read_philox_kat():
        assert o.philox4x32_10(np.array(c), np.array(k)).tolist() == r
        assert _philox_py(c, k) == r


def pin_gumbel_layout(o):
    """Uniform map and the (seed, t, v) -> word layout of the stated reading,
    from the Python-integer generator and math.log; the first block of seed 0,
    position 0 is the published all-zero vector."""
    u = o.uniform_from_word(np.array([0, 0xFFFFFFFF, 0x80000000, 511, 512]))
    assert u.tolist() == [2.0 ** -24, 1 - 2.0 ** -24, 0.5 + 2.0 ** -24, 2.0 ** -24, 3 * 2.0 ** -24]
    kat0 = read_philox_kat()[0][2]
    g = o.gumbel_noise(0, 0, 4)
    for v in range(4):
        U = ((kat0[v] >> 9) * 2 + 1) * 2.0 ** -24
        assert abs(g[v] - (-math.log(-math.log(U)))) <= 1e-15 * (1 + abs(g[v]))
    for seed, t, V in ((1, 0, 9), (0x123456789ABCDEF0, 77, 6), (5, (3 << 32) + 11, 5)):
        g = o.gumbel_noise(seed, t, V)
        for v in range(V):
            w = _philox_py([v >> 2, t & 0xFFFFFFFF, t >> 32, 0],
                           [seed & 0xFFFFFFFF, seed >> 32])[v & 3]
            U = ((w >> 9) * 2 + 1) * 2.0 ** -24
            assert abs(g[v] - (-math.log(-math.log(U)))) <= 1e-15 * (1 + abs(g[v])), (seed, t, v)


def pin_gumbel_max_distribution(o):
    """Gumbel-max gives exact samples of softmax(z / T) ([Exactness] 12.5):
    chi-square of 24,000 seeded draws against softmax(z / T) at two
    temperatures, and the Gumbel law's mean (Euler's constant) and variance
    (pi^2 / 6) over the noise itself."""
    z = np.array([[1.0, 0.2, -0.5, 2.0, 0.0, 1.5]])
    n = 24000
    for T, seed in ((1.0, 7), (0.5, 8)):
        tok = o.sample(np.repeat(z, n, axis=0), T, [seed] * n, list(range(n)))["token"]
        counts = np.bincount(tok, minlength=6).astype(np.float64)
        p = np.exp(z[0] / T - np.max(z[0] / T))
        p /= p.sum()
        chi2 = float(np.sum((counts - n * p) ** 2 / (n * p)))
        assert chi2 < 20.5, (T, chi2, counts, n * p)      # df = 5, p = 0.001
    G = np.concatenate([o.gumbel_noise(3, t, 1000) for t in range(40)])
    assert abs(G.mean() - 0.5772156649) < 0.02
    assert abs(G.var() - math.pi ** 2 / 6) < 0.05


def pin_sample_invariants(o):
    """Rows are independent (same seed and position, same draw, whatever the
    other rows); a tiny temperature gives the greedy token; a tie of scores
    goes to the lower index."""
    rng = np.random.default_rng(31)
    z = rng.normal(0, 2, size=(5, 40))
    seeds, pos = [11, 12, 11, 13, 11], [0, 0, 0, 1, 5]
    joint = o.sample(z, 0.8, seeds, pos)
    for n in range(5):
        one = o.sample(z[n:n + 1], 0.8, seeds[n:n + 1], pos[n:n + 1])
        assert one["token"][0] == joint["token"][n] and one["m"][0] == joint["m"][n]
    zz = np.stack([z[0], z[0]])
    two = o.sample(zz, 0.8, [11, 11], [0, 0])
    assert two["token"][0] == two["token"][1] == joint["token"][0]
    diff = o.sample(zz, 0.8, [11, 12], [0, 0])
    assert diff["m"][0] != diff["m"][1]           # the seed keys the noise
    later = o.sample(zz, 0.8, [11, 11], [0, 1])
    assert later["m"][0] != later["m"][1]         # so does the position
    big = [(1 << 64) - 3, 7, (1 << 63) + 12345]     # keys above and below 2^63 together
    mixed = o.sample(z[:3], 0.8, big, [(1 << 40) + 1, 2, 3])
    for n in range(3):
        one = o.sample(z[n:n + 1], 0.8, big[n:n + 1], [[(1 << 40) + 1, 2, 3][n]])
        assert one["m"][0] == mixed["m"][n]
    g = o.gumbel_noise((1 << 64) - 3, 9, 4)
    for v in range(4):
        w = _philox_py([0, 9, 0, 0], [0xFFFFFFFD, 0xFFFFFFFF])[v]
        assert abs(g[v] + math.log(-math.log(((w >> 9) * 2 + 1) * 2.0 ** -24))) < 1e-14
    # int64 views of the same keys read as the same bits
    assert o.sample(z[:1], 0.8, np.array([-3], np.int64), [9])["m"][0] == \
        o.sample(z[:1], 0.8, [(1 << 64) - 3], [9])["m"][0]
    cold = o.sample(z, 1e-9, seeds, pos)
    assert (cold["token"] == np.argmax(z, axis=1)).all()
    # an exact tie of scores: duplicate columns with equal noise cannot be
    # arranged, so check the index rule on the returned scores
    sc = joint["score"]
    assert (joint["token"] == np.argmax(sc, axis=1)).all()
    assert (joint["m"] >= joint["s"]).all()
    assert (joint["m"] - joint["s"] == np.sort(sc, axis=1)[:, -1] - np.sort(sc, axis=1)[:, -2]).all()


# ---- integer front end

def _quantize_exact(row):
    """One row by exact rationals: M by search, q by Python's round() of a
    Fraction (half to even)."""
    xs = [Fraction(float(v)) for v in row]
    amax = max(abs(v) for v in xs)
    if amax == 0:
        return [0] * len(xs), 0, 0
    E = 0
    while Fraction(2) ** (E + 1) <= amax:
        E += 1
    while Fraction(2) ** E > amax:
        E -= 1
    S = E + 8
    lo, hi = 0, 1 << 20
    while hi - lo > 1:                         # largest M with M * amax <= 127 * 2^S
        mid = (lo + hi) // 2
        if mid * amax <= 127 * Fraction(2) ** S:
            lo = mid
        else:
            hi = mid
    M = lo
    return [round(v * M / Fraction(2) ** S) for v in xs], M, S


def pin_quantize_rows(o):
    """Per-row int8 quantization: hand-worked rows, exact-rational brute force
    on bf16 / fp16 / fp32 rows (subnormal and huge values included), and the
    invariants of the reading (the largest element maps to +-127, the
    multiplier stays in [16256, 32512], scaling a row by 2^j only moves S,
    rows are independent, the error is at most half a step)."""
    q, M, S = o.quantize_rows(np.array([[1.0, -0.5, 0.25], [0.0, 0.0, 0.0], [3.0, -1.0, 0.0],
                                        [-2.0, 1.0, 0.015625],
                                        [1.984375, 0.0078125, -0.0390625],
                                        [1.984375, 0.0234375, 0.0]]))
    # amax = 127/64 gives M = 2^14: q = 64 x, and 0.5 / -2.5 / 1.5 are exact ties
    assert q.tolist() == [[127, -64, 32], [0, 0, 0], [127, -42, 0], [-127, 64, 1],
                          [127, 0, -2], [127, 2, 0]]
    assert M.tolist() == [32512, 0, 21674, 32512, 16384, 16384]
    assert S.tolist() == [8, 0, 9, 9, 8, 8]
    rng = np.random.default_rng(41)
    rows = []
    for fmt, bits in (("bf16", rng.integers(0, 1 << 16, size=(6, 9)) & 0xBF7F),
                      ("fp16", rng.integers(0, 1 << 16, size=(6, 9)) & 0xFBFF),
                      ("fp32", rng.integers(0, 1 << 32, size=(6, 9), dtype=np.uint64)
                       .astype(np.uint32) & np.uint32(0xFF7FFFFF))):
        x = o.decode(bits.astype(np.uint16) if fmt != "fp32" else bits, fmt)
        x = x * np.exp2(rng.integers(-4, 4, size=(6, 1)))
        rows.append(x)
    rows.append(np.array([[2.0 ** -149, -2.0 ** -148, 0.0, 2.0 ** -140] + [0.0] * 5]))
    rows.append(np.array([[3.0e38, -1.0e38, 1.0, 2.0 ** 100, -3.4e38, 0.0, 5.0, -7.0, 1e-30]]))
    X = np.concatenate(rows)
    X = X[np.all(np.isfinite(X), axis=1)]
    q, M, S = o.quantize_rows(X)
    for n in range(X.shape[0]):
        qe, Me, Se = _quantize_exact(X[n])
        assert q[n].tolist() == qe and int(M[n]) == Me and int(S[n]) == Se, n
        if Me:
            assert 16256 <= Me <= 32512
            assert int(np.max(np.abs(q[n].astype(int)))) == 127
            step = Fraction(2) ** Se / Me
            for xv, qv in zip(X[n], qe):
                assert abs(Fraction(float(xv)) - qv * step) <= step / 2
    q2, M2, S2 = o.quantize_rows(X * 8.0)
    assert (q2 == q).all() and (M2 == M).all() and (S2[M != 0] == S[M != 0] + 3).all()
    for n in range(X.shape[0]):
        qn, Mn, Sn = o.quantize_rows(X[n:n + 1])
        assert (qn[0] == q[n]).all() and Mn[0] == M[n] and Sn[0] == S[n]


ALL_PINS = [pin_tiny_golden, pin_bruteforce_float, pin_logsumexp_mpmath,
            pin_closed_forms, pin_page_examples, pin_int_head, pin_invariants,
            pin_gap_from_top2, pin_verify_accept, pin_round_to_format,
            pin_gated_greedy, pin_philox_kat, pin_gumbel_layout,
            pin_gumbel_max_distribution, pin_sample_invariants, pin_quantize_rows]


def failing_pins(o):
    """Names of the pins that fail (AssertionError or any exception)."""
    bad = []
    for p in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                p(o)
        except Exception:   # noqa: BLE001 - a mutated oracle may fail any way
            bad.append(p.__name__)
    return bad
