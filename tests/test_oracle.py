"""The CPU oracle against its pins, and planted mistakes against the pins.

No GPU: these run in the CPU suite.
"""
import os
import types

import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "head.py")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle)


# Each mutant is a plausible mistake in the oracle: (snippet, replacement).
MUTANTS = {
    "tie_to_highest_id": ("token = np.argmax(z, axis=1).astype(np.int64)\n    m = z[np.arange(z.shape[0]), token]\n    if z.shape[1] >= 2:\n        s = np.sort(z, axis=1)[:, -2]\n    else:\n        s = np.full(z.shape[0], -np.inf",
                          "token = (z.shape[1] - 1 - np.argmax(z[:, ::-1], axis=1)).astype(np.int64)\n    m = z[np.arange(z.shape[0]), token]\n    if z.shape[1] >= 2:\n        s = np.sort(z, axis=1)[:, -2]\n    else:\n        s = np.full(z.shape[0], -np.inf"),
    "runner_up_distinct": ("        s = np.sort(z, axis=1)[:, -2]\n    else:\n        s = np.full(z.shape[0], -np.inf",
                           "        s = np.array([np.unique(r)[-2] if len(np.unique(r)) > 1 else r[0] for r in z])\n    else:\n        s = np.full(z.shape[0], -np.inf"),
    "ulp_exponent_off_by_one": ("return np.ldexp(1.0, E - 7)", "return np.ldexp(1.0, E - 8)"),
    "ulp_no_clamp": ("E = np.where(m == 0, -126, np.maximum(e - 1, -126))",
                     "E = np.where(m == 0, -126, e - 1)"),
    "ulp_floor_wrong": ("np.maximum(e - 1, -126)", "np.maximum(e, -126)"),
    "logits_transposed": ("    z = h @ W.T\n", "    z = (W @ h.T)\n"),
    "logits_dropped_term": ("    z = h @ W.T\n", "    z = h[:, :-1] @ W[:, :-1].T\n"),
    "logits_sign": ("    z = h @ W.T\n", "    z = -(h @ W.T)\n"),
    "abs_bound_signed": ("A = np.abs(h) @ np.abs(W).T", "A = np.abs(h @ W.T)"),
    "lse_no_shift": ("return M + np.log(np.sum(np.exp(z - M[:, None]), axis=1))",
                     "return np.log(np.sum(np.exp(z), axis=1))"),
    "lse_drops_max": ("return M + np.log(np.sum(np.exp(z - M[:, None]), axis=1))",
                      "return np.log(np.sum(np.exp(z - M[:, None]), axis=1))"),
    "logp_sign": ("return zt - logsumexp(z)", "return logsumexp(z) - zt"),
    "logp_wrong_index": ("zt = np.where(ok, z[np.arange(B), np.where(ok, t, 0)], np.nan)",
                         "zt = np.where(ok, z[np.arange(B), np.where(ok, (t + 1) % V, 0)], np.nan)"),
    "bf16_decode_shift": ("astype(np.uint32) << np.uint32(16)", "astype(np.uint32) << np.uint32(15)"),
    "fp16_as_bf16": ("return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)",
                     "return decode_bf16(bits)"),
    "int_narrow_accumulator": ("return np.asarray(h, dtype=np.int64) @ np.asarray(W, dtype=np.int64).T",
                               "return (np.asarray(h, dtype=np.int64) @ np.asarray(W, dtype=np.int64).T).astype(np.int16).astype(np.int64)"),
    "int_gap_reversed": ("        gap = m - s\n", "        gap = s - m\n"),
    "int_f64_narrowed": ("    return z.astype(np.int64)\n", "    return z.astype(np.float32).astype(np.int64)\n"),
    "int_f64_transposed": ("    z = np.asarray(h, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T\n",
                           "    z = (np.asarray(W, dtype=np.float64) @ np.asarray(h, dtype=np.float64).T).T[:, ::-1]\n"),
    "verify_accept_counts_all_matches": ("        while a < P and drafts[r, a] == tokens[r, a]:\n            a += 1",
                                         "        a = int((drafts[r] == tokens[r]).sum())"),
    "verify_accept_off_by_one": ("        out[r] = a\n", "        out[r] = min(a + 1, P)\n"),
    "round_toward_zero": ("        r = np.rint(ax / q) * q\n", "        r = np.trunc(ax / q) * q\n"),
    "round_ties_away": ("        r = np.rint(ax / q) * q\n", "        r = np.floor(ax / q + 0.5) * q\n"),
    "round_no_overflow": ("    r = np.where(r > vmax, np.inf, r)\n", ""),
    "round_no_subnormal_clamp": ("    E = np.maximum(e - 1, emin)\n", "    E = e - 1\n"),
    "gate_base_highest_on_tie": ("    base = np.argmax(z16, axis=1).astype(np.int64)\n",
                                 "    base = (z16.shape[1] - 1 - np.argmax(z16[:, ::-1], axis=1)).astype(np.int64)\n"),
    "gate_margin_unrounded": ("        margin = (M16 - S16).astype(np.float32)\n",
                              "        margin = (np.sort(z, axis=1)[:, -1] - (np.sort(z, axis=1)[:, -2] if z.shape[1] > 1 else -np.inf)).astype(np.float32)\n"),
    "gate_fires_at_equality": ("    fired = margin < np.float32(tau)\n", "    fired = margin <= np.float32(tau)\n"),
    "gate_token_always_base": ("    token = np.where(fired, full, base)\n", "    token = base\n"),
    "gate_token_always_full": ("    token = np.where(fired, full, base)\n", "    token = full\n"),
    "philox_no_key_bump": ("        k0 = (k0 + PHILOX_W[0]) & _M32\n", ""),
    "philox_multipliers_swapped": ("        p0 = PHILOX_M[0] * c0\n        p1 = PHILOX_M[1] * c2\n",
                                   "        p0 = PHILOX_M[1] * c0\n        p1 = PHILOX_M[0] * c2\n"),
    "philox_nine_rounds": ("    for _ in range(10):\n        p0 = PHILOX_M[0] * c0", "    for _ in range(9):\n        p0 = PHILOX_M[0] * c0"),
    "uniform_can_be_zero": ("((x >> np.uint64(9)) * np.uint64(2) + np.uint64(1)).astype(np.float64) * 2.0 ** -24",
                            "(x >> np.uint64(8)).astype(np.float64) * 2.0 ** -24"),
    "gumbel_layout_t_first": ("    counter = np.stack([v >> np.uint64(2), t_lo, t_hi, np.zeros_like(v)], axis=-1)",
                              "    counter = np.stack([t_lo, v >> np.uint64(2), t_hi, np.zeros_like(v)], axis=-1)"),
    "gumbel_word_zero": ("    x = np.take_along_axis(words, (v & np.uint64(3)).astype(np.int64)[..., None], axis=-1)[..., 0]",
                         "    x = words[..., 0]"),
    "gumbel_sign": ("    return -np.log(-np.log(uniform_from_word(x)))", "    return np.log(-np.log(uniform_from_word(x)))"),
    "sample_temperature_multiplies": ("    score = z / float(temperature) + gumbel_rows",
                                      "    score = z * float(temperature) + gumbel_rows"),
    "sample_seed_ignored": ("gumbel_rows(seeds, positions, z.shape[1])",
                            "gumbel_rows([0] * z.shape[0], positions, z.shape[1])"),
    "sample_position_ignored": ("gumbel_rows(seeds, positions, z.shape[1])",
                                "gumbel_rows(seeds, [0] * z.shape[0], z.shape[1])"),
    "sample_keys_through_float": ("    seeds = _u64_list(seeds)\n", "    seeds = [int(x) for x in np.asarray(seeds).reshape(-1)]\n"),
    "quantize_ties_away": ("        q[n] = np.rint(x[n] * float(m) * 2.0 ** (-s)).astype(np.int8)",
                           "        q[n] = (np.sign(x[n]) * np.floor(np.abs(x[n]) * float(m) * 2.0 ** (-s) + 0.5)).astype(np.int8)"),
    "quantize_multiplier_ceil": ("        m = (Fraction(127) * Fraction(2) ** s) // Fraction(amax)",
                                 "        m = -((-Fraction(127) * Fraction(2) ** s) // Fraction(amax))"),
    "quantize_shift_off_by_one": ("        s = E + 8\n", "        s = E + 7\n"),
    "quantize_signed_max": ("        amax = float(np.max(np.abs(x[n]))) if d > 0 else 0.0",
                            "        amax = float(np.max(x[n])) if d > 0 else 0.0"),
    "quantize_batch_scale": ("        amax = float(np.max(np.abs(x[n]))) if d > 0 else 0.0",
                             "        amax = float(np.max(np.abs(x))) if d > 0 else 0.0"),
    "gap_f32_rounded_difference": ("    with np.errstate(invalid=\"ignore\"):\n        return ((m - s) / ulp_bf16(m)).astype(np.float32)",
                                   "    with np.errstate(invalid=\"ignore\"):\n        return ((m - s) / ulp_bf16(s)).astype(np.float32)"),
}


def _mutant(name):
    src = open(ORACLE_SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutant {name}: snippet not found in the oracle"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def test_unmutated_copy_passes():
    src = open(ORACLE_SRC).read()
    mod = types.ModuleType("oracle_copy")
    exec(compile(src, "<copy>", "exec"), mod.__dict__)
    assert pins.failing_pins(mod) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    assert pins.failing_pins(_mutant(name)), f"no pin catches mutant {name}"


def test_synth_is_deterministic_and_formats():
    import synth
    a = synth.small_float(1, 50, 24, 3)
    b = synth.small_float(1, 50, 24, 3)
    assert (a["W"] == b["W"]).all() and (a["h"] == b["h"]).all()
    assert a["W"].dtype == np.uint16 and a["W"].shape == (50, 24)
    x = np.array([1.0, 1.00390625, 1.01171875, -3.0], np.float32)
    # ties to even at the halfway points 1 + 2^-8 and 1 + 3 * 2^-8
    assert synth.bf16_bits_from_f32(x).tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC040]
