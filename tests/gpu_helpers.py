"""Helpers for the GPU tests: move generator output to the device, and the
parity checks against the oracle (tolerances stated here, once)."""
from __future__ import annotations

import numpy as np

import oracle

# fp32 logits of the float heads: |z_gpu - z_ref| <= 1e-6 * sum_k |w_k h_k|
LOGIT_RTOL = 1e-6

# Every parity check's rows and its listed exceptions (decisions that differ
# from the oracle's inside the tolerance), printed at the end of the session
# by the terminal-summary hook in conftest.py: listed, not hidden.
PARITY_REPORT = []


def dev(arr: np.ndarray, fmt: str):
    import torch
    a = np.ascontiguousarray(arr)
    if fmt == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    if fmt == "fp16":
        return torch.from_numpy(a.view(np.int16)).view(torch.float16).cuda()
    if fmt == "int8":
        return torch.from_numpy(a.astype(np.int8, copy=False)).cuda()
    if fmt == "int32":
        return torch.from_numpy(a.astype(np.int32, copy=False)).cuda()
    raise ValueError(fmt)


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def oracle_float_rows(W_raw, h_raw, fmt, v_chunk=16384):
    """Oracle logits and error base for the given rows, W taken in V-chunks
    (each logit is still one plain dot product)."""
    h = oracle.decode(h_raw, fmt)
    zs, As = [], []
    for v0 in range(0, W_raw.shape[0], v_chunk):
        z, A = oracle.logits_float(oracle.decode(W_raw[v0:v0 + v_chunk], fmt), h)
        zs.append(z)
        As.append(A)
    return np.concatenate(zs, axis=1), np.concatenate(As, axis=1)


def check_float_greedy(z_ref, A, tok_g, gap_g, z_g=None, label=""):
    """Parity of one float greedy call. Returns the listed near-tie exceptions.

    * logits: |z_g - z_ref| <= 1e-6 * A, element by element;
    * token: equal to the oracle's, except in rows whose oracle top-2 lie
      within the tolerance of each other; there the GPU token must be one of
      the tied candidates, and the row is listed;
    * self-consistency (bitwise): the token is the lowest-index argmax of the
      GPU's own logits, and the gap is the oracle's gap function of the GPU's
      own top-2 fp32 values;
    * gap against the oracle: within 2 * max_v e[n, v] in logit units.
    """
    e = LOGIT_RTOL * A
    B = z_ref.shape[0]
    t_ref, gap_ref, m_ref, s_ref = oracle.greedy(z_ref)
    exceptions = []
    if z_g is not None:
        z_g = np.asarray(z_g)
        err = np.abs(z_g.astype(np.float64) - z_ref)
        bad = err > e
        assert not bad.any(), (label, "logits outside 1e-6*sum|wh|",
                               np.argwhere(bad)[:5], err[bad][:5], e[bad][:5])
        # self-consistency against the GPU's own logits
        t_self = np.argmax(z_g, axis=1)
        assert (tok_g == t_self).all(), (label, "token != argmax of own logits")
        if z_g.shape[1] >= 2:
            srt = np.sort(z_g, axis=1)
            g_self = oracle.gap_from_top2_f32(srt[:, -1], srt[:, -2])
            assert (gap_g.view(np.uint32) == g_self.view(np.uint32)).all(), \
                (label, "gap != gap of own top-2", gap_g[:4], g_self[:4])
    for n in range(B):
        t = int(t_ref[n])
        if int(tok_g[n]) == t:
            continue
        tg = int(tok_g[n])
        near = z_ref[n, t] - z_ref[n, tg] <= e[n, t] + e[n, tg]
        assert near, (label, "token differs outside the tolerance", n, t, tg,
                      z_ref[n, t] - z_ref[n, tg], e[n, t] + e[n, tg])
        exceptions.append({"row": n, "oracle": t, "gpu": tg,
                           "gap_ulp": float(gap_ref[n])})
    PARITY_REPORT.append((label, B, exceptions))
    if z_ref.shape[1] >= 2:
        ulp = oracle.ulp_bf16(m_ref)
        emax = e.max(axis=1)
        d_gap = np.abs(gap_g.astype(np.float64) * oracle.ulp_bf16(
            m_ref if z_g is None else np.max(z_g, axis=1)) - gap_ref * ulp)
        assert (d_gap <= 2 * emax + 1e-30).all(), (label, "gap off", d_gap.max())
    return exceptions


def logprob_tol(A, lse_ref, targets):
    """Tolerance of the fp32 log-probability (derived in the design notes):
    the logits' own bound at the target and at the worst entry (log-sum-exp is
    1-Lipschitz in the max norm), plus the GPU's own fp32 evaluation of the
    log-sum-exp: one rounding of lse (<= 1e-6 relative) and at most ~20 merge
    levels of exp/fma rounding, each <= 4e-7 relative in the sum (8e-6 in log)."""
    e = LOGIT_RTOL * A
    B = A.shape[0]
    et = e[np.arange(B), targets]
    return et + e.max(axis=1) + 1e-6 * (1.0 + np.abs(lse_ref)) + 8e-6


def sample_tol(z_ref, A, T, G):
    """Bound on |score_gpu - score_ref| of the sampling call, per entry:
    the logit's own bound over T, the rounding of z / T, the fp32 Gumbel
    transform (two logf calls, each within 1 ulp by CUDA's documented bound;
    U is exact: 2^-23 from the inner log, 2^-23 |G| from the outer, doubled
    for margin) and the rounding of the final add."""
    zt = np.abs(z_ref) / T
    return (LOGIT_RTOL * A / T + 2.0 ** -24 * zt + 2.0 ** -22 * (1.0 + np.abs(G))
            + 2.0 ** -24 * (zt + np.abs(G)))


def check_sample(z_ref, A, T, seeds, positions, tok_g, gap_g, label=""):
    """Sampled tokens against the oracle's draws; rows where the oracle's two
    best scores lie within the sum of their bounds are listed, and there the
    GPU token must be one of those candidates."""
    ref = oracle.sample(z_ref, T, seeds, positions)
    G = oracle.gumbel_rows(seeds, positions, z_ref.shape[1])
    e = sample_tol(z_ref, A, T, G)
    sc = ref["score"]
    listed = []
    for n in range(z_ref.shape[0]):
        t, tg = int(ref["token"][n]), int(tok_g[n])
        if tg != t:
            assert sc[n, t] - sc[n, tg] <= e[n, t] + e[n, tg], (
                label, "sampled token differs outside the bound", n, t, tg,
                sc[n, t] - sc[n, tg], e[n, t] + e[n, tg])
            listed.append({"row": n, "oracle": t, "gpu": tg,
                           "gap_score": float(sc[n, t] - sc[n, tg])})
        if z_ref.shape[1] >= 2 and gap_g is not None and tg == t:
            srt = np.argsort(-sc[n], kind="stable")
            bound = e[n, srt[0]] + 2 * e[n, srt[1:3]].max() + 2.0 ** -24 * abs(float(gap_g[n]))
            assert abs(float(gap_g[n]) - (ref["m"][n] - ref["s"][n])) <= bound, (
                label, "score gap", n, gap_g[n], ref["m"][n] - ref["s"][n], bound)
    PARITY_REPORT.append((label, z_ref.shape[0], listed))
    return listed
