"""The margin-gated greedy call ("Greedy Decoding Has a Precision Clause",
section on correcting the vulnerable token decisions) against the oracle.

Checks, per call:
* bitwise self-consistency: the oracle's gate applied to the GPU's own fp32
  logits gives the GPU's token, base token and margin exactly (the 16-bit
  rounding and the gate are decided in the same precision on both sides);
* against the exact logits: the same results, except in rows where a
  16-bit rounding among the top candidates falls on different sides of a
  rounding boundary for the GPU's fp32 value and the exact value (both
  within the 1e-6 * sum|w h| logit tolerance); such rows are listed;
* with tau > 0 the gated token is the plain greedy token, bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import (LOGIT_RTOL, check_float_greedy, dev, host,
                               oracle_float_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import invariant_output_head_gb300 as ioh
    ioh.load_library()
    return torch


def check_gated(z_ref, A, z_g, tok, base, margin, tau, fmt, label=""):
    """Returns the listed rows: a 16-bit rounding among the top candidates
    that straddles a boundary, or a fired row whose fp32 winner is a tie
    within the logit tolerance (the plain greedy call's exception)."""
    own = oracle.gated_greedy(z_g.astype(np.float64), tau, fmt)
    assert (tok == own["token"]).all(), (label, "token vs own logits")
    assert (base == own["base"]).all(), (label, "base token vs own logits")
    assert (margin.view(np.uint32) == own["margin"].view(np.uint32)).all(), (label, "margin")
    ref = oracle.gated_greedy(z_ref, tau, fmt)
    r_g = oracle.round_to_format(z_g.astype(np.float64), fmt)
    r_ref = oracle.round_to_format(z_ref, fmt)
    e = LOGIT_RTOL * A
    listed = []
    for n in range(z_ref.shape[0]):
        same_gate = (base[n] == ref["base"][n]
                     and margin[n].view(np.uint32) == ref["margin"][n].view(np.uint32))
        if same_gate and tok[n] == ref["token"][n]:
            continue
        if same_gate:
            # the gate agrees and fired; the fp32 winners differ only on a
            # tie within the tolerance
            t, tg = int(ref["token"][n]), int(tok[n])
            assert bool(ref["fired"][n]), (label, "unfired row with a different token", n)
            assert z_ref[n, t] - z_ref[n, tg] <= e[n, t] + e[n, tg], (label, "fp32 winner", n)
            listed.append({"row": n, "fp32_tie": (t, tg)})
            continue
        s_lo = min(np.sort(r_g[n])[-2] if z_ref.shape[1] > 1 else -np.inf,
                   np.sort(r_ref[n])[-2] if z_ref.shape[1] > 1 else -np.inf)
        top = (r_g[n] >= s_lo) | (r_ref[n] >= s_lo)
        straddle = np.nonzero(top & (r_g[n] != r_ref[n]))[0]
        assert straddle.size > 0, (label, "gate differs without a rounding straddle", n,
                                   tok[n], ref["token"][n], base[n], ref["base"][n],
                                   margin[n], ref["margin"][n])
        listed.append({"row": n, "straddle": straddle.tolist()})
    return listed


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
@pytest.mark.parametrize("V,d", [(1000, 520), (129, 8), (16, 64)])
@pytest.mark.parametrize("B", [1, 17, 300])
def test_gated_parity(torch_cuda, fmt, V, d, B):
    from invariant_output_head_gb300 import Head
    case = synth.small_float(300 + V + d + B, V, d, B, fmt=fmt, n_ties=min(1, B),
                             n_near=min(6, max(B - 1, 0)))
    head = Head(dev(case["W"], fmt), fmt)
    h = dev(case["h"], fmt)
    tau = 0.001
    tok, gap, z, base, margin = head.greedy_gated(h, tau, with_logits=True)
    t_plain, g_plain, _ = head.greedy(h)
    tok, gap, z, base, margin = host(tok), host(gap), host(z), host(base), host(margin)
    assert head.check() == 0
    z_ref, A = oracle_float_rows(case["W"], case["h"], fmt)
    check_float_greedy(z_ref, A, tok, gap, z, label=f"gated {fmt}")
    listed = check_gated(z_ref, A, z, tok, base, margin, tau, fmt, label=fmt)
    assert sum("straddle" in x for x in listed) <= max(1, B // 50), listed
    assert (tok == host(t_plain)).all()
    assert (gap.view(np.uint32) == host(g_plain).view(np.uint32)).all()


@pytest.mark.parametrize("tau", [0.0, -1.0, 0.05, float("inf")])
def test_gated_thresholds(torch_cuda, tau):
    """tau <= 0 never fires (the ordinary head's tokens); tau = inf always
    fires (the fp32 tokens)."""
    from invariant_output_head_gb300 import Head
    case = synth.small_float(41, 700, 264, 64, n_ties=2, n_near=20)
    head = Head(dev(case["W"], "bf16"), "bf16")
    tok, _, z, base, margin = head.greedy_gated(dev(case["h"], "bf16"), tau, with_logits=True)
    tok, z, base, margin = host(tok), host(z), host(base), host(margin)
    assert head.check() == 0
    z_ref, A = oracle_float_rows(case["W"], case["h"], "bf16")
    check_gated(z_ref, A, z, tok, base, margin, tau, "bf16", label=f"tau={tau}")
    if tau <= 0:
        assert (tok == base).all()
    if tau == float("inf"):
        assert (tok == np.argmax(z, axis=1)).all()
    # the planted near ties give rounded ties that fire at tau > 0
    assert (margin[2:22] == 0).sum() >= 10


def test_gated_sweep_full_size(torch_cuda):
    """The tie sweep at full size (d=2048, V=32000, 64 rows with 8 planted
    near-tie pairs): every planted row ties in bf16, so the gate fires and
    the fp32 recompute decides; at least one planted row's ordinary bf16
    token differs from the fp32 token."""
    from invariant_output_head_gb300 import Head
    c = synth.sweep()
    head = Head(dev(c["W"], "bf16"), "bf16")
    h = dev(c["h"], "bf16")
    tok, gap, z, base, margin = head.greedy_gated(h, 0.001, with_logits=True)
    tok, gap, z, base, margin = host(tok), host(gap), host(z), host(base), host(margin)
    assert head.check() == 0
    z_ref, A = oracle_float_rows(c["W"], c["h"], "bf16")
    check_float_greedy(z_ref, A, tok, gap, z, label="gated sweep")
    listed = check_gated(z_ref, A, z, tok, base, margin, 0.001, "bf16", label="sweep")
    assert sum("straddle" in x for x in listed) <= 2, listed
    assert (margin[:8] < 0.001).all()
    assert (base[:8] != tok[:8]).any()
    for B in (1, 3, 17):
        parts = [head.greedy_gated(h[r0:r0 + B], 0.001) for r0 in range(0, 64, B)]
        tb = np.concatenate([host(p[0]) for p in parts])[:64]
        bb = np.concatenate([host(p[3]) for p in parts])[:64]
        mb = np.concatenate([host(p[4]) for p in parts])[:64]
        assert (tb == tok).all() and (bb == base).all(), B
        assert (mb.view(np.uint32) == margin.view(np.uint32)).all(), B


def test_gated_rejects(torch_cuda):
    import invariant_output_head_gb300 as ioh
    from invariant_output_head_gb300 import Head, DetlmError
    c8 = synth.small_int8(5, 200, 64, 4)
    head8 = Head(dev(c8["W"], "int8"), "int8")
    with pytest.raises(DetlmError) as ei:
        head8.greedy_gated(dev(c8["h"], "int8"), 0.001)
    assert ei.value.status == ioh.DETLM_EUNSUPPORTED
    cf = synth.small_float(6, 200, 64, 4)
    head = Head(dev(cf["W"], "bf16"), "bf16")
    with pytest.raises(DetlmError) as ei:
        head.greedy_gated(dev(cf["h"], "bf16"), float("nan"))
    assert ei.value.status == ioh.DETLM_EINVAL
