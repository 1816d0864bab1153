"""The five workloads at their full sizes, in the launch configuration the
benchmark times, against the oracle on every row it can afford (all rows for
the d=2048 heads, sampled rows for the large ones) and by properties that
hold at any size (self-consistency of the decision with the GPU's own
logits, bit-identity across batch sizes)."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import (check_float_greedy, dev, host, logprob_tol,
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


def test_pr1_greedy_b1(torch_cuda):
    """16 independent hidden rows, each a B=1 call (d=2048, V=32000)."""
    from invariant_output_head_gb300 import Head
    c = synth.pr1()
    head = Head(dev(c["W"], "bf16"), "bf16")
    h = dev(c["h"], "bf16")
    toks, gaps, zs = [], [], []
    for r in range(16):
        t, g, z = head.greedy(h[r:r + 1], with_logits=True)
        toks.append(host(t))
        gaps.append(host(g))
        zs.append(host(z))
    assert head.check() == 0
    z_ref, A = oracle_float_rows(c["W"], c["h"], "bf16")
    check_float_greedy(z_ref, A, np.concatenate(toks), np.concatenate(gaps),
                       np.concatenate(zs), label="PR1")


def test_spec_verify_b256(torch_cuda):
    """16 requests x 16 draft positions = 256 rows (d=3584, V=152064)."""
    from invariant_output_head_gb300 import Head
    c = synth.spec_verify()
    head = Head(dev(c["W"], "bf16"), "bf16")
    h = dev(c["h"], "bf16")
    t, g, z = head.greedy(h, with_logits=True)
    t, g, z = host(t), host(g), host(z)
    assert head.check() == 0
    # decision vs the GPU's own logits, every row (bitwise)
    assert (t == np.argmax(z, axis=1)).all()
    srt = np.partition(z, -2, axis=1)
    assert (g.view(np.uint32) == oracle.gap_from_top2_f32(
        srt[:, -1], srt[:, -2]).view(np.uint32)).all()
    # oracle on sampled rows
    rows = np.array([0, 1, 17, 100, 128, 200, 254, 255])
    z_ref, A = oracle_float_rows(c["W"], c["h"][rows], "bf16")
    check_float_greedy(z_ref, A, t[rows], g[rows], z[rows], label="spec-verify")
    # the first request's 16 rows alone give the same bits
    t16, g16, z16 = head.greedy(h[:16], with_logits=True)
    assert (host(t16) == t[:16]).all()
    assert (host(z16).view(np.uint32) == z[:16].view(np.uint32)).all()


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
def test_trainer_logprob_8192(torch_cuda, fmt):
    """8 sequences x 1024 tokens (d=1536, V=151936): one call of 8192 rows
    versus 8 calls of 1024 rows, bitwise; oracle on sampled rows."""
    from invariant_output_head_gb300 import Head
    c = synth.logprob(fmt=fmt)
    head = Head(dev(c["W"], fmt), fmt)
    h = dev(c["h"], fmt)
    t = dev(c["targets"], "int32")
    lp_all = host(head.logprob(h, t))
    lp_seq = np.concatenate([host(head.logprob(h[s * 1024:(s + 1) * 1024],
                                               t[s * 1024:(s + 1) * 1024]))
                             for s in range(8)])
    assert head.check() == 0
    assert (lp_all.view(np.uint32) == lp_seq.view(np.uint32)).all()
    for B in (1, 2, 3, 8, 17, 64, 256):
        sub = np.concatenate([host(head.logprob(h[r0:r0 + B], t[r0:r0 + B]))
                              for r0 in range(0, 256, B)])[:256]
        assert (sub.view(np.uint32) == lp_all[:256].view(np.uint32)).all(), B
    rows = np.array([0, 5, 1023, 1024, 4097, 8191])
    z_ref, A = oracle_float_rows(c["W"], c["h"][rows], fmt)
    lse = oracle.logsumexp(z_ref)
    lp_ref = oracle.logprob(z_ref, c["targets"][rows])
    err = np.abs(lp_all[rows].astype(np.float64) - lp_ref)
    assert (err <= logprob_tol(A, lse, c["targets"][rows])).all(), err
    assert (lp_all <= 0).all() and np.isfinite(lp_all).all()


@pytest.mark.parametrize("B", [1, 32, 512])
def test_int8_head_exact(torch_cuda, B):
    """int8 d=4096, V=128256: exact int32 logits and tokens on sampled rows,
    planted duplicate W rows (exact ties) resolved to the lower id."""
    from invariant_output_head_gb300 import Head
    c = synth.int8_head(B=512)
    head = Head(dev(c["W"], "int8"), "int8")
    h = dev(c["h"][:B], "int8")
    t, g, z = head.greedy(h, with_logits=True)
    t, g, z = host(t), host(g), host(z)
    assert head.check() == 0
    rows = np.unique(np.array([0, 1, 2, B // 2, B - 1]) % B)
    z_ref = oracle.logits_int(c["W"], c["h"][rows])
    assert (z[rows].astype(np.int64) == z_ref).all()
    tr, gr, _, _ = oracle.greedy_int(z_ref)
    assert (t[rows] == tr).all() and (g[rows].astype(np.int64) == gr).all()
    rng = np.random.default_rng(B)
    for _ in range(4):   # big-integer spot checks
        r, v = int(rng.choice(rows)), int(rng.integers(0, c["V"]))
        assert int(z[r, v]) == oracle.bigint_dot(c["W"][v], c["h"][r])
    # every row: decision against the GPU's own exact logits
    assert (t == np.argmax(z, axis=1)).all()
    for k, (a, b) in enumerate(c["dup_pairs"][:min(B, len(c["dup_pairs"]))]):
        assert int(t[k]) == min(a, b) and int(g[k]) == 0


def test_spec_verify_accept_b256(torch_cuda):
    """The speculative-verify block through the verify call: 16 requests x 16
    positions. Requests 0 and 9 get drafts planted from the oracle's tokens
    and must match the oracle's accepted lengths; the rest get drafts planted
    from a seeded random sequence and must follow the acceptance rule on the
    call's own tokens. Tokens and gaps are bitwise those of the plain call."""
    from invariant_output_head_gb300 import Head
    torch = torch_cuda
    c = synth.spec_verify()
    R, P = 16, 16
    head = Head(dev(c["W"], "bf16"), "bf16")
    h = dev(c["h"], "bf16")
    checked = [0, 9]
    rows = np.concatenate([np.arange(r * P, (r + 1) * P) for r in checked])
    z_ref, A = oracle_float_rows(c["W"], c["h"][rows], "bf16")
    t_ref = np.argmax(z_ref, axis=1)
    seq = np.random.default_rng(77).integers(0, c["V"], size=(R, P))
    for k, r in enumerate(checked):
        seq[r] = t_ref[k * P:(k + 1) * P]
    drafts, _ = synth.plant_drafts(seq, c["V"], seed=78)
    t_plain, g_plain, _ = head.greedy(h)
    tok, gap, z, acc = head.verify(h, torch.from_numpy(drafts).cuda(), with_logits=True)
    tok, acc = host(tok), host(acc)
    assert head.check() == 0
    assert (tok == host(t_plain)).all()
    assert (host(gap).view(np.uint32) == host(g_plain).view(np.uint32)).all()
    check_float_greedy(z_ref, A, tok[rows], host(gap)[rows], host(z)[rows],
                       label="spec-verify accept")
    acc_ref = oracle.verify_accept(t_ref.reshape(len(checked), P), drafts[checked])
    assert (acc[checked] == acc_ref).all()
    assert (acc == oracle.verify_accept(tok.reshape(R, P), drafts)).all()
