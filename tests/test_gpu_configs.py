"""The five workloads at their full sizes, in the launch configuration the
benchmark times, against the oracle element by element on every row of the
PR1, speculative-verify and integer workloads and on 1,280 rows of the 8,192
trainer rows (the float64 oracle takes seconds per thousand rows there), and
by properties that hold at any size (self-consistency of the decision with
the GPU's own logits, bit-identity across batch sizes). Near-tie exceptions
are collected and printed at the end of the session."""
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
    # oracle on every row, 64 rows at a time (float64 logits and error base)
    for r0 in range(0, 256, 64):
        rows = np.arange(r0, r0 + 64)
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
    # the oracle on the first sequence's 1024 rows and on 32 rows of each of
    # the others (sequence starts and ends included), 128 rows at a time
    rows_all = np.concatenate([np.arange(1024)] +
                              [s * 1024 + np.r_[0:16, 1008:1024] for s in range(1, 8)])
    for k in range(0, rows_all.size, 128):
        rows = rows_all[k:k + 128]
        z_ref, A = oracle_float_rows(c["W"], c["h"][rows], fmt)
        lse = oracle.logsumexp(z_ref)
        lp_ref = oracle.logprob(z_ref, c["targets"][rows])
        err = np.abs(lp_all[rows].astype(np.float64) - lp_ref)
        assert (err <= logprob_tol(A, lse, c["targets"][rows])).all(), (k, err.max())
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
    # every row, exactly (the oracle's integer logits through its exact float64
    # product), 64 rows at a time
    for r0 in range(0, B, 64):
        rows = np.arange(r0, min(B, r0 + 64))
        z_ref = oracle.logits_int_f64(c["W"], c["h"][rows])
        assert (z[rows].astype(np.int64) == z_ref).all(), r0
        tr, gr, _, _ = oracle.greedy_int(z_ref)
        assert (t[rows] == tr).all() and (g[rows].astype(np.int64) == gr).all(), r0
    rng = np.random.default_rng(B)
    for _ in range(4):   # big-integer spot checks
        r, v = int(rng.integers(0, B)), int(rng.integers(0, c["V"]))
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


def test_int8_wide_call_after_reserve_allocates_nothing(torch_cuda):
    """A head reserved for 512 rows makes the wide path's fp16 copies at the
    reserve; the B = 512 calls then leave the free device memory unchanged and
    give the exact logits."""
    from invariant_output_head_gb300 import Head, binding as bd
    torch = torch_cuda
    c = synth.small_int8(123, 9000, 1024, 512)
    head = Head(dev(c["W"], "int8"), "int8")
    bd.detlm_head_reserve(head.handle, 512)
    h = dev(c["h"], "int8")
    out = (torch.empty(512, dtype=torch.int32, device="cuda"),
           torch.empty(512, dtype=torch.int32, device="cuda"),
           torch.empty((512, 9000), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        head.greedy(h, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert head.check() == 0
    z_ref = oracle.logits_int(c["W"], c["h"][:64])
    assert (host(out[2])[:64].astype(np.int64) == z_ref).all()
    assert (host(out[0])[:64] == oracle.greedy_int(z_ref)[0]).all()
    head.close()
