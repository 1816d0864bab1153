"""GPU parity against the oracle at sizes the oracle finishes in seconds:
several vocabulary tiles with a ragged tail, several K blocks with a ragged
tail, one and several column tiles, all three dtypes."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import (check_float_greedy, dev, host, logprob_tol,
                               oracle_float_rows)

pytestmark = pytest.mark.gpu

SHAPES = [  # (V, d): tiles of 128 vocabulary rows, K blocks of 128 bytes
    (1000, 520),   # 7 full tiles + 104-row tail; 8 K blocks of bf16 + 8-element tail
    (16, 64),      # one partial tile, one K block
    (129, 8),      # one full tile + 1 row; K shorter than a block
    (1, 32),       # a single vocabulary entry
]


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import invariant_output_head_gb300 as ioh
    ioh.load_library()
    return torch


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
@pytest.mark.parametrize("V,d", SHAPES)
@pytest.mark.parametrize("B", [1, 5, 17, 64, 300])
def test_float_greedy_parity(torch_cuda, fmt, V, d, B):
    from invariant_output_head_gb300 import Head
    case = synth.small_float(100 + V + d + B, V, d, B, fmt=fmt, n_ties=min(2, B))
    Wt = dev(case["W"], fmt)
    head = Head(Wt, fmt)
    tok, gap, z = head.greedy(dev(case["h"], fmt), with_logits=True)
    torch_cuda.cuda.synchronize()
    assert head.check() == 0
    z_ref, A = oracle_float_rows(case["W"], case["h"], fmt)
    check_float_greedy(z_ref, A, host(tok), host(gap), host(z), label=f"{fmt} {V}x{d} B={B}")
    # the same call without the logits store gives the same decision bits
    tok2, gap2, _ = head.greedy(dev(case["h"], fmt), with_logits=False)
    assert (host(tok2) == host(tok)).all()
    assert (host(gap2).view(np.uint32) == host(gap).view(np.uint32)).all()


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
@pytest.mark.parametrize("V,d", SHAPES[:3])
@pytest.mark.parametrize("B", [1, 17, 300])
def test_float_logprob_parity(torch_cuda, fmt, V, d, B):
    from invariant_output_head_gb300 import Head
    case = synth.small_float(200 + V + d + B, V, d, B, fmt=fmt)
    head = Head(dev(case["W"], fmt), fmt)
    t = case["targets"]
    lp = host(head.logprob(dev(case["h"], fmt), dev(t, "int32")))
    assert head.check() == 0
    z_ref, A = oracle_float_rows(case["W"], case["h"], fmt)
    lse = oracle.logsumexp(z_ref)
    lp_ref = oracle.logprob(z_ref, t)
    tol = logprob_tol(A, lse, t)
    err = np.abs(lp.astype(np.float64) - lp_ref)
    assert (err <= tol).all(), (err.max(), tol[np.argmax(err - tol)])
    assert (lp <= 0).all()


@pytest.mark.parametrize("V,d,B", [(300, 200, 600), (1, 32, 5), (257, 64, 257), (512, 72, 256)])
def test_float_logprob_pair_tiling(torch_cuda, V, d, B):
    """The log-prob projection's units are 256 hidden rows x 256 vocabulary
    entries on a CTA pair (each CTA 128 rows and one 128-entry half of the
    W tile): ragged row tiles (a pair whose second CTA has no valid row),
    vocabulary tiles whose second half is partly or wholly past V, K shorter
    than or not a multiple of a 64-element box."""
    from invariant_output_head_gb300 import Head
    case = synth.small_float(900 + V + d + B, V, d, B, fmt="bf16")
    head = Head(dev(case["W"], "bf16"), "bf16")
    t = case["targets"]
    lp = host(head.logprob(dev(case["h"], "bf16"), dev(t, "int32")))
    assert head.check() == 0
    z_ref, A = oracle_float_rows(case["W"], case["h"], "bf16")
    lp_ref = oracle.logprob(z_ref, t)
    tol = logprob_tol(A, oracle.logsumexp(z_ref), t)
    err = np.abs(lp.astype(np.float64) - lp_ref)
    assert (err <= tol).all(), (err.max(), tol[np.argmax(err - tol)])


@pytest.mark.parametrize("sigma_h", [60.0, 1e-3])
def test_float_logprob_extreme_scales(torch_cuda, sigma_h):
    """Logits up to ~125 in magnitude (most exp(z - max) flush to zero; the
    rounding of max * log2(e) is largest here) and below ~2e-3 (every entry
    contributes almost exactly 1)."""
    from invariant_output_head_gb300 import Head
    case = synth.small_float(77, 1000, 520, 300, fmt="bf16", sigma_h=sigma_h)
    head = Head(dev(case["W"], "bf16"), "bf16")
    t = case["targets"]
    lp = host(head.logprob(dev(case["h"], "bf16"), dev(t, "int32")))
    assert head.check() == 0
    z_ref, A = oracle_float_rows(case["W"], case["h"], "bf16")
    lp_ref = oracle.logprob(z_ref, t)
    tol = logprob_tol(A, oracle.logsumexp(z_ref), t)
    err = np.abs(lp.astype(np.float64) - lp_ref)
    assert (err <= tol).all(), (err.max(), tol[np.argmax(err - tol)])
    # the greedy call on the same rows (gap in bf16 ulps at large and tiny m)
    tok, gap, z = head.greedy(dev(case["h"], "bf16"), with_logits=True)
    check_float_greedy(z_ref, A, host(tok), host(gap), host(z), label=f"scale {sigma_h}")


def test_float_logprob_equal_logits(torch_cuda):
    """Every vocabulary row the same: all logits of a row are equal, so
    logp = -log V for every target (ties inside every tile and across
    tiles)."""
    from invariant_output_head_gb300 import Head
    V, d, B = 700, 264, 40
    case = synth.small_float(78, V, d, B, fmt="bf16")
    W = np.repeat(case["W"][:1], V, axis=0)
    head = Head(dev(W, "bf16"), "bf16")
    t = case["targets"]
    lp = host(head.logprob(dev(case["h"], "bf16"), dev(t, "int32")))
    assert head.check() == 0
    z_ref, A = oracle_float_rows(W, case["h"], "bf16")
    assert np.allclose(oracle.logprob(z_ref, t), -np.log(V), rtol=0, atol=1e-12)
    tol = logprob_tol(A, oracle.logsumexp(z_ref), t)
    assert (np.abs(lp.astype(np.float64) + np.log(V)) <= tol).all()


@pytest.mark.parametrize("V,d", [(1000, 1040), (16, 16), (130, 2064), (1, 32)])
@pytest.mark.parametrize("B", [1, 5, 33, 100])
def test_int8_greedy_exact(torch_cuda, V, d, B):
    from invariant_output_head_gb300 import Head
    case = synth.small_int8(300 + V + d + B, V, d, B, n_ties=min(2, B), lo=-128, hi=127)
    head = Head(dev(case["W"], "int8"), "int8")
    tok, gap, z = head.greedy(dev(case["h"], "int8"), with_logits=True)
    assert head.check() == 0
    ref = oracle.head_greedy(case["W"], case["h"], "int8")
    assert (host(z).astype(np.int64) == ref["logits"]).all()
    assert (host(tok) == ref["token"]).all()
    assert (host(gap).astype(np.int64) == np.minimum(ref["gap"], 2**31 - 1)).all()


def test_int8_extreme_values_exact(torch_cuda):
    """Partial sums at the edge of fp32's exact-integer range: 1024 products
    of (-128)(-128) = 2^24 per K chunk, mixed with +-1 products."""
    from invariant_output_head_gb300 import Head
    V, d = 256, 4096
    W = np.full((V, d), -128, np.int8)
    W[1::2] = 127
    W[5, ::3] = 1
    W[7, 1024:2048] = -1
    h = np.full((4, d), -128, np.int8)
    h[1] = 127
    h[2, ::2] = 1
    h[3] = np.where(np.arange(d) % 1024 == 1023, 1, -128).astype(np.int8)
    head = Head(dev(W, "int8"), "int8")
    tok, gap, z = head.greedy(dev(h, "int8"), with_logits=True)
    ref = oracle.head_greedy(W, h, "int8")
    assert (host(z).astype(np.int64) == ref["logits"]).all()
    assert (host(tok) == ref["token"]).all()


@pytest.mark.parametrize("V,d", [(1000, 1040), (300, 4096), (129, 16)])
def test_int8_wide_batch_path_exact(torch_cuda, V, d):
    """B >= 256 runs the integer head on fp16 copies through the float
    projection kernel; exact, so it must agree bit for bit with the oracle
    and with the int8-streaming path used for small B."""
    from invariant_output_head_gb300 import Head
    case = synth.small_int8(500 + V, V, d, 300, n_ties=3, lo=-128, hi=127)
    head = Head(dev(case["W"], "int8"), "int8")
    h = dev(case["h"], "int8")
    tok, gap, z = head.greedy(h, with_logits=True)
    assert head.check() == 0
    ref = oracle.head_greedy(case["W"], case["h"], "int8")
    assert (host(z).astype(np.int64) == ref["logits"]).all()
    assert (host(tok) == ref["token"]).all()
    assert (host(gap).astype(np.int64) == np.minimum(ref["gap"], 2**31 - 1)).all()
    t2, g2, z2 = head.greedy(h[:40], with_logits=True)      # narrow path
    assert (host(z2) == host(z)[:40]).all() and (host(t2) == host(tok)[:40]).all()


@pytest.mark.parametrize("fmt", ["bf16", "int8"])
def test_verify_accept(torch_cuda, fmt):
    """Greedy speculative verify on 16 requests x 16 positions: tokens and
    gaps bitwise those of the plain greedy call, tokens equal to the oracle's,
    accepted lengths equal to the oracle's rule on drafts planted from the
    oracle's tokens."""
    from invariant_output_head_gb300 import Head
    torch = torch_cuda
    R, P = 16, 16
    if fmt == "int8":
        case = synth.small_int8(61, 1000, 1040, R * P)
        t_ref = oracle.head_greedy(case["W"], case["h"], "int8")["token"]
    else:
        case = synth.small_float(61, 1000, 520, R * P)
        t_ref = oracle.head_greedy(case["W"], case["h"], "bf16")["token"]
    drafts, cut = synth.plant_drafts(t_ref.reshape(R, P), case["V"], seed=3)
    acc_ref = oracle.verify_accept(t_ref.reshape(R, P), drafts)
    assert (acc_ref == cut).all()            # the planted mismatch is the first
    head = Head(dev(case["W"], fmt), fmt)
    h = dev(case["h"], fmt)
    t_plain, g_plain, _ = head.greedy(h)
    tok, gap, _, acc = head.verify(h, torch.from_numpy(drafts).cuda())
    assert head.check() == 0
    assert (host(tok) == t_ref).all()
    assert (host(tok) == host(t_plain)).all()
    assert (host(gap).view(np.uint32) == host(g_plain).view(np.uint32)).all()
    assert (host(acc) == acc_ref).all()


@pytest.mark.parametrize("R,P", [(1, 1), (3, 1), (1, 33), (5, 40), (9, 7)])
def test_verify_accept_shapes(torch_cuda, R, P):
    """Ragged request counts and draft lengths: single-position requests,
    P above a warp's 32 lanes, and request counts that leave the last merge
    blocks of a request in different waves (each row's block lowers its
    request's first-miss word with an order-free atomicMin)."""
    from invariant_output_head_gb300 import Head
    torch = torch_cuda
    case = synth.small_float(62 + P, 300, 136, R * P)
    t_ref = oracle.head_greedy(case["W"], case["h"], "bf16")["token"]
    drafts, _ = synth.plant_drafts(t_ref.reshape(R, P), case["V"], seed=R * 100 + P)
    head = Head(dev(case["W"], "bf16"), "bf16")
    tok, _, _, acc = head.verify(dev(case["h"], "bf16"), torch.from_numpy(drafts).cuda())
    assert head.check() == 0
    assert (host(tok) == t_ref).all()
    assert (host(acc) == oracle.verify_accept(t_ref.reshape(R, P), drafts)).all()


def test_verify_accept_call_sequence(torch_cuda):
    """Verify calls of changing shapes on one handle, interleaved with plain
    greedy calls: the per-request workspace returns to its idle state after
    every call, so each call's accepted lengths stand alone."""
    from invariant_output_head_gb300 import Head
    torch = torch_cuda
    case = synth.small_float(70, 400, 200, 360)
    t_ref = oracle.head_greedy(case["W"], case["h"], "bf16")["token"]
    head = Head(dev(case["W"], "bf16"), "bf16")
    h = dev(case["h"], "bf16")
    for k, (R, P) in enumerate([(4, 8), (4, 8), (2, 3), (30, 12), (9, 40), (4, 8)]):
        n = R * P
        drafts, _ = synth.plant_drafts(t_ref[:n].reshape(R, P), case["V"], seed=500 + k)
        _, _, _, acc = head.verify(h[:n], torch.from_numpy(drafts).cuda())
        head.greedy(h[:7])
        assert (host(acc) == oracle.verify_accept(t_ref[:n].reshape(R, P), drafts)).all(), (R, P)
    assert head.check() == 0


@pytest.mark.parametrize("fmt", ["bf16", "int8"])
def test_pair_kernel_logits_store_paths(torch_cuda, fmt):
    """Calls of more than 128 rows run on the CTA-pair kernel, whose logits go
    out through a tensor map when they are device memory with 16-byte aligned
    rows, and through plain stores otherwise (an unaligned logits pointer,
    pinned host memory written through its mapping). Every path gives the
    same bits, equal to the oracle's integer logits for the int8 head."""
    from invariant_output_head_gb300 import Head, binding
    torch = torch_cuda
    V, d, B = 1000, 256, 300 if fmt == "int8" else 200
    if fmt == "int8":
        case = synth.small_int8(611, V, d, B, n_ties=2)
    else:
        case = synth.small_float(611, V, d, B, fmt=fmt, n_ties=2)
    head = Head(dev(case["W"], fmt), fmt)
    h = dev(case["h"], fmt)
    tok, gap, z = (host(x) for x in head.greedy(h, with_logits=True))
    assert head.check() == 0
    s = torch.cuda.current_stream().cuda_stream
    # device logits starting 4 bytes into a buffer: rows not 16-byte aligned
    buf = torch.zeros(B * V + 1, dtype=torch.int32, device="cuda")
    tk = torch.empty(B, dtype=torch.int32, device="cuda")
    gp = torch.empty(B, dtype=torch.int32 if fmt == "int8" else torch.float32, device="cuda")
    binding.detlm_head_greedy(head.handle, h.data_ptr(), B, tk.data_ptr(), gp.data_ptr(),
                              buf.data_ptr() + 4, s)
    assert head.check() == 0
    zu = host(buf)[1:].reshape(B, V).view(z.dtype)
    assert (zu.view(np.uint32) == z.view(np.uint32)).all()
    assert (host(tk) == tok).all()
    # pinned host result buffers, written by the kernels directly
    h_pin = torch.from_numpy(np.ascontiguousarray(case["h"]).view(
        np.int8 if fmt == "int8" else np.int16)).pin_memory()
    o_tok = torch.empty(B, dtype=torch.int32).pin_memory()
    o_gap = torch.empty(B, dtype=gp.dtype).pin_memory()
    o_log = torch.empty((B, V), dtype=torch.int32 if fmt == "int8" else torch.float32).pin_memory()
    binding.detlm_head_greedy_host_async(head.handle, h_pin.data_ptr(), B, o_tok.data_ptr(),
                                         o_gap.data_ptr(), o_log.data_ptr(), s)
    assert head.check() == 0
    assert (o_log.numpy().view(np.uint32) == z.view(np.uint32)).all()
    assert (o_tok.numpy() == tok).all()
    assert (o_gap.numpy().view(np.uint32) == gap.view(np.uint32)).all()
    if fmt == "int8":
        assert (z.astype(np.int64) == oracle.logits_int(case["W"], case["h"])).all()
    head.close()
