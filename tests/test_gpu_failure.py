"""Failure detection without faulting the GPU.

A device-side wait that runs out is provoked on purpose: the test hook makes
the MMA issuer wait on a barrier nothing arrives on, with a 20 ms limit. The
kernel gives up, records the timeout in the handle's error word and returns;
the host reads DETLM_ETIMEOUT, and the next call on the same context
succeeds. Bad arguments are refused on the host before any GPU work; an
out-of-range target id yields NaN and DETLM_ETARGET.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import check_float_greedy, dev, host, logprob_tol, oracle_float_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from invariant_output_head_gb300 import binding
    binding.load_library()
    return torch, binding


@pytest.mark.parametrize("fmt", ["bf16", "int8"])
def test_stalled_wait_reports_timeout_and_context_survives(env, fmt):
    torch, b = env
    if fmt == "int8":
        case = synth.small_int8(3, 700, 256, 9)
    else:
        case = synth.small_float(3, 700, 256, 9)
    head = b.Head(dev(case["W"], fmt), fmt)
    h = dev(case["h"], fmt)
    b.detlm_head_debug(head.handle, b.DETLM_DEBUG_STALL, 20_000_000)
    head.greedy(h, with_logits=True)
    torch.cuda.synchronize()
    assert head.check() == b.DETLM_ETIMEOUT
    b.detlm_head_debug(head.handle, 0, 0)
    t, g, z = head.greedy(h, with_logits=True)
    assert head.check() == b.DETLM_OK
    ref = oracle.head_greedy(case["W"], case["h"], fmt)
    assert (host(t) == ref["token"]).all()


def test_stalled_logprob_pair_kernel_times_out_and_recovers(env):
    """The log-prob projection runs on CTA pairs: the stalled leader's MMA
    warp gives up, both CTAs' waits run out, and the next call is right."""
    torch, b = env
    case = synth.small_float(5, 900, 384, 300)
    head = b.Head(dev(case["W"], "bf16"), "bf16")
    h, t = dev(case["h"], "bf16"), dev(case["targets"], "int32")
    b.detlm_head_debug(head.handle, b.DETLM_DEBUG_STALL, 20_000_000)
    head.logprob(h, t)
    torch.cuda.synchronize()
    assert head.check() == b.DETLM_ETIMEOUT
    b.detlm_head_debug(head.handle, 0, 0)
    lp = host(head.logprob(h, t))
    assert head.check() == b.DETLM_OK
    z_ref, A = oracle_float_rows(case["W"], case["h"], "bf16")
    lp_ref = oracle.logprob(z_ref, case["targets"])
    tol = logprob_tol(A, oracle.logsumexp(z_ref), case["targets"])
    assert (np.abs(lp.astype(np.float64) - lp_ref) <= tol).all()


@pytest.mark.parametrize("fmt", ["bf16", "int8"])
def test_stalled_wide_greedy_pair_kernel_times_out_and_recovers(env, fmt):
    """Greedy calls of more than 128 rows (integer: 256 or more) run on CTA
    pairs: the stalled leader's MMA warp gives up, both CTAs' waits run out,
    the loads already issued land before either CTA leaves, and the next
    call (logits through the tensor-map stores) is right."""
    torch, b = env
    B = 300
    if fmt == "int8":
        case = synth.small_int8(6, 1000, 256, B)
    else:
        case = synth.small_float(6, 1000, 256, B)
    head = b.Head(dev(case["W"], fmt), fmt)
    h = dev(case["h"], fmt)
    b.detlm_head_debug(head.handle, b.DETLM_DEBUG_STALL, 20_000_000)
    head.greedy(h, with_logits=True)
    torch.cuda.synchronize()
    assert head.check() == b.DETLM_ETIMEOUT
    b.detlm_head_debug(head.handle, 0, 0)
    t, g, z = head.greedy(h, with_logits=True)
    assert head.check() == b.DETLM_OK
    if fmt == "int8":
        assert (host(z).astype(np.int64) == oracle.logits_int(case["W"], case["h"])).all()
    else:
        z_ref, A = oracle_float_rows(case["W"], case["h"][:32], fmt)
        check_float_greedy(z_ref, A, host(t)[:32], host(g)[:32], host(z)[:32], label="pair stall")
    head.close()


def test_out_of_range_target_gives_nan_and_status(env):
    torch, b = env
    case = synth.small_float(4, 500, 128, 6)
    head = b.Head(dev(case["W"], "bf16"), "bf16")
    tg = case["targets"].copy()
    tg[1], tg[4] = -1, 500
    lp = host(head.logprob(dev(case["h"], "bf16"), dev(tg, "int32")))
    assert head.check() == b.DETLM_ETARGET
    assert np.isnan(lp[[1, 4]]).all() and np.isfinite(lp[[0, 2, 3, 5]]).all()
    assert head.check() == b.DETLM_OK        # the error word was cleared


def test_host_side_argument_errors(env):
    torch, b = env
    lib = b.load_library()
    case = synth.small_float(5, 300, 64, 4)
    W = dev(case["W"], "bf16")
    head = b.Head(W, "bf16")
    h = dev(case["h"], "bf16")
    tok = torch.empty(4, dtype=torch.int32, device="cuda")
    gap = torch.empty(4, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # misaligned hidden rows, null outputs, negative B
    assert lib.detlm_head_greedy(head.handle, h.data_ptr() + 2, 4, tok.data_ptr(),
                                 gap.data_ptr(), None, s) == b.DETLM_EINVAL
    assert lib.detlm_head_greedy(head.handle, h.data_ptr(), 4, None, gap.data_ptr(),
                                 None, s) == b.DETLM_EINVAL
    assert lib.detlm_head_greedy(head.handle, h.data_ptr(), -1, tok.data_ptr(),
                                 gap.data_ptr(), None, s) == b.DETLM_EINVAL
    # B = 0 is a no-op
    assert lib.detlm_head_greedy(head.handle, h.data_ptr(), 0, tok.data_ptr(),
                                 gap.data_ptr(), None, s) == b.DETLM_OK
    # log-prob is not defined for the integer head
    Wi = dev(synth.small_int8(5, 300, 64, 1)["W"], "int8")
    hi = b.Head(Wi, "int8")
    assert lib.detlm_head_logprob(hi.handle, h.data_ptr(), tok.data_ptr(), 4,
                                  gap.data_ptr(), s) == b.DETLM_EUNSUPPORTED
    # misaligned weight at create
    out = ctypes.c_void_p()
    assert lib.detlm_head_create(ctypes.byref(out), W.data_ptr() + 8, 300, 64,
                                 b.DETLM_BF16) == b.DETLM_EINVAL


def test_host_buffer_calls_match_device_calls(env):
    torch, b = env
    case = synth.small_float(6, 900, 256, 7)
    head = b.Head(dev(case["W"], "bf16"), "bf16")
    t, g, z = head.greedy(dev(case["h"], "bf16"), with_logits=True)
    lp = head.logprob(dev(case["h"], "bf16"), dev(case["targets"], "int32"))
    B, V = 7, 900
    th = np.empty(B, np.int32)
    gh = np.empty(B, np.float32)
    zh = np.empty((B, V), np.float32)
    lh = np.empty(B, np.float32)
    hb = np.ascontiguousarray(case["h"])
    s = torch.cuda.current_stream().cuda_stream
    b.detlm_head_greedy_host(head.handle, hb.ctypes.data, B, th.ctypes.data, gh.ctypes.data,
                             zh.ctypes.data, s)
    b.detlm_head_logprob_host(head.handle, hb.ctypes.data, case["targets"].ctypes.data, B,
                              lh.ctypes.data, s)
    assert (th == host(t)).all()
    assert (gh.view(np.uint32) == host(g).view(np.uint32)).all()
    assert (zh.view(np.uint32) == host(z).view(np.uint32)).all()
    assert (lh.view(np.uint32) == host(lp).view(np.uint32)).all()


def test_async_host_buffer_calls_match_device_calls(env):
    """Many asynchronous host-buffer calls of changing batch size (one result
    buffer set per call, pinned or pageable), one check at the end: every
    call's results equal the device call's bit for bit, whether the kernels
    wrote them to pinned host memory directly or they were staged and copied
    back while the next call ran."""
    torch, b = env
    V, d = 900, 256
    case = synth.small_float(16, V, d, 40)
    head = b.Head(dev(case["W"], "bf16"), "bf16")
    hd = dev(case["h"], "bf16")
    td = dev(case["targets"], "int32")
    t, g, z = (host(x) for x in head.greedy(hd, with_logits=True))
    lp = host(head.logprob(hd, td))
    h_pin = torch.from_numpy(np.ascontiguousarray(case["h"]).view(np.int16)).pin_memory()
    tg_pin = torch.from_numpy(case["targets"]).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    calls = [(0, 1), (1, 7), (8, 40 - 8), (3, 5), (0, 40), (39, 1)]
    outs = []
    for k, (r0, B) in enumerate(calls):
        # pinned result buffers (written by the kernels directly) and, every
        # other call, pageable ones (staged on the device, copied back)
        alloc = ((lambda *a, **kw: torch.empty(*a, **kw).pin_memory()) if k % 2 == 0
                 else (lambda *a, **kw: torch.empty(*a, **kw)))
        o = (alloc(B, dtype=torch.int32), alloc(B, dtype=torch.float32),
             alloc((B, V), dtype=torch.float32), alloc(B, dtype=torch.float32))
        hp = h_pin.data_ptr() + r0 * d * 2
        b.detlm_head_greedy_host_async(head.handle, hp, B, o[0].data_ptr(), o[1].data_ptr(),
                                       o[2].data_ptr(), s)
        b.detlm_head_logprob_host_async(head.handle, hp, tg_pin.data_ptr() + 4 * r0, B,
                                        o[3].data_ptr(), s)
        outs.append(o)
    assert head.check() == 0
    for (r0, B), o in zip(calls, outs):
        sl = slice(r0, r0 + B)
        assert (o[0].numpy() == t[sl]).all()
        assert (o[1].numpy().view(np.uint32) == g[sl].view(np.uint32)).all()
        assert (o[2].numpy().view(np.uint32) == z[sl].view(np.uint32)).all()
        assert (o[3].numpy().view(np.uint32) == lp[sl].view(np.uint32)).all()
    head.close()


def test_reserved_workspace_and_tiles(env):
    torch, b = env
    case = synth.small_float(7, 1000, 128, 300)
    head = b.Head(dev(case["W"], "bf16"), "bf16")
    b.detlm_head_reserve(head.handle, 300)
    assert head.tiles(1) == (8, 16)
    assert head.tiles(17) == (8, 32)
    assert head.tiles(128) == (8, 128)
    assert head.tiles(300) == (8, 256)
    t, g, _ = head.greedy(dev(case["h"], "bf16"))
    z_ref, A = oracle_float_rows(case["W"], case["h"], "bf16")
    check_float_greedy(z_ref, A, host(t), host(g), label="reserved")


def test_async_host_calls_with_large_logits(env):
    """Asynchronous host-buffer calls with several MB of logits written into
    pinned buffers (by the pair kernel, through the host mapping): several
    calls in a row, one check at the end, every result bitwise the device
    call's."""
    torch, b = env
    V, d, B = 6000, 256, 200                # 4.8 MB of logits per call
    case = synth.small_float(17, V, d, B)
    head = b.Head(dev(case["W"], "bf16"), "bf16")
    hd = dev(case["h"], "bf16")
    t, g, z = (host(x) for x in head.greedy(hd, with_logits=True))
    h_pin = torch.from_numpy(np.ascontiguousarray(case["h"]).view(np.int16)).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    outs = []
    for k in range(4):
        o = (torch.empty(B, dtype=torch.int32).pin_memory(),
             torch.empty(B, dtype=torch.float32).pin_memory(),
             torch.empty((B, V), dtype=torch.float32).pin_memory())
        b.detlm_head_greedy_host_async(head.handle, h_pin.data_ptr(), B, o[0].data_ptr(),
                                       o[1].data_ptr(), o[2].data_ptr(), s)
        outs.append(o)
    assert head.check() == 0
    for o in outs:
        assert (o[0].numpy() == t).all()
        assert (o[1].numpy().view(np.uint32) == g.view(np.uint32)).all()
        assert (o[2].numpy().view(np.uint32) == z.view(np.uint32)).all()
    head.close()


@pytest.mark.parametrize("B", [1, 160])
def test_device_calls_write_pinned_outputs(env, B):
    """Output pointers of the device calls may be page-locked host memory the
    device can address: the gated, sampling, verify and float-fed integer
    calls write their results straight into pinned buffers, bitwise what they
    write into device memory (B = 160: the wide kernels)."""
    torch, b = env
    V, d = 900, 256
    case = synth.small_float(21, V, d, B)
    head = b.Head(dev(case["W"], "bf16"), "bf16")
    h = dev(case["h"], "bf16")
    s = torch.cuda.current_stream().cuda_stream

    def outs(pinned, extra):
        mk = (lambda *a, **k: torch.empty(*a, **k).pin_memory()) if pinned else \
             (lambda *a, **k: torch.empty(*a, device="cuda", **k))
        return (mk(B, dtype=torch.int32), mk(B, dtype=torch.float32), mk((B, V), dtype=torch.float32),
                mk(max(extra, 1), dtype=torch.int32))
    res = {}
    for pinned in (False, True):
        o = outs(pinned, 2 * B)
        b.detlm_head_greedy_gated(head.handle, h.data_ptr(), B, 0.001, o[0].data_ptr(), o[1].data_ptr(),
                                  o[2].data_ptr(), o[3].data_ptr(), o[3].data_ptr() + 4 * B, s)
        seeds = torch.arange(1, B + 1, dtype=torch.int64, device="cuda") * 977
        pos = torch.arange(B, dtype=torch.int64, device="cuda")
        o2 = outs(pinned, 0)
        b.detlm_head_sample(head.handle, h.data_ptr(), B, 1.0, seeds.data_ptr(), pos.data_ptr(),
                            o2[0].data_ptr(), o2[1].data_ptr(), o2[2].data_ptr(), s)
        torch.cuda.synchronize()
        res[pinned] = [x.cpu() for x in o + o2[:3]]    # (o2[3] is not an output of sample)
    assert head.check() == 0
    for a, c in zip(res[False], res[True]):
        assert torch.equal(a.view(torch.int32), c.view(torch.int32))
    head.close()
