"""The greedy entry point that allocates no device memory.

Some callers may not allocate GPU memory at all (an inference server that has
already reserved all of HBM for itself, a plugin whose execute step must not
allocate, a latency-critical path that cannot take the synchronisation an
allocation implies). ``detlm_greedy_noalloc`` serves them: its workspace is a
static device array inside the library. This file checks, through the C ABI,
that two calls in a row give the same results as the handle-based
``detlm_head_greedy`` (bit for bit, since the kernels and their parameters are
the same; against the oracle within the tolerance every float parity test
uses), that the largest batch the static array holds gives the handle path's
bits too while one more row is refused before any GPU work, and that later
calls leave the device's free memory unchanged.

The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import LOGIT_RTOL, dev, host, oracle_float_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from invariant_output_head_gb300 import binding
    return torch, binding.load_library(), binding


def _noalloc(lib, torch, W, V, d, dtype, h, B, with_err=True):
    tok = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    gap = torch.full((B,), float("nan"), dtype=torch.float32, device="cuda")
    lg = torch.empty((B, V), dtype=torch.float32, device="cuda")
    err = torch.full((1,), 7, dtype=torch.int32, device="cuda") if with_err else None
    st = lib.detlm_greedy_noalloc(W.data_ptr(), V, d, dtype, h.data_ptr(), B,
                                  tok.data_ptr(), gap.data_ptr(), lg.data_ptr(),
                                  err.data_ptr() if err is not None else None,
                                  torch.cuda.current_stream().cuda_stream)
    return st, tok, gap, lg, err


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
def test_noalloc_matches_handle_path_two_calls(env, fmt):
    torch, lib, b = env
    V, d = 1000, 520
    case = synth.small_float(4242, V, d, 40, fmt=fmt, n_ties=2)
    W = dev(case["W"], fmt)
    hall = dev(case["h"], fmt)
    dtype = b.DTYPES[fmt]
    head = b.Head(W, fmt)
    z_ref, A = oracle_float_rows(case["W"], case["h"], fmt)
    # two calls in a row with different rows and batch sizes: the second must
    # not see anything the first left in the shared array
    for r0, B in ((0, 37), (5, 3)):
        h = hall[r0:r0 + B]
        st, tok, gap, lg, err = _noalloc(lib, torch, W, V, d, dtype, h, B)
        assert st == b.DETLM_OK, b.status_string(st)
        t_ref, g_ref, l_ref = head.greedy(h, with_logits=True)
        torch.cuda.synchronize()
        assert int(host(err)[0]) == 0
        assert (host(tok) == host(t_ref)).all()
        assert (host(lg).view(np.uint32) == host(l_ref).view(np.uint32)).all()
        assert (host(gap).view(np.uint32) == host(g_ref).view(np.uint32)).all()
        e = LOGIT_RTOL * A[r0:r0 + B]
        assert (np.abs(host(lg).astype(np.float64) - host(l_ref)) <= e).all()
        assert (np.abs(host(lg).astype(np.float64) - z_ref[r0:r0 + B]) <= e).all()
        m = np.max(host(l_ref), axis=1).astype(np.float64)
        assert (np.abs(host(gap) - host(g_ref)) * oracle.ulp_bf16(m) <= 2 * e.max(axis=1)).all()
    head.close()


def _max_rows(V):
    """Largest B the static array holds: the error word's 256 bytes and three
    record arrays of 4 * ceil(V / 128) * B bytes, each rounded up to 256."""
    n_vt = (V + 127) // 128

    def need(B):
        return 256 + 3 * ((4 * n_vt * B + 255) // 256 * 256)
    B = (8 << 20) // (12 * n_vt)
    while need(B) > (8 << 20):
        B -= 1
    while need(B + 1) <= (8 << 20):
        B += 1
    return B


def test_noalloc_largest_batch_bitwise(env):
    """V = 32000: the largest batch that fits (several 256-row column tiles)
    gives the handle path's bits; one row more is refused."""
    torch, lib, b = env
    V, d = 32000, 64
    Bmax = _max_rows(V)
    assert Bmax > 256
    case = synth.small_float(4343, V, d, Bmax)
    W = dev(case["W"], "bf16")
    h = dev(case["h"], "bf16")
    st, tok, gap, lg, err = _noalloc(lib, torch, W, V, d, b.DETLM_BF16, h, Bmax)
    assert st == b.DETLM_OK, b.status_string(st)
    head = b.Head(W, "bf16")
    t_ref, g_ref, l_ref = head.greedy(h, with_logits=True)
    torch.cuda.synchronize()
    assert int(host(err)[0]) == 0
    assert (host(tok) == host(t_ref)).all()
    assert (host(gap).view(np.uint32) == host(g_ref).view(np.uint32)).all()
    assert (host(lg).view(np.uint32) == host(l_ref).view(np.uint32)).all()
    rows = np.array([0, 255, 256, Bmax - 1])
    z_ref, A = oracle_float_rows(case["W"], case["h"][rows], "bf16")
    assert (np.abs(host(lg)[rows].astype(np.float64) - z_ref) <= LOGIT_RTOL * A).all()
    head.close()
    h1 = torch.zeros((Bmax + 1, d), dtype=torch.bfloat16, device="cuda")
    st, *_ = _noalloc(lib, torch, W, V, d, b.DETLM_BF16, h1, Bmax + 1)
    assert st == b.DETLM_EINVAL


def test_noalloc_refuses_oversized_batch_and_int8(env):
    torch, lib, b = env
    V, d = 32000, 64
    W = torch.zeros((V, d), dtype=torch.bfloat16, device="cuda")
    too_big = _max_rows(V) + 1
    h = torch.zeros((too_big, d), dtype=torch.bfloat16, device="cuda")
    st, *_ = _noalloc(lib, torch, W, V, d, b.DETLM_BF16, h, too_big)
    assert st == b.DETLM_EINVAL
    Wi = torch.zeros((V, d), dtype=torch.int8, device="cuda")
    hi = torch.zeros((1, d), dtype=torch.int8, device="cuda")
    st, *_ = _noalloc(lib, torch, Wi, V, d, b.DETLM_INT8, hi, 1)
    assert st == b.DETLM_EUNSUPPORTED


def test_noalloc_leaves_free_memory_unchanged(env):
    torch, lib, b = env
    V, d, B = 4096, 256, 8
    case = synth.small_float(77, V, d, B)
    W = dev(case["W"], "bf16")
    h = dev(case["h"], "bf16")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    gap = torch.empty(B, dtype=torch.float32, device="cuda")
    sp = torch.cuda.current_stream().cuda_stream
    assert lib.detlm_greedy_noalloc(W.data_ptr(), V, d, b.DETLM_BF16, h.data_ptr(), B,
                                    tok.data_ptr(), gap.data_ptr(), None, None, sp) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert lib.detlm_greedy_noalloc(W.data_ptr(), V, d, b.DETLM_BF16, h.data_ptr(), B,
                                        tok.data_ptr(), gap.data_ptr(), None, None, sp) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    ref = oracle.head_greedy(case["W"], case["h"], "bf16")
    assert (host(tok) == ref["token"]).all()
