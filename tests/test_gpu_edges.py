"""Edge cases across the entry points: empty batches (every call returns at
once and the handle keeps working), the largest supported integer K
(d = 16384, |logit| up to 2^28, streaming and wide paths), a long float K
and d = 8 (one partial K box).
"""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import check_float_greedy, dev, host, oracle_float_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import invariant_output_head_gb300 as ioh
    ioh.load_library()
    return torch


def test_empty_batches(torch_cuda):
    import invariant_output_head_gb300 as ioh
    from invariant_output_head_gb300 import Head
    torch = torch_cuda
    cf = synth.small_float(11, 500, 136, 3)
    head = Head(dev(cf["W"], "bf16"), "bf16")
    h0 = dev(cf["h"], "bf16")[:0]
    t, g, z = head.greedy(h0, with_logits=True)
    assert t.numel() == 0 and z.shape == (0, 500)
    assert head.logprob(h0, torch.empty(0, dtype=torch.int32, device="cuda")).numel() == 0
    assert head.greedy_gated(h0, 0.001)[0].numel() == 0
    e64 = torch.empty(0, dtype=torch.int64, device="cuda")
    assert head.sample(h0, 1.0, e64, e64)[0].numel() == 0
    ioh.detlm_head_verify(head.handle, None, 0, 16, None, None, None, None, None, None)
    # the handle still works, exactly as before
    t3, g3, z3 = head.greedy(dev(cf["h"], "bf16"), with_logits=True)
    z_ref, A = oracle_float_rows(cf["W"], cf["h"], "bf16")
    check_float_greedy(z_ref, A, host(t3), host(g3), host(z3), label="after empty calls")
    c8 = synth.small_int8(12, 300, 64, 2)
    head8 = Head(dev(c8["W"], "int8"), "int8")
    assert head8.greedy(dev(c8["h"], "int8")[:0])[0].numel() == 0
    x0 = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    assert head8.greedy_from_float(x0)[0].numel() == 0
    q, m, s = ioh.quantize_rows(x0)
    assert q.shape == (0, 64)
    t8, _, _ = head8.greedy(dev(c8["h"], "int8"))
    assert (host(t8) == oracle.greedy_int(oracle.logits_int(c8["W"], c8["h"]))[0]).all()
    assert head.check() == 0 and head8.check() == 0


@pytest.mark.parametrize("B", [3, 300])
def test_int8_largest_k_extremes(torch_cuda, B):
    """d = 16384 with every value -128: each logit is 2^28, the largest the
    integer head admits; plus random rows, both exact."""
    from invariant_output_head_gb300 import Head
    V, d = 200, 16384
    rng = np.random.default_rng(5)
    W = rng.integers(-128, 128, size=(V, d), dtype=np.int8)
    h = rng.integers(-128, 128, size=(B, d), dtype=np.int8)
    W[7] = -128
    h[0] = -128
    head = Head(dev(W, "int8"), "int8")
    t, g, z = head.greedy(dev(h, "int8"), with_logits=True)
    t, g, z = host(t), host(g), host(z)
    assert head.check() == 0
    rows = np.unique(np.array([0, 1, B // 2, B - 1]))
    z_ref = oracle.logits_int(W, h[rows])
    assert int(z_ref[0, 7]) == 2 ** 28
    assert (z[rows].astype(np.int64) == z_ref).all()
    tr, gr, _, _ = oracle.greedy_int(z_ref)
    assert (t[rows] == tr).all() and (g[rows].astype(np.int64) == gr).all()


def test_float_long_k(torch_cuda):
    """bf16, d = 16384 (128 K chunks), within the logit tolerance."""
    from invariant_output_head_gb300 import Head
    c = synth.small_float(13, 700, 16384, 5, sigma_w=0.01)
    head = Head(dev(c["W"], "bf16"), "bf16")
    t, g, z = head.greedy(dev(c["h"], "bf16"), with_logits=True)
    assert head.check() == 0
    z_ref, A = oracle_float_rows(c["W"], c["h"], "bf16")
    check_float_greedy(z_ref, A, host(t), host(g), host(z), label="d=16384")


def test_smallest_d(torch_cuda):
    """d = 8: one K box, mostly zero fill."""
    from invariant_output_head_gb300 import Head
    c = synth.small_float(14, 333, 8, 20)
    head = Head(dev(c["W"], "bf16"), "bf16")
    t, g, z = head.greedy(dev(c["h"], "bf16"), with_logits=True)
    z_ref, A = oracle_float_rows(c["W"], c["h"], "bf16")
    check_float_greedy(z_ref, A, host(t), host(g), host(z), label="d=8")
    assert head.check() == 0
