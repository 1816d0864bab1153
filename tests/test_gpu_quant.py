"""The integer front end ("Eliminating Nondeterminism in LLM Inference with
Integer-Only Arithmetic", section DetLLM): float rows quantized per token to
int8 with a dyadic multiplier, bit-exact against the oracle, and the int8
head fed by float rows, exact end to end."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import invariant_output_head_gb300 as ioh
    ioh.load_library()
    return torch


def fdev(torch, bits, fmt):
    if fmt == "fp32":
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.float32).copy()).cuda()
    return dev(bits, fmt)


@pytest.mark.parametrize("fmt", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("B,d", [(1, 8), (6, 1), (5, 7), (9, 33), (300, 1040), (64, 4096)])
def test_quantize_rows_exact(torch_cuda, fmt, B, d):
    import invariant_output_head_gb300 as ioh
    torch = torch_cuda
    bits = synth.float_rows(900 + B + d, B, d, fmt)
    q, m, s = ioh.quantize_rows(fdev(torch, bits, fmt))
    q_ref, m_ref, s_ref = oracle.quantize_rows(oracle.decode(bits, fmt))
    assert (host(q) == q_ref).all()
    assert (host(m).astype(np.int64) == m_ref).all()
    assert (host(s).astype(np.int64) == s_ref).all()
    # each row alone gives the same bits
    for n in range(min(B, 5)):
        q1, m1, s1 = ioh.quantize_rows(fdev(torch, bits[n:n + 1], fmt))
        assert (host(q1)[0] == q_ref[n]).all() and int(host(m1)[0]) == m_ref[n]


@pytest.mark.parametrize("fmt", ["bf16", "fp32"])
@pytest.mark.parametrize("B", [1, 17, 300])
def test_int8_head_from_float(torch_cuda, fmt, B):
    """float rows -> int8 -> exact int32 logits and lowest-index token."""
    from invariant_output_head_gb300 import Head
    torch = torch_cuda
    c = synth.small_int8(37, 1000, 1024, 1, n_ties=0)
    bits = synth.float_rows(950 + B, B, 1024, fmt)
    head = Head(dev(c["W"], "int8"), "int8")
    tok, gap, z, m, s = head.greedy_from_float(fdev(torch, bits, fmt), with_logits=True)
    assert head.check() == 0
    q_ref, m_ref, s_ref = oracle.quantize_rows(oracle.decode(bits, fmt))
    z_ref = oracle.logits_int(c["W"], q_ref)
    t_ref, g_ref, _, _ = oracle.greedy_int(z_ref)
    assert (host(z).astype(np.int64) == z_ref).all()
    assert (host(tok) == t_ref).all() and (host(gap).astype(np.int64) == g_ref).all()
    assert (host(m).astype(np.int64) == m_ref).all() and (host(s).astype(np.int64) == s_ref).all()
    # the same rows through the standalone quantizer and the int8 call
    import invariant_output_head_gb300 as ioh
    q, _, _ = ioh.quantize_rows(fdev(torch, bits, fmt))
    t2, g2, _ = head.greedy(q)
    assert (host(t2) == host(tok)).all() and (host(g2) == host(gap)).all()


def test_int8_head_from_float_full_size(torch_cuda):
    """The int8 head d=4096, V=128256 fed by 32 bf16 rows (the wide path at
    B >= 256 is covered by 300 rows on the small head above)."""
    from invariant_output_head_gb300 import Head
    torch = torch_cuda
    c = synth.int8_head(B=1)
    bits = synth.float_rows(977, 32, 4096, "bf16")
    head = Head(dev(c["W"], "int8"), "int8")
    tok, gap, z, _, _ = head.greedy_from_float(fdev(torch, bits, "bf16"), with_logits=True)
    assert head.check() == 0
    q_ref, _, _ = oracle.quantize_rows(oracle.decode(bits, "bf16"))
    rows = np.array([0, 1, 2, 3, 4, 17, 31])
    z_ref = oracle.logits_int(c["W"], q_ref[rows])
    assert (host(z)[rows].astype(np.int64) == z_ref).all()
    t_ref, g_ref, _, _ = oracle.greedy_int(z_ref)
    assert (host(tok)[rows] == t_ref).all() and (host(gap)[rows].astype(np.int64) == g_ref).all()
    assert (host(tok) == np.argmax(host(z), axis=1)).all()


def test_front_end_rejects(torch_cuda):
    import invariant_output_head_gb300 as ioh
    from invariant_output_head_gb300 import Head, DetlmError
    torch = torch_cuda
    cf = synth.small_float(6, 200, 64, 4)
    head = Head(dev(cf["W"], "bf16"), "bf16")
    x = dev(cf["h"], "bf16")
    with pytest.raises(DetlmError) as ei:
        ioh.detlm_head_greedy_from_float(head.handle, x.data_ptr(), ioh.DETLM_BF16, 4,
                                         x.data_ptr(), x.data_ptr(), None, None, None, None)
    assert ei.value.status == ioh.DETLM_EUNSUPPORTED
    q = torch.empty((4, 64), dtype=torch.int8, device="cuda")
    w = torch.empty(8, dtype=torch.int32, device="cuda")
    with pytest.raises(DetlmError) as ei:
        ioh.detlm_quantize_rows(x.data_ptr(), ioh.DETLM_INT8, 4, 64, q.data_ptr(), w.data_ptr(),
                                w.data_ptr(), None)
    assert ei.value.status == ioh.DETLM_EINVAL
    with pytest.raises(DetlmError) as ei:
        ioh.detlm_quantize_rows(x.data_ptr(), ioh.DETLM_BF16, 4, 0, q.data_ptr(), w.data_ptr(),
                                w.data_ptr(), None)
    assert ei.value.status == ioh.DETLM_EINVAL
    assert head.check() == 0
