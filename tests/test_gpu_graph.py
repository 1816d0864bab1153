"""Calls captured into a CUDA graph and replayed: after detlm_head_reserve a
call allocates nothing and launches only kernels (programmatic-dependent and
cluster launches included), so it can be captured; the replayed results must
equal the eagerly launched ones bit for bit -- for the one-CTA kernel, the
CTA-pair kernel (with its tensor-map logits stores), the log-prob kernel and
both integer paths."""
import numpy as np
import pytest

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


def _capture_and_compare(torch, run, outs):
    """run(stream_ptr) enqueues the calls writing into `outs`; eager first,
    then captured, the outputs cleared, replayed twice."""
    s = torch.cuda.current_stream().cuda_stream
    run(s)
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(ref, outs):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_float_calls_replay_bitwise(torch_cuda):
    from invariant_output_head_gb300 import Head, binding
    torch = torch_cuda
    V, d = 1000, 256
    case = synth.small_float(900, V, d, 300)
    head = Head(dev(case["W"], "bf16"), "bf16")
    head.reserve(300)
    h = dev(case["h"], "bf16")
    t = dev(case["targets"], "int32")
    outs = []
    calls = []
    for B in (1, 17, 300):         # one-CTA kernel (N = 16, 32), pair kernel
        o = (torch.empty(B, dtype=torch.int32, device="cuda"),
             torch.empty(B, dtype=torch.float32, device="cuda"),
             torch.empty((B, V), dtype=torch.float32, device="cuda"))
        outs += list(o)
        calls.append(("g", B, o))
    lp = torch.empty(64, dtype=torch.float32, device="cuda")
    outs.append(lp)

    def run(sp):
        for _, B, (tk, gp, lg) in calls:
            binding.detlm_head_greedy(head.handle, h.data_ptr(), B, tk.data_ptr(), gp.data_ptr(),
                                      lg.data_ptr(), sp)
        binding.detlm_head_logprob(head.handle, h.data_ptr(), t.data_ptr(), 64, lp.data_ptr(), sp)

    _capture_and_compare(torch, run, outs)
    assert head.check() == 0
    head.close()


def test_int8_calls_replay_bitwise(torch_cuda):
    from invariant_output_head_gb300 import Head, binding
    torch = torch_cuda
    V, d = 2000, 512
    case = synth.small_int8(901, V, d, 300, n_ties=2)
    head = Head(dev(case["W"], "int8"), "int8")
    binding.detlm_head_reserve(head.handle, 300)     # fp16 copies of the wide path
    h = dev(case["h"], "int8")
    outs, calls = [], []
    for B in (3, 300):             # streaming kernel, pair kernel on fp16 copies
        o = (torch.empty(B, dtype=torch.int32, device="cuda"),
             torch.empty(B, dtype=torch.int32, device="cuda"),
             torch.empty((B, V), dtype=torch.int32, device="cuda"))
        outs += list(o)
        calls.append((B, o))

    def run(sp):
        for B, (tk, gp, lg) in calls:
            binding.detlm_head_greedy(head.handle, h.data_ptr(), B, tk.data_ptr(), gp.data_ptr(),
                                      lg.data_ptr(), sp)

    _capture_and_compare(torch, run, outs)
    assert head.check() == 0
    z = host(outs[-1]).astype(np.int64)
    assert (z[:4] == np.asarray(case["h"][:4], np.int64) @ np.asarray(case["W"], np.int64).T).all()
    head.close()


def test_next_row_calls_replay_bitwise(torch_cuda):
    """The gated, sampling and speculative-verify calls captured and replayed
    (the verify call's per-request workspace words reset themselves, so
    every replay accepts the same lengths)."""
    from invariant_output_head_gb300 import Head, binding
    torch = torch_cuda
    V, d, B = 1000, 256, 160
    case = synth.small_float(902, V, d, B)
    head = Head(dev(case["W"], "bf16"), "bf16")
    head.reserve(B)
    h = dev(case["h"], "bf16")
    f32 = lambda *shape: torch.empty(*shape, dtype=torch.float32, device="cuda")  # noqa: E731
    i32 = lambda *shape: torch.empty(*shape, dtype=torch.int32, device="cuda")    # noqa: E731
    g_out = (i32(B), f32(B), f32(B, V), i32(B), f32(B))
    s_out = (i32(B), f32(B), f32(B, V))
    v_out = (i32(B), f32(B), f32(B, V), i32(B // 16))
    seeds = torch.arange(1, B + 1, dtype=torch.int64, device="cuda") * 0x3779B97F4A7C15 % (2**62)
    pos = torch.arange(B, dtype=torch.int64, device="cuda") * 7 + 3
    tok_ref, _, _ = head.greedy(h)
    drafts = tok_ref.clone()
    drafts[5] += 1                 # request 0 accepts 5 positions, the others all 16
    torch.cuda.synchronize()

    def run(sp):
        binding.detlm_head_greedy_gated(head.handle, h.data_ptr(), B, 0.001, g_out[0].data_ptr(),
                                        g_out[1].data_ptr(), g_out[2].data_ptr(),
                                        g_out[3].data_ptr(), g_out[4].data_ptr(), sp)
        binding.detlm_head_sample(head.handle, h.data_ptr(), B, 1.0, seeds.data_ptr(),
                                  pos.data_ptr(), s_out[0].data_ptr(), s_out[1].data_ptr(),
                                  s_out[2].data_ptr(), sp)
        binding.detlm_head_verify(head.handle, h.data_ptr(), B // 16, 16, drafts.data_ptr(),
                                  v_out[0].data_ptr(), v_out[1].data_ptr(), v_out[2].data_ptr(),
                                  v_out[3].data_ptr(), sp)

    _capture_and_compare(torch, run, list(g_out) + list(s_out) + list(v_out))
    assert head.check() == 0
    acc = host(v_out[3])
    assert acc[0] == 5 and (acc[1:] == 16).all()
    head.close()
