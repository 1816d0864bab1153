"""Vocabulary-parallel heads on one GPU: P shard heads over row ranges of W,
their 16-byte records per hidden row stacked shard-major (the layout an
all-gather leaves), merged -- against the single head, bit for bit, and
against the oracle. The split follows "TandemLLM docs, 12 Exactness", 12.2:
the reduction order is fixed by the weight's shape, so it must not change with
the number of shards either."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import check_float_greedy, dev, host, logprob_tol, oracle_float_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import invariant_output_head_gb300 as ioh
    ioh.load_library()
    return torch


def _shards(W_raw, V, P, fmt):
    from invariant_output_head_gb300 import ShardHead, detlm_shard_range
    heads = []
    for r in range(P):
        v0, v1 = detlm_shard_range(V, P, r)
        heads.append(ShardHead(dev(W_raw[v0:v1], fmt), V, P, r, fmt))
    return heads


# (V, d, fmt, B): the PR1 head; the trainer head (594 log-prob tiles, so
# every leaf holds 4 or 5 tiles); a small fp16 head; a ragged vocabulary.
FLOAT_CASES = [(32000, 2048, "bf16", 5), (151936, 1536, "bf16", 300),
               (5000, 520, "fp16", 17), (20001, 264, "bf16", 64)]


@pytest.mark.parametrize("V,d,fmt,B", FLOAT_CASES)
def test_shards_match_single_head_bitwise(torch_cuda, V, d, fmt, B):
    from invariant_output_head_gb300 import Head, merge_greedy, merge_logprob
    torch = torch_cuda
    case = synth.small_float(7000 + V % 113 + B, V, d, B, fmt=fmt, n_ties=1, n_near=1)
    h = dev(case["h"], fmt)
    t = dev(case["targets"], "int32")
    single = Head(dev(case["W"], fmt), fmt)
    tok1, gap1, z1 = (host(x) for x in single.greedy(h, with_logits=True))
    lp1 = host(single.logprob(h, t))
    assert single.check() == 0
    single.close()
    n_tiles = (V + 255) // 256
    for P in (1, 2, 4, 8):
        if P > n_tiles:
            continue
        heads = _shards(case["W"], V, P, fmt)
        recs, zs = [], []
        for hd in heads:
            rec, z = hd.greedy_records(h, with_logits=True)
            recs.append(rec)
            zs.append(z)
        tok, gap = merge_greedy(torch.stack(recs), fmt)
        lrecs = torch.stack([hd.logprob_records(h, t) for hd in heads])
        lp = merge_logprob(lrecs, V, t)
        for hd in heads:
            assert hd.check() == 0
        assert (host(tok) == tok1).all(), P
        assert (host(gap).view(np.uint32) == gap1.view(np.uint32)).all(), P
        assert (host(torch.cat(zs, dim=1)).view(np.uint32) == z1.view(np.uint32)).all(), P
        assert (host(lp).view(np.uint32) == lp1.view(np.uint32)).all(), P
        for hd in heads:
            hd.close()
    rows = np.unique(np.array([0, 1, B - 1]))
    z_ref, A = oracle_float_rows(case["W"], case["h"][rows], fmt)
    check_float_greedy(z_ref, A, tok1[rows], gap1[rows], z1[rows], label=f"shards {V}")
    lp_ref = oracle.logprob(z_ref, case["targets"][rows])
    tol = logprob_tol(A, oracle.logsumexp(z_ref), case["targets"][rows])
    assert (np.abs(lp1[rows].astype(np.float64) - lp_ref) <= tol).all()


@pytest.mark.parametrize("B", [3, 300])
def test_int8_shards_exact(torch_cuda, B):
    """Integer head (streaming kernel at B = 3, wide path at B = 300) in 4
    shards, planted exact ties across shard boundaries."""
    from invariant_output_head_gb300 import Head, merge_greedy
    torch = torch_cuda
    V, d, P = 20000, 512, 4
    case = synth.small_int8(77 + B, V, d, B)
    W = case["W"].copy()
    from invariant_output_head_gb300 import detlm_shard_range
    b1 = detlm_shard_range(V, P, 1)[0]
    W[b1] = W[b1 - 3]            # a tie across the boundary of shards 0 and 1
    h = case["h"].copy()
    h[0] = W[b1]
    single = Head(dev(W, "int8"), "int8")
    tok1, gap1, z1 = (host(x) for x in single.greedy(dev(h, "int8"), with_logits=True))
    single.close()
    heads = _shards(W, V, P, "int8")
    hd8 = dev(h, "int8")
    recs, zs = zip(*[hd.greedy_records(hd8, with_logits=True) for hd in heads])
    tok, gap = merge_greedy(torch.stack(list(recs)), "int8")
    assert (host(tok) == tok1).all() and (host(gap) == gap1).all()
    assert (np.concatenate([host(z) for z in zs], axis=1) == z1).all()
    assert int(host(tok)[0]) == b1 - 3 and int(host(gap)[0]) == 0
    zr = oracle.logits_int(W, h[:2])
    assert (z1[:2].astype(np.int64) == zr).all()
    for hd in heads:
        assert hd.check() == 0
        hd.close()


def test_shard_errors(torch_cuda):
    from invariant_output_head_gb300 import (DETLM_EINVAL, DETLM_EUNSUPPORTED, DetlmError,
                                             ShardHead, binding, merge_logprob)
    torch = torch_cuda
    V, d = 2000, 64
    case = synth.small_float(5, V, d, 4)
    W = dev(case["W"], "bf16")
    with pytest.raises(DetlmError) as e:
        binding.detlm_head_create_shard(W.data_ptr(), V, d, 0, 3, 0)      # P not a power of two
    assert e.value.status == DETLM_EINVAL
    with pytest.raises(DetlmError) as e:                                   # 8 tiles, 16 shards
        binding.detlm_head_create_shard(W.data_ptr(), V, d, 0, 16, 0)
    assert e.value.status == DETLM_EINVAL
    v0, v1 = binding.detlm_shard_range(V, 2, 1)
    sh = ShardHead(dev(case["W"][v0:v1], "bf16"), V, 2, 1)
    h = dev(case["h"], "bf16")
    with pytest.raises(DetlmError) as e:
        sh.greedy(h)                                   # a whole-head call on a shard
    assert e.value.status == DETLM_EUNSUPPORTED
    # a target outside [0, V): NaN and the error bit
    sh0 = ShardHead(dev(case["W"][:v0], "bf16"), V, 2, 0)
    tg = torch.tensor([0, V, 1999, -1], dtype=torch.int32, device="cuda")
    recs = torch.stack([sh0.logprob_records(h, tg), sh.logprob_records(h, tg)])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp = host(merge_logprob(recs, V, tg, err=err))
    assert np.isnan(lp[1]) and np.isnan(lp[3]) and np.isfinite(lp[[0, 2]]).all()
    assert int(host(err)[0]) == 2
    sh.close()
    sh0.close()
