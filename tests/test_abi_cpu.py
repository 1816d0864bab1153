"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
entry point the header declares, and rejects bad arguments on the host
before touching CUDA. No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "detlm_head.h")


@pytest.fixture(scope="module")
def lib():
    from invariant_output_head_gb300 import build, binding
    build.build()
    return binding.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char\s*\*)\s+(detlm_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_entry_points():
    syms = declared_symbols()
    for name in ("detlm_head_create", "detlm_head_greedy", "detlm_head_logprob",
                 "detlm_head_destroy", "detlm_status_string"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in the header but not exported"


def test_binding_covers_every_declared_symbol():
    from invariant_output_head_gb300 import binding
    for name in declared_symbols():
        assert name in binding._SIGS, name
        assert hasattr(binding, name), name


def test_status_strings(lib):
    from invariant_output_head_gb300 import binding as b
    for st in (b.DETLM_OK, b.DETLM_EINVAL, b.DETLM_EUNSUPPORTED, b.DETLM_ECUDA,
               b.DETLM_ETIMEOUT, b.DETLM_ENOMEM, b.DETLM_ETARGET):
        s = b.status_string(st)
        assert s and s != "unknown status"
    assert b.status_string(12345) == "unknown status"


def _create(lib, ptr, V, d, dtype):
    out = ctypes.c_void_p(0)
    st = lib.detlm_head_create(ctypes.byref(out), ptr, V, d, dtype)
    return st, out.value


def test_create_rejects_bad_arguments_before_cuda(lib):
    from invariant_output_head_gb300 import binding as b
    fake = 0x7F0000000000          # never dereferenced: validation fails first
    assert lib.detlm_head_create(None, fake, 10, 16, 0) == b.DETLM_EINVAL
    cases = [
        (None, 10, 16, b.DETLM_BF16),          # null weight
        (fake + 8, 10, 16, b.DETLM_BF16),      # W not 16-byte aligned
        (fake, 0, 16, b.DETLM_BF16),           # V = 0
        (fake, 2**31, 16, b.DETLM_BF16),       # V too large
        (fake, 10, 0, b.DETLM_BF16),           # d = 0
        (fake, 10, 12, b.DETLM_BF16),          # bf16 row not a multiple of 16 bytes
        (fake, 10, 12, b.DETLM_FP16),
        (fake, 10, 24, b.DETLM_INT8),          # int8 row not a multiple of 16 bytes
        (fake, 10, 32768, b.DETLM_INT8),       # int8 d above the exact-sum limit
        (fake, 10, 16, 7),                     # unknown dtype
    ]
    for ptr, V, d, dt in cases:
        st, h = _create(lib, ptr, V, d, dt)
        assert st == b.DETLM_EINVAL and not h, (ptr, V, d, dt, st)


def test_calls_on_null_handle_are_rejected(lib):
    from invariant_output_head_gb300 import binding as b
    assert lib.detlm_head_greedy(None, None, 1, None, None, None, None) == b.DETLM_EINVAL
    assert lib.detlm_head_logprob(None, None, None, 1, None, None) == b.DETLM_EINVAL
    assert lib.detlm_head_greedy_host(None, None, 1, None, None, None, None) == b.DETLM_EINVAL
    assert lib.detlm_head_logprob_host(None, None, None, 1, None, None) == b.DETLM_EINVAL
    assert lib.detlm_head_check(None, None) == b.DETLM_EINVAL
    assert lib.detlm_head_reserve(None, 4) == b.DETLM_EINVAL
    assert lib.detlm_head_debug(None, 0, 0) == b.DETLM_EINVAL
    assert lib.detlm_head_time_next(None, None, None) == b.DETLM_EINVAL
    nv, nc = ctypes.c_int32(), ctypes.c_int32()
    assert lib.detlm_head_tiles(None, 1, ctypes.byref(nv), ctypes.byref(nc)) == b.DETLM_EINVAL
    lib.detlm_head_destroy(None)   # no-op


def test_create_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from invariant_output_head_gb300 import binding as b
    st, h = _create(lib, 0x7F0000000000, 32000, 2048, b.DETLM_BF16)
    assert st == b.DETLM_ECUDA and not h


def test_package_has_no_cpu_fallback():
    """The product package never imports the oracle or computes on the CPU."""
    pkg = os.path.join(ROOT, "invariant_output_head_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "numpy" not in text or f == "build.py", f


def test_shard_calls_reject_bad_arguments_on_the_host(lib):
    from invariant_output_head_gb300 import binding as b
    buf = ctypes.create_string_buffer(64)
    assert lib.detlm_head_greedy_shard(None, buf, 1, buf, None, None) == b.DETLM_EINVAL
    assert lib.detlm_head_logprob_shard(None, buf, buf, 1, buf, None) == b.DETLM_EINVAL
    for P in (0, 3, 256):
        assert lib.detlm_merge_greedy_shards(buf, P, 1, b.DETLM_BF16, buf, buf, None) == \
            b.DETLM_EINVAL
        assert lib.detlm_merge_logprob_shards(buf, P, 1, 100, buf, buf, None, None) == \
            b.DETLM_EINVAL
    assert lib.detlm_merge_greedy_shards(buf, 2, 1, 7, buf, buf, None) == b.DETLM_EINVAL
    assert lib.detlm_merge_logprob_shards(buf, 2, 1, 0, buf, buf, None, None) == b.DETLM_EINVAL
    assert lib.detlm_merge_greedy_shards(None, 2, 1, b.DETLM_BF16, buf, buf, None) == \
        b.DETLM_EINVAL
    assert lib.detlm_merge_greedy_shards(buf, 2, 0, b.DETLM_BF16, None, None, None) == b.DETLM_OK
    out = ctypes.c_void_p(0)
    assert lib.detlm_head_create_shard(ctypes.byref(out), buf, 1000, 64, b.DETLM_BF16, 3, 0) == \
        b.DETLM_EINVAL


def test_peak_probe_library_loads_and_exports_its_entry_point():
    from invariant_output_head_gb300 import build
    build.build()
    probe = ctypes.CDLL(build.PEAK_LIB)
    assert hasattr(probe, "detlm_mma_f16_peak")
