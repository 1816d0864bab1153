"""Thin ctypes binding of the C ABI in ``include/detlm_head.h``.

Argument marshalling only: every step of the output head runs in the CUDA
library. Functions keep the C names; ``Head`` wraps a handle for torch
tensors (device memory and streams come from PyTorch). There is no fallback:
if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib",
                         "libdetlm_head.so")

DETLM_BF16, DETLM_FP16, DETLM_INT8, DETLM_FP32 = 0, 1, 2, 3
DTYPES = {"bf16": DETLM_BF16, "fp16": DETLM_FP16, "int8": DETLM_INT8}
DETLM_OK, DETLM_EINVAL, DETLM_EUNSUPPORTED, DETLM_ECUDA = 0, -1, -2, -3
DETLM_ETIMEOUT, DETLM_ENOMEM, DETLM_ETARGET = -4, -5, -6
DETLM_DEBUG_STALL = 1

_vp, _i64, _i32, _u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
_SIGS = {
    "detlm_head_create": (_i32, [ctypes.POINTER(_vp), _vp, _i64, _i64, _i32]),
    "detlm_head_reserve": (_i32, [_vp, _i64]),
    "detlm_head_greedy": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp]),
    "detlm_head_logprob": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "detlm_head_verify": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "detlm_head_greedy_gated": (_i32, [_vp, _vp, _i64, ctypes.c_float, _vp, _vp, _vp, _vp, _vp,
                                       _vp]),
    "detlm_head_sample": (_i32, [_vp, _vp, _i64, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp]),
    "detlm_quantize_rows": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp, _vp, _vp]),
    "detlm_head_greedy_from_float": (_i32, [_vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "detlm_head_greedy_host": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp]),
    "detlm_head_logprob_host": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "detlm_head_greedy_host_async": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _vp]),
    "detlm_head_logprob_host_async": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "detlm_head_check": (_i32, [_vp, _vp]),
    "detlm_head_time_next": (_i32, [_vp, _vp, _vp]),
    "detlm_head_debug": (_i32, [_vp, _i32, _u64]),
    "detlm_head_tiles": (_i32, [_vp, _i64, ctypes.POINTER(ctypes.c_int32),
                                ctypes.POINTER(ctypes.c_int32)]),
    "detlm_head_destroy": (None, [_vp]),
    "detlm_status_string": (ctypes.c_char_p, [_i32]),
    "detlm_greedy_noalloc": (_i32, [_vp, _i64, _i64, _i32, _vp, _i64, _vp, _vp, _vp, _vp, _vp]),
    "detlm_shard_range": (_i32, [_i64, _i32, _i32, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
    "detlm_head_create_shard": (_i32, [ctypes.POINTER(_vp), _vp, _i64, _i64, _i32, _i32, _i32]),
    "detlm_head_greedy_shard": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp]),
    "detlm_head_logprob_shard": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "detlm_merge_greedy_shards": (_i32, [_vp, _i32, _i64, _i32, _vp, _vp, _vp]),
    "detlm_merge_logprob_shards": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp, _vp, _vp]),
}

_lib = None


def _float_dtype_code(x) -> int:
    import torch
    codes = {torch.bfloat16: DETLM_BF16, torch.float16: DETLM_FP16, torch.float32: DETLM_FP32}
    if x.dtype not in codes:
        raise ValueError("float rows must be bfloat16, float16 or float32")
    return codes[x.dtype]


def quantize_rows(x, stream=None):
    """Integer front end on a float CUDA tensor x [B, d]: returns (q int8
    [B, d], mult int32 [B], shift int32 [B])."""
    import torch
    xd = _float_dtype_code(x)
    if not x.is_cuda or not x.is_contiguous() or x.dim() != 2:
        raise ValueError("x must be a contiguous 2-D CUDA tensor")
    B, d = int(x.shape[0]), int(x.shape[1])
    q = torch.empty((B, d), dtype=torch.int8, device=x.device)
    mult = torch.empty(B, dtype=torch.int32, device=x.device)
    shift = torch.empty(B, dtype=torch.int32, device=x.device)
    detlm_quantize_rows(x.data_ptr(), xd, B, d, q.data_ptr(), mult.data_ptr(),
                        shift.data_ptr(), _stream_ptr(stream))
    return q, mult, shift


class DetlmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the CUDA library (built by ``invariant_output_head_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with "
            "`python -m invariant_output_head_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().detlm_status_string(status).decode()


def _check(st: int, what: str):
    if st != DETLM_OK:
        raise DetlmError(st, what)


# ---- the C entry points, by name (pointers and streams as ints) ----------

def detlm_head_create(W_ptr: int, V: int, d: int, dtype: int) -> int:
    out = _vp()
    _check(load_library().detlm_head_create(ctypes.byref(out), W_ptr, V, d, dtype),
           "detlm_head_create")
    return out.value


def detlm_head_reserve(handle: int, max_B: int) -> None:
    _check(load_library().detlm_head_reserve(handle, max_B), "detlm_head_reserve")


def detlm_head_greedy(handle, h_ptr, B, token_ptr, gap_ptr, logits_ptr, stream) -> None:
    _check(load_library().detlm_head_greedy(handle, h_ptr, B, token_ptr, gap_ptr,
                                            logits_ptr, stream), "detlm_head_greedy")


def detlm_head_logprob(handle, h_ptr, targets_ptr, B, logp_ptr, stream) -> None:
    _check(load_library().detlm_head_logprob(handle, h_ptr, targets_ptr, B, logp_ptr,
                                             stream), "detlm_head_logprob")


def detlm_head_greedy_gated(handle, h_ptr, B, tau, token_ptr, gap_ptr, logits_ptr,
                            base_token_ptr, margin_ptr, stream) -> None:
    _check(load_library().detlm_head_greedy_gated(handle, h_ptr, B, tau, token_ptr, gap_ptr,
                                                  logits_ptr, base_token_ptr, margin_ptr,
                                                  stream),
           "detlm_head_greedy_gated")


def detlm_head_sample(handle, h_ptr, B, temperature, seeds_ptr, positions_ptr, token_ptr,
                      score_gap_ptr, logits_ptr, stream) -> None:
    _check(load_library().detlm_head_sample(handle, h_ptr, B, temperature, seeds_ptr,
                                            positions_ptr, token_ptr, score_gap_ptr, logits_ptr,
                                            stream),
           "detlm_head_sample")


def detlm_quantize_rows(x_ptr, dtype, B, d, q_ptr, mult_ptr, shift_ptr, stream) -> None:
    _check(load_library().detlm_quantize_rows(x_ptr, dtype, B, d, q_ptr, mult_ptr, shift_ptr,
                                              stream),
           "detlm_quantize_rows")


def detlm_head_greedy_from_float(handle, x_ptr, x_dtype, B, token_ptr, gap_ptr, logits_ptr,
                                 mult_ptr, shift_ptr, stream) -> None:
    _check(load_library().detlm_head_greedy_from_float(handle, x_ptr, x_dtype, B, token_ptr,
                                                       gap_ptr, logits_ptr, mult_ptr, shift_ptr,
                                                       stream),
           "detlm_head_greedy_from_float")


def detlm_head_verify(handle, h_ptr, n_req, P, drafts_ptr, token_ptr, gap_ptr, logits_ptr,
                      accepted_ptr, stream) -> None:
    _check(load_library().detlm_head_verify(handle, h_ptr, n_req, P, drafts_ptr, token_ptr,
                                            gap_ptr, logits_ptr, accepted_ptr, stream),
           "detlm_head_verify")


def detlm_head_greedy_host(handle, h_ptr, B, token_ptr, gap_ptr, logits_ptr, stream) -> None:
    _check(load_library().detlm_head_greedy_host(handle, h_ptr, B, token_ptr, gap_ptr,
                                                 logits_ptr, stream),
           "detlm_head_greedy_host")


def detlm_head_logprob_host(handle, h_ptr, targets_ptr, B, logp_ptr, stream) -> None:
    _check(load_library().detlm_head_logprob_host(handle, h_ptr, targets_ptr, B,
                                                  logp_ptr, stream),
           "detlm_head_logprob_host")


def detlm_head_greedy_host_async(handle, h_ptr, B, token_ptr, gap_ptr, logits_ptr,
                                 stream) -> None:
    _check(load_library().detlm_head_greedy_host_async(handle, h_ptr, B, token_ptr, gap_ptr,
                                                       logits_ptr, stream),
           "detlm_head_greedy_host_async")


def detlm_head_logprob_host_async(handle, h_ptr, targets_ptr, B, logp_ptr, stream) -> None:
    _check(load_library().detlm_head_logprob_host_async(handle, h_ptr, targets_ptr, B,
                                                        logp_ptr, stream),
           "detlm_head_logprob_host_async")


def detlm_head_check(handle, stream) -> int:
    return load_library().detlm_head_check(handle, stream)


def detlm_head_time_next(handle, start_evt: int, stop_evt: int) -> None:
    _check(load_library().detlm_head_time_next(handle, start_evt, stop_evt),
           "detlm_head_time_next")


def detlm_head_debug(handle, flags: int, timeout_ns: int = 0) -> None:
    _check(load_library().detlm_head_debug(handle, flags, timeout_ns), "detlm_head_debug")


def detlm_head_tiles(handle, B: int):
    nv, nc = ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().detlm_head_tiles(handle, B, ctypes.byref(nv), ctypes.byref(nc)),
           "detlm_head_tiles")
    return nv.value, nc.value


def detlm_head_destroy(handle) -> None:
    if handle:
        load_library().detlm_head_destroy(handle)


def detlm_status_string(status: int) -> str:
    return status_string(status)


def detlm_greedy_noalloc(W_ptr, V, d, dtype, h_ptr, B, token_ptr, gap_ptr, logits_ptr,
                         err_ptr, stream) -> None:
    """Greedy call that allocates no device memory (its workspace is a static
    device array inside the library); for callers that may not allocate."""
    _check(load_library().detlm_greedy_noalloc(W_ptr, V, d, dtype, h_ptr, B, token_ptr,
                                               gap_ptr, logits_ptr, err_ptr, stream),
           "detlm_greedy_noalloc")


def detlm_shard_range(V: int, P: int, rank: int):
    """(v_begin, v_end): the vocabulary rows shard `rank` of P holds (host only)."""
    a, b = _i64(), _i64()
    _check(load_library().detlm_shard_range(V, P, rank, ctypes.byref(a), ctypes.byref(b)),
           "detlm_shard_range")
    return a.value, b.value


def detlm_head_create_shard(W_ptr: int, V: int, d: int, dtype: int, P: int, rank: int) -> int:
    out = _vp()
    _check(load_library().detlm_head_create_shard(ctypes.byref(out), W_ptr, V, d, dtype, P, rank),
           "detlm_head_create_shard")
    return out.value


def detlm_head_greedy_shard(handle, h_ptr, B, rec_ptr, logits_ptr, stream) -> None:
    _check(load_library().detlm_head_greedy_shard(handle, h_ptr, B, rec_ptr, logits_ptr, stream),
           "detlm_head_greedy_shard")


def detlm_head_logprob_shard(handle, h_ptr, targets_ptr, B, rec_ptr, stream) -> None:
    _check(load_library().detlm_head_logprob_shard(handle, h_ptr, targets_ptr, B, rec_ptr,
                                                   stream),
           "detlm_head_logprob_shard")


def detlm_merge_greedy_shards(recs_ptr, P, B, dtype, token_ptr, gap_ptr, stream) -> None:
    _check(load_library().detlm_merge_greedy_shards(recs_ptr, P, B, dtype, token_ptr, gap_ptr,
                                                    stream),
           "detlm_merge_greedy_shards")


def detlm_merge_logprob_shards(recs_ptr, P, B, V, targets_ptr, logp_ptr, err_ptr, stream) -> None:
    _check(load_library().detlm_merge_logprob_shards(recs_ptr, P, B, V, targets_ptr, logp_ptr,
                                                     err_ptr, stream),
           "detlm_merge_logprob_shards")


# ---- torch convenience wrapper ------------------------------------------

def _stream_ptr(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Head:
    """One output head over a device weight W [V, d] (bf16, fp16 or int8 tensor).

    The handle borrows W: keep the tensor alive while the Head is in use.
    """

    def __init__(self, W, dtype: str | None = None):
        import torch
        if dtype is None:
            dtype = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.int8: "int8"}[W.dtype]
        if not W.is_cuda or not W.is_contiguous() or W.dim() != 2:
            raise ValueError("W must be a contiguous 2-D CUDA tensor [V, d]")
        self.W = W
        self.dtype = dtype
        self.V, self.d = int(W.shape[0]), int(W.shape[1])
        self.handle = detlm_head_create(W.data_ptr(), self.V, self.d, DTYPES[dtype])

    def close(self):
        if getattr(self, "handle", None):
            detlm_head_destroy(self.handle)
            self.handle = None

    def reserve(self, max_B: int) -> None:
        """Workspace (and, for an int8 head, the wide path's fp16 copies) for
        calls of up to max_B rows: such calls then allocate nothing and can be
        captured into a CUDA graph (detlm_head_reserve)."""
        detlm_head_reserve(self.handle, int(max_B))

    def __del__(self):
        try:
            self.close()
        except Exception:   # noqa: BLE001 - interpreter shutdown
            pass

    def _check_h(self, h):
        if not h.is_cuda or not h.is_contiguous() or h.dim() != 2 or h.shape[1] != self.d:
            raise ValueError(f"h must be a contiguous CUDA tensor [B, {self.d}]")

    def greedy(self, h, with_logits: bool = False, stream=None, out=None):
        """Returns (token int32 [B], gap [B], logits [B, V] or None) on h's device."""
        import torch
        self._check_h(h)
        B = int(h.shape[0])
        gdt = torch.int32 if self.dtype == "int8" else torch.float32
        if out is None:
            token = torch.empty(B, dtype=torch.int32, device=h.device)
            gap = torch.empty(B, dtype=gdt, device=h.device)
            logits = torch.empty((B, self.V), dtype=gdt, device=h.device) if with_logits else None
        else:
            token, gap, logits = out
        detlm_head_greedy(self.handle, h.data_ptr(), B, token.data_ptr(), gap.data_ptr(),
                          logits.data_ptr() if logits is not None else None,
                          _stream_ptr(stream))
        return token, gap, logits

    def logprob(self, h, targets, stream=None, out=None):
        import torch
        self._check_h(h)
        B = int(h.shape[0])
        if targets.dtype != torch.int32 or not targets.is_cuda or targets.numel() != B:
            raise ValueError("targets must be an int32 CUDA tensor [B]")
        logp = torch.empty(B, dtype=torch.float32, device=h.device) if out is None else out
        detlm_head_logprob(self.handle, h.data_ptr(), targets.data_ptr(), B, logp.data_ptr(),
                           _stream_ptr(stream))
        return logp

    def greedy_gated(self, h, tau: float = 0.001, with_logits: bool = False, stream=None):
        """Margin-gated greedy call. Returns (token, gap, logits or None,
        base_token, margin)."""
        import torch
        self._check_h(h)
        B = int(h.shape[0])
        token = torch.empty(B, dtype=torch.int32, device=h.device)
        gap = torch.empty(B, dtype=torch.float32, device=h.device)
        base = torch.empty(B, dtype=torch.int32, device=h.device)
        margin = torch.empty(B, dtype=torch.float32, device=h.device)
        logits = (torch.empty((B, self.V), dtype=torch.float32, device=h.device)
                  if with_logits else None)
        detlm_head_greedy_gated(self.handle, h.data_ptr(), B, float(tau), token.data_ptr(),
                                gap.data_ptr(), logits.data_ptr() if logits is not None else None,
                                base.data_ptr(), margin.data_ptr(), _stream_ptr(stream))
        return token, gap, logits, base, margin

    def sample(self, h, temperature, seeds, positions, with_logits: bool = False, stream=None):
        """Seeded sampling. seeds, positions: int64/uint64 CUDA tensors [B]
        (read as unsigned 64-bit). Returns (token, score_gap, logits or None)."""
        import torch
        self._check_h(h)
        B = int(h.shape[0])
        for name, t in (("seeds", seeds), ("positions", positions)):
            if (not t.is_cuda or t.dim() != 1 or int(t.shape[0]) != B
                    or t.element_size() != 8 or t.is_floating_point()):
                raise ValueError(f"{name} must be a 64-bit integer CUDA tensor [B]")
        token = torch.empty(B, dtype=torch.int32, device=h.device)
        gap = torch.empty(B, dtype=torch.float32, device=h.device)
        logits = (torch.empty((B, self.V), dtype=torch.float32, device=h.device)
                  if with_logits else None)
        detlm_head_sample(self.handle, h.data_ptr(), B, float(temperature),
                          seeds.contiguous().data_ptr(), positions.contiguous().data_ptr(),
                          token.data_ptr(), gap.data_ptr(),
                          logits.data_ptr() if logits is not None else None, _stream_ptr(stream))
        return token, gap, logits

    def greedy_from_float(self, x, with_logits: bool = False, stream=None):
        """int8 head fed by float rows x [B, d] (bf16, fp16 or fp32 CUDA
        tensor). Returns (token, gap, logits or None, mult, shift)."""
        import torch
        if self.dtype != "int8":
            raise DetlmError(DETLM_EUNSUPPORTED, "greedy_from_float")
        xd = _float_dtype_code(x)
        if not x.is_cuda or not x.is_contiguous() or x.dim() != 2 or x.shape[1] != self.d:
            raise ValueError(f"x must be a contiguous CUDA tensor [B, {self.d}]")
        B = int(x.shape[0])
        token = torch.empty(B, dtype=torch.int32, device=x.device)
        gap = torch.empty(B, dtype=torch.int32, device=x.device)
        mult = torch.empty(B, dtype=torch.int32, device=x.device)
        shift = torch.empty(B, dtype=torch.int32, device=x.device)
        logits = (torch.empty((B, self.V), dtype=torch.int32, device=x.device)
                  if with_logits else None)
        detlm_head_greedy_from_float(self.handle, x.data_ptr(), xd, B, token.data_ptr(),
                                     gap.data_ptr(),
                                     logits.data_ptr() if logits is not None else None,
                                     mult.data_ptr(), shift.data_ptr(), _stream_ptr(stream))
        return token, gap, logits, mult, shift

    def verify(self, h, drafts, with_logits: bool = False, stream=None):
        """Greedy speculative verify. h [R*P, d] request-major, drafts int32
        [R, P]. Returns (token [R*P], gap, logits or None, accepted [R])."""
        import torch
        self._check_h(h)
        if drafts.dtype != torch.int32 or not drafts.is_cuda or drafts.dim() != 2:
            raise ValueError("drafts must be an int32 CUDA tensor [R, P]")
        R, P = int(drafts.shape[0]), int(drafts.shape[1])
        if R * P != int(h.shape[0]):
            raise ValueError("h must hold R * P rows")
        gdt = torch.int32 if self.dtype == "int8" else torch.float32
        token = torch.empty(R * P, dtype=torch.int32, device=h.device)
        gap = torch.empty(R * P, dtype=gdt, device=h.device)
        logits = torch.empty((R * P, self.V), dtype=gdt, device=h.device) if with_logits else None
        accepted = torch.empty(R, dtype=torch.int32, device=h.device)
        detlm_head_verify(self.handle, h.data_ptr(), R, P, drafts.contiguous().data_ptr(),
                          token.data_ptr(), gap.data_ptr(),
                          logits.data_ptr() if logits is not None else None,
                          accepted.data_ptr(), _stream_ptr(stream))
        return token, gap, logits, accepted

    def check(self, stream=None) -> int:
        return detlm_head_check(self.handle, _stream_ptr(stream))

    def tiles(self, B: int):
        return detlm_head_tiles(self.handle, B)


# ---- vocabulary-parallel heads -------------------------------------------

SHARD_REC_INT32S = 4     # one detlm_shard_rec_t = 16 bytes = 4 int32 words


class ShardHead(Head):
    """Shard `rank` of P of a head split by vocabulary rows. W_shard holds the
    rows detlm_shard_range(V, P, rank) of the full weight (V rows in all)."""

    def __init__(self, W_shard, V: int, P: int, rank: int, dtype: str | None = None):
        import torch
        if dtype is None:
            dtype = {torch.bfloat16: "bf16", torch.float16: "fp16",
                     torch.int8: "int8"}[W_shard.dtype]
        if not W_shard.is_cuda or not W_shard.is_contiguous() or W_shard.dim() != 2:
            raise ValueError("W_shard must be a contiguous 2-D CUDA tensor")
        v0, v1 = detlm_shard_range(V, P, rank)
        if int(W_shard.shape[0]) != v1 - v0:
            raise ValueError(f"shard {rank} of {P} holds rows [{v0}, {v1})")
        self.W = W_shard
        self.dtype = dtype
        self.V, self.d = int(W_shard.shape[0]), int(W_shard.shape[1])
        self.V_total, self.P, self.rank, self.v_begin, self.v_end = V, P, rank, v0, v1
        self.handle = detlm_head_create_shard(W_shard.data_ptr(), V, self.d, DTYPES[dtype], P, rank)

    def greedy_records(self, h, with_logits: bool = False, stream=None):
        """Records int32 [B, 4] (detlm_shard_rec_t) and the shard's logits or None."""
        import torch
        self._check_h(h)
        B = int(h.shape[0])
        rec = torch.empty((B, SHARD_REC_INT32S), dtype=torch.int32, device=h.device)
        gdt = torch.int32 if self.dtype == "int8" else torch.float32
        logits = torch.empty((B, self.V), dtype=gdt, device=h.device) if with_logits else None
        detlm_head_greedy_shard(self.handle, h.data_ptr(), B, rec.data_ptr(),
                                logits.data_ptr() if logits is not None else None,
                                _stream_ptr(stream))
        return rec, logits

    def logprob_records(self, h, targets, stream=None):
        import torch
        self._check_h(h)
        B = int(h.shape[0])
        if targets.dtype != torch.int32 or not targets.is_cuda or targets.numel() != B:
            raise ValueError("targets must be an int32 CUDA tensor [B]")
        rec = torch.empty((B, SHARD_REC_INT32S), dtype=torch.int32, device=h.device)
        detlm_head_logprob_shard(self.handle, h.data_ptr(), targets.data_ptr(), B, rec.data_ptr(),
                                 _stream_ptr(stream))
        return rec


def merge_greedy(recs, dtype: str, stream=None):
    """recs int32 [P, B, 4] (shard-major) -> (token int32 [B], gap [B])."""
    import torch
    if recs.dtype != torch.int32 or recs.dim() != 3 or recs.shape[2] != SHARD_REC_INT32S:
        raise ValueError("recs must be an int32 tensor [P, B, 4]")
    recs = recs.contiguous()
    P, B = int(recs.shape[0]), int(recs.shape[1])
    token = torch.empty(B, dtype=torch.int32, device=recs.device)
    gap = torch.empty(B, dtype=torch.int32 if dtype == "int8" else torch.float32,
                      device=recs.device)
    detlm_merge_greedy_shards(recs.data_ptr(), P, B, DTYPES[dtype], token.data_ptr(),
                              gap.data_ptr(), _stream_ptr(stream))
    return token, gap


def merge_logprob(recs, V: int, targets, err=None, stream=None):
    """recs int32 [P, B, 4] -> logp float32 [B]."""
    import torch
    if recs.dtype != torch.int32 or recs.dim() != 3 or recs.shape[2] != SHARD_REC_INT32S:
        raise ValueError("recs must be an int32 tensor [P, B, 4]")
    recs = recs.contiguous()
    P, B = int(recs.shape[0]), int(recs.shape[1])
    logp = torch.empty(B, dtype=torch.float32, device=recs.device)
    detlm_merge_logprob_shards(recs.data_ptr(), P, B, V, targets.data_ptr(), logp.data_ptr(),
                               err.data_ptr() if err is not None else None, _stream_ptr(stream))
    return logp


def gather_records(rec, group=None):
    """All-gather one rank's records [B, 4] into [P, B, 4] in rank order (the
    layout the merge calls read). torch.distributed provides the collective
    (NCCL between GPUs, gloo on CPU tensors)."""
    import torch
    import torch.distributed as dist
    P = dist.get_world_size(group)
    B = int(rec.shape[0])
    out = torch.empty((P * B,) + tuple(rec.shape[1:]), dtype=rec.dtype, device=rec.device)
    dist.all_gather_into_tensor(out, rec.contiguous(), group=group)
    return out.view((P, B) + tuple(rec.shape[1:]))


class VocabParallelHead:
    """The output head split by vocabulary over the ranks of a process group:
    rank r holds W rows detlm_shard_range(V, P, r). A call runs this rank's
    shard, all-gathers one 16-byte record per hidden row and merges them, so
    every rank returns the single-device head's outputs bit for bit."""

    def __init__(self, W_shard, V: int, group=None, dtype: str | None = None):
        import torch.distributed as dist
        self.group = group
        P, r = dist.get_world_size(group), dist.get_rank(group)
        self.shard = ShardHead(W_shard, V, P, r, dtype)

    def greedy(self, h, stream=None):
        rec, _ = self.shard.greedy_records(h, stream=stream)
        return merge_greedy(gather_records(rec, self.group), self.shard.dtype, stream=stream)

    def logprob(self, h, targets, stream=None):
        rec = self.shard.logprob_records(h, targets, stream=stream)
        return merge_logprob(gather_records(rec, self.group), self.shard.V_total, targets,
                             stream=stream)

    def close(self):
        self.shard.close()
