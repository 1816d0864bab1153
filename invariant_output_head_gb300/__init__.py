"""GB300-native batch-invariant LLM output head (lm_head).

The CUDA library (``_lib/libdetlm_head.so``, C ABI in ``include/detlm_head.h``)
computes logits = h . W^T on sm_103a tensor cores and fuses the greedy
decision (lowest-index argmax, top-2 gap in bf16 ulps), the target
log-probability, the margin-gated decision, seeded sampling or speculative
verification, bit-identical for a row whatever the batch size; an integer
front end quantizes float rows for the exact int8 head. This package is the
thin Python binding; see ``binding.Head``.
"""
from .binding import (  # noqa: F401
    Head, DetlmError, load_library, library_path, status_string,
    detlm_head_create, detlm_head_reserve, detlm_head_greedy, detlm_head_logprob,
    detlm_head_greedy_host, detlm_head_logprob_host, detlm_head_check,
    detlm_head_greedy_host_async, detlm_head_logprob_host_async,
    detlm_head_time_next, detlm_head_debug, detlm_head_tiles, detlm_head_destroy,
    detlm_status_string, detlm_greedy_noalloc, detlm_head_verify,
    detlm_head_greedy_gated, detlm_head_sample, detlm_quantize_rows,
    detlm_head_greedy_from_float, quantize_rows,
    detlm_shard_range, detlm_head_create_shard, detlm_head_greedy_shard,
    detlm_head_logprob_shard, detlm_merge_greedy_shards, detlm_merge_logprob_shards,
    ShardHead, VocabParallelHead, merge_greedy, merge_logprob, gather_records,
    DETLM_BF16, DETLM_FP16, DETLM_INT8, DETLM_FP32, DETLM_OK, DETLM_EINVAL, DETLM_EUNSUPPORTED,
    DETLM_ECUDA, DETLM_ETIMEOUT, DETLM_ENOMEM, DETLM_ETARGET, DETLM_DEBUG_STALL,
)
