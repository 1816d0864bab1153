"""CPU oracle of the output head -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the output head
computes, used to check the CUDA library. Only the tests, the smoke check and
the benchmark's CPU-baseline leg may import it; the library never does, and
the library shares no code with it (only the seeded generators in ``synth``
serve both sides).

Everything is computed exactly or in float64 with numpy:

* float heads: inputs decoded exactly from their bf16 / fp16 bit patterns to
  float64; logits by a float64 matrix product; the per-entry error base
  ``A = |h|·|W|ᵀ`` for the tolerance ``1e-6·A``;
* the integer head: exact int64 matrix product (every partial sum is far
  below 2^63), cross-checked on samples with Python big-integer dots; for
  large row counts the same exact integers through a float64 product (every
  partial sum is an integer below 2^53);
* greedy token (lowest index among the maxima), runner-up value of the
  multiset, top-2 gap in bf16 ulps of the winning logit, logsumexp and the
  log-probability of a target;
* the accepted draft length of greedy speculative verification;
* the margin-gated decision: rounding of the logits to bf16 / fp16, the
  rounded head's token and top-two margin, the gate and the gated token;
* seeded Gumbel-max sampling: the Philox4x32-10 generator, the uniform and
  Gumbel transforms and the sampled token;
* the integer front end: per-row int8 quantization of float rows with a
  dyadic multiplier M / 2^S.

Parity pins: every function here is pinned by tests that do not re-use its
own formula (hand-worked tiny cases, brute force with exact rationals,
closed forms, invariants, and planted-mistake checks). Nothing is marked
"parity unpinned".
"""
from .head import (  # noqa: F401
    decode_bf16, decode_fp16, decode_fp32, decode_int8, decode,
    logits_float, logits_int, logits_int_f64, bigint_dot,
    ulp_bf16, top2, greedy, greedy_int, gap_from_top2_f32,
    logsumexp, logprob,
    head_greedy, head_logprob, verify_accept,
    round_to_format, gated_greedy,
    philox4x32_10, uniform_from_word, gumbel_rows, gumbel_noise, sample,
    quantize_rows,
)
