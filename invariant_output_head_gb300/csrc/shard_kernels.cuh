// shard_kernels.cuh -- the output head split by vocabulary over P shards.
//
// A vocabulary-parallel head holds W's rows [v_begin, v_end) on each of P
// devices (shard r of P; the ranges come from detlm_shard_range). Each shard
// runs the usual projection kernel over its rows -- the same K chunks and
// fold, so the same logits -- and folds its tile records into ONE 16-byte
// record per hidden row (shard_fold_kernel). The P records of a row are then
// all that crosses devices; shard_merge_kernel combines them into the token
// and gap, or the log-probability.
//
// The result is the single-device result bit for bit:
//  * greedy: the record is (max, lowest global index of it, runner-up); the
//    merge rule (value desc, index asc; runner-up = max of the loser's max
//    and both runners-up) is exact, so any grouping gives the same bits;
//  * log-prob: the single-device merge is a balanced tree over 128 leaves,
//    leaf g the contiguous 256-entry tiles [g n / 128, (g + 1) n / 128)
//    (head_kernels.cuh, leaf_lo). Shard r of P (P a power of two up to 128)
//    holds exactly the tiles of leaves [128 r / P, 128 (r + 1) / P), folds
//    them into that subtree's root, and the merge combines the P roots in a
//    balanced tree -- the top levels of the same tree. Subtrees are computed
//    with the leaves in threads 0 .. 128/P - 1 and identity elements
//    elsewhere; lse_merge with the identity returns its other operand bit
//    for bit, so the padding changes nothing. The target's logit is taken
//    from the one shard that holds the target.
//
// This follows "TandemLLM docs, 12 Exactness", 12.2: the reduction order is
// fixed by the weight's shape (here V and P), never by the row count.
#pragma once
#include "head_kernels.cuh"

namespace detlm {

// One row's record of one shard (16 bytes; the C ABI's detlm_shard_rec_t).
//   greedy float: m = max logit, i = lowest global index of it, s = runner-up
//   greedy int8 : the same with m and s holding int32 bit patterns
//   log-prob    : m = max logit, i = 1 if the shard holds the row's target,
//                 s = sum over the shard of exp(z - m), zt = target's logit
struct ShardRec {
  float m;
  int32_t i;
  float s;
  float zt;
};
static_assert(sizeof(ShardRec) == 16, "16-byte shard record");

enum : int { SHARD_GREEDY = 0, SHARD_GREEDY_INT = 1, SHARD_LOGPROB = 2 };

struct ShardFoldParams {
  int32_t B, n_vt;           // rows; this shard's tiles (records [B][n_vt])
  int32_t mode;              // SHARD_*
  int32_t n_tiles;           // log-prob: 256-entry tiles of the whole vocabulary
  int32_t leaf0, n_leaves;   // log-prob: this shard's leaves of the 128-leaf tree
  int32_t t0;                // log-prob: global index of this shard's first tile
  int32_t v_begin, v_end;    // this shard's vocabulary rows
  const float* rec_m;
  const int32_t* rec_i;
  const float* rec_s;
  const float* zt;           // log-prob: [B], valid where the target is here
  const int32_t* targets;    // log-prob: [B] global target ids
  ShardRec* out;             // [B]
};
static_assert(sizeof(ShardFoldParams) <= 128, "kernel parameter struct above 128 bytes");

// One 128-thread block per hidden row: this shard's tile records -> one record.
__global__ void __launch_bounds__(kMergeThreads) shard_fold_kernel(const ShardFoldParams p) {
  grid_dep_launch();
  grid_dep_wait();   // records of the projection kernel are complete and visible
  const int n = blockIdx.x;
  const int g = threadIdx.x;
  const size_t base = static_cast<size_t>(n) * p.n_vt;
  if (p.mode == SHARD_GREEDY) {
    __shared__ Top2 part[4];
    Top2 acc{-INFINITY, INT32_MAX, -INFINITY};
    for (int t = g; t < p.n_vt; t += kMergeThreads)
      acc = top2_merge(acc, Top2{p.rec_m[base + t], p.rec_i[base + t], p.rec_s[base + t]});
    const Top2 tot = block_tree128(acc, top2_merge, part);
    if (g == 0) p.out[n] = ShardRec{tot.m, tot.i, tot.s, 0.0f};
  } else if (p.mode == SHARD_GREEDY_INT) {
    __shared__ ITop2 part[4];
    const int32_t* rm = reinterpret_cast<const int32_t*>(p.rec_m);
    const int32_t* rs = reinterpret_cast<const int32_t*>(p.rec_s);
    ITop2 acc{INT32_MIN, INT32_MAX, INT32_MIN};
    for (int t = g; t < p.n_vt; t += kMergeThreads)
      acc = itop2_merge(acc, ITop2{rm[base + t], p.rec_i[base + t], rs[base + t]});
    const ITop2 tot = block_tree128(acc, itop2_merge, part);
    if (g == 0) p.out[n] = ShardRec{__int_as_float(tot.m), tot.i, __int_as_float(tot.s), 0.0f};
  } else {
    __shared__ Lse part[4];
    Lse acc{-INFINITY, 0.0f};
    if (g < p.n_leaves) {
      const int leaf = p.leaf0 + g;
      acc = lse_fold_range(p.rec_m + base, p.rec_s + base, leaf_lo(leaf, p.n_tiles) - p.t0,
                           leaf_lo(leaf + 1, p.n_tiles) - p.t0);
    }
    const Lse tot = block_tree128(acc, lse_merge, part);
    if (g == 0) {
      const int tg = p.targets[n];
      const bool here = tg >= p.v_begin && tg < p.v_end;
      p.out[n] = ShardRec{tot.m, here ? 1 : 0, tot.S, here ? p.zt[n] : 0.0f};
    }
  }
}

struct ShardMergeParams {
  int32_t P, B, V, mode;     // shards, rows, whole vocabulary, SHARD_*
  const ShardRec* recs;      // [P][B], shard-major (as an all-gather leaves them)
  int32_t* token;            // greedy: [B]
  void* gap;                 // greedy: [B] float (bf16 ulps) or int32 (int8 head)
  const int32_t* targets;    // log-prob: [B]
  float* logp;               // log-prob: [B]
  int* err;                  // log-prob: optional error word (ERR_TARGET)
};
static_assert(sizeof(ShardMergeParams) <= 128, "kernel parameter struct above 128 bytes");

// One 128-thread block per hidden row: the P shard records -> the decision.
// Record k sits in thread k, identity elements in the others, so the block
// tree is a balanced tree over the P records (P a power of two).
__global__ void __launch_bounds__(kMergeThreads) shard_merge_kernel(const ShardMergeParams p) {
  grid_dep_launch();
  grid_dep_wait();
  const int n = blockIdx.x;
  const int k = threadIdx.x;
  if (p.mode == SHARD_GREEDY) {
    __shared__ Top2 part[4];
    Top2 x{-INFINITY, INT32_MAX, -INFINITY};
    if (k < p.P) {
      const ShardRec r = p.recs[static_cast<size_t>(k) * p.B + n];
      x = Top2{r.m, r.i, r.s};
    }
    const Top2 tot = block_tree128(x, top2_merge, part);
    if (k == 0) {
      p.token[n] = tot.i;
      static_cast<float*>(p.gap)[n] = gap_ulp_bf16(tot.m, tot.s);
    }
  } else if (p.mode == SHARD_GREEDY_INT) {
    __shared__ ITop2 part[4];
    ITop2 x{INT32_MIN, INT32_MAX, INT32_MIN};
    if (k < p.P) {
      const ShardRec r = p.recs[static_cast<size_t>(k) * p.B + n];
      x = ITop2{__float_as_int(r.m), r.i, __float_as_int(r.s)};
    }
    const ITop2 tot = block_tree128(x, itop2_merge, part);
    if (k == 0) {
      p.token[n] = tot.i;
      static_cast<int32_t*>(p.gap)[n] = tot.s == INT32_MIN ? INT32_MAX : tot.m - tot.s;
    }
  } else {
    __shared__ Lse part[4];
    __shared__ float zt_sh;
    __shared__ int have_sh;
    if (k == 0) { have_sh = 0; zt_sh = 0.0f; }
    __syncthreads();
    Lse x{-INFINITY, 0.0f};
    if (k < p.P) {
      const ShardRec r = p.recs[static_cast<size_t>(k) * p.B + n];
      x = Lse{r.m, r.s};
      if (r.i == 1) { zt_sh = r.zt; have_sh = 1; }   // at most one shard holds the target
    }
    const Lse tot = block_tree128(x, lse_merge, part);   // its barrier orders zt_sh
    if (k == 0) {
      const int tg = p.targets[n];
      if (tg < 0 || tg >= p.V || !have_sh) {
        p.logp[n] = __int_as_float(0x7fc00000);
        if (p.err != nullptr) atomicOr(p.err, ERR_TARGET);
      } else {
        p.logp[n] = zt_sh - (tot.m + logf(tot.S));
      }
    }
  }
}

}  // namespace detlm
