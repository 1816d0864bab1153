// rows_kernels.cuh -- the log-prob projection, with the hidden rows on the
// tensor core's M axis, on CTA pairs.
//
// Kernel 1b (head_rows_kernel): the same logits as head_gemm_kernel -- the
// same K chunks, the same fp32 round-to-nearest fold of the chunk sums --
// with the roles of the operands exchanged: a unit is 256 hidden rows (the
// MMA's M axis) x 256 vocabulary entries (N), computed by a cluster of two
// CTAs with tcgen05.mma.cta_group::2. Each CTA of the pair loads its own 128
// hidden rows and its own half of the unit's 256 W rows (rank 0 the first
// 128, rank 1 the second) -- 32 KB per 64-element K step instead of the
// 48 KB that one CTA computing 128 x 256 alone would load -- and finds its
// 128 rows x 256 columns of the product in its own tensor memory. The
// tensor core's result for one output element does not depend on which
// operand is A or on its position in the tile (checked bit for bit on GB300
// with standalone probes), so a row's logits are the same bits as in
// head_gemm_kernel.
//
// The epilogue is where the layout pays: a thread holds 128 logits of its own
// row, so the log-sum-exp record is a thread-local fold over registers. The
// record is per (row, 256-entry vocabulary tile): each 128-entry half takes
// its exact maximum m, then adds exp(z - m), evaluated as
// 2^(fma(z, log2 e, -m log2 e)), in ascending vocabulary order; the two
// halves merge in a fixed order. The log-prob call uses this kernel
// for every B, so the rounding tree never depends on B.
//
// Synchronisation of the pair. Rank 0 (the leader) issues every MMA. Both
// producers' TMA loads complete on the leader's full barrier of the stage
// (the leader arms it for the whole 64 KB); the MMA's commit arrives on the
// stage's empty barrier in both CTAs, so each producer refills its own half
// only after the pair's MMAs have read it. A chunk's accumulator slot is
// signalled full in both CTAs (multicast commit) and handed back when the
// eight epilogue warps of both CTAs have arrived on the leader's
// slot-empty barrier (the peer's arrivals are remote, with the arrive's
// default semantics). Every wait is bounded; a cluster barrier before the
// tensor memory is freed keeps either CTA from leaving while the leader's
// MMAs may still touch its memory.
//
// Warp roles (384 threads per CTA): warp 0 TMA producer, warp 1 MMA issuer
// (leader) and tensor-memory allocation (both), warps 2..3 idle (warpgroup
// 0 runs with 40 registers), warps 4..11 the epilogue (two warps per TMEM
// lane quarter, 128 vocabulary columns each, 232 registers).
#pragma once
#include "head_kernels.cuh"

namespace detlm {

constexpr int kRowsM = 256;       // hidden rows per unit (MMA M over the pair)
constexpr int kRowsN = 256;       // vocabulary entries per unit (MMA N)
constexpr int kRowsHalf = 128;    // rows of h and of W that one CTA loads
constexpr int kRowsThreads = 384;
constexpr int kRowsMaxStages = 7;
constexpr uint64_t kPairSettleNs = 1000000;   // abort: let a peer's loads land
constexpr float kLog2e = 1.4426950408889634f;

struct RowsLayout {
  uint32_t a_bytes, b_bytes, stage_bytes, ctrl_off, red_off, total;
};

// Stage s: this CTA's hidden-row box [128 rows x 128 B] then its W box
// [128 rows x 128 B], both 128-byte swizzled; then the barriers and the
// half-row records.
__host__ __device__ inline RowsLayout rows_layout(int stages) {
  RowsLayout L;
  L.a_bytes = kRowsHalf * kRowBytes;
  L.b_bytes = kRowsHalf * kRowBytes;
  L.stage_bytes = L.a_bytes + L.b_bytes;
  L.ctrl_off = static_cast<uint32_t>(stages) * L.stage_bytes;
  // full[S], empty[S], slot_full[2], slot_empty[2], never, drain; then the
  // TMEM address holder and the abort flag
  L.red_off = L.ctrl_off + (2u * stages + 6u) * 8u + 16u;
  L.total = L.red_off + 2u * kRowsHalf * 4u;          // [2][128] words
  return L;
}

__global__ void __launch_bounds__(kRowsThreads, 1)
head_rows_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                 const HeadParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  const RowsLayout L = rows_layout(S);
  const uint32_t rank = cluster_rank();            // 0: leader, 1: peer
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int n_pairs = static_cast<int>(gridDim.x >> 1);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.ctrl_off);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t never_bar = bar0 + 8u * (2 * S + 4);
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 5);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.ctrl_off + (2 * S + 6) * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  uint32_t* red = reinterpret_cast<uint32_t*>(smem + L.red_off);      // [2][128]
  const uint32_t smem_base = smem_u32(smem);
  auto sA = [&](int s) { return smem_base + static_cast<uint32_t>(s) * L.stage_bytes; };
  auto sB = [&](int s) { return sA(s) + L.a_bytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);       // the leader's arrival (+ 64 KB of both CTAs' loads)
      mbar_init(empty_bar(s), 1);      // the leader's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);       // the leader's MMA commit
      mbar_init(acce_bar(b), 16);      // eight epilogue warps of each CTA
    }
    mbar_init(never_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmH);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), 512u);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised before any load or arrival of the
  // other CTA can reach them
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int n_units = p.n_vt * p.n_nt;
  const int kElems = kRowBytes / 2;     // 16-bit elements per 128-byte box row
  const int spu = p.nk;                 // one K box per stage
  const int half = static_cast<int>(rank) * kRowsHalf;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsWg0Wide));
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      const bool leader = rank == 0;
      // W is read-only for the head's life: the W boxes of the first S
      // stages are requested before waiting for the previous kernels on the
      // stream; the hidden rows (which a previous kernel may write) after.
      const int n_my = (n_units - pair + n_pairs - 1) / n_pairs;
      const int pre = min(S, n_my > 0 ? n_my * spu : 0);
      for (int j = 0; j < pre; ++j) {
        const int u = pair + (j / spu) * n_pairs;
        const int vt = u / p.n_nt, kb = j - (j / spu) * spu;
        if (leader) mbar_expect_tx(full_bar(j), 2u * L.stage_bytes);
        tma_load_2d_pair(sB(j), &tmW, kb * kElems, vt * kRowsN + half,
                         cluster_addr(full_bar(j), 0), pol_w);
      }
      grid_dep_wait();
      uint32_t stage = 0, phase = 0, outstanding = 0, out_par = 0;
      bool ok = true;
      int j = 0;
      for (int u = pair; u < n_units && ok; u += n_pairs) {
        const int vt = u / p.n_nt, rt = u - (u / p.n_nt) * p.n_nt;
        for (int kb = 0; kb < spu; ++kb, ++j) {
          const uint32_t fb = cluster_addr(full_bar(stage), 0);
          if (j < pre) {
            tma_load_2d_pair(sA(stage), &tmH, kb * kElems, rt * kRowsM + half, fb, pol_h);
            if (leader) mbar_arrive(full_bar(stage));
          } else {
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
            if (leader) mbar_arrive_expect_tx(full_bar(stage), 2u * L.stage_bytes);
            tma_load_2d_pair(sB(stage), &tmW, kb * kElems, vt * kRowsN + half, fb, pol_w);
            tma_load_2d_pair(sA(stage), &tmH, kb * kElems, rt * kRowsM + half, fb, pol_h);
          }
          outstanding |= 1u << stage;
          out_par = (out_par & ~(1u << stage)) | (phase << stage);
          if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, ERR_TIMEOUT);
        if (leader) {
          // the armed stages complete once both CTAs' loads have landed
          const int zero = 0;
          for (int s = 0; s < S; ++s)
            if ((outstanding >> s) & 1u) mbar_wait(full_bar(s), (out_par >> s) & 1u, &zero, p.timeout_ns);
        } else {
          // the peer's loads complete on the leader's barriers: give the
          // ones in flight time to land before this CTA may leave
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < kPairSettleNs) __nanosleep(1000);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsWg0Wide));
    if (lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0, slot = 0, sph = 0;
      bool ok = true;
      if (p.stall) ok = mbar_wait(never_bar, 0, abort_flag, p.timeout_ns);
      for (int u = pair; u < n_units && ok; u += n_pairs) {
        for (int c = 0; c < p.n_chunks && ok; ++c) {
          if (!mbar_wait(acce_bar(slot), sph ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + slot * static_cast<uint32_t>(kRowsN);
#pragma unroll
          for (int sc = 0; sc < kBlocksPerChunk; ++sc) {
            const int kb = c * kBlocksPerChunk + sc;
            if (kb >= p.nk) break;
            if (!mbar_wait(full_bar(stage), phase, abort_flag, p.timeout_ns)) { ok = false; break; }
            tc_fence_after();
            const uint64_t da = sdesc_sw128(sA(stage));
            const uint64_t db = sdesc_sw128(sB(stage));
#pragma unroll
            for (int k = 0; k < 4; ++k)   // K = 16 per MMA: 32 bytes = 2 descriptor units
              mma_f16_pair(d_tmem, da + 2u * k, db + 2u * k, p.idesc, !(sc == 0 && k == 0));
            mma_commit_pair(empty_bar(stage), 3);
            if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          mma_commit_pair(accf_bar(slot), 3);
          if (++slot == 2u) { slot = 0; sph ^= 1u; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, ERR_TIMEOUT);
      }
      mma_commit_pair(drain_bar, 1);
      const int zero = 0;
      mbar_wait(drain_bar, 0, &zero, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < 4) {
    // warps 2 and 3: no role, fewer registers
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsWg0Wide));
  } else {
    // --------------------------------------------------------- epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kRegsEpiWide));
    grid_dep_wait();          // outputs and records: only after the previous kernels
    const int q = warp & 3;                    // TMEM lane quarter
    const int g = (warp - 4) >> 2;             // vocabulary half of the unit
    const int r = q * 32 + lane;               // hidden row within this CTA's half
    const uint32_t tlane = static_cast<uint32_t>(q * 32) << 16;
    uint32_t slot = 0, sph = 0;
    bool failed = false;
    for (int u = pair; u < n_units; u += n_pairs) {
      const int vt = u / p.n_nt, rt = u - (u / p.n_nt) * p.n_nt;
      const int n = rt * kRowsM + half + r;
      const bool row_ok = n < p.B;
      const bool warp_rows = rt * kRowsM + half + q * 32 < p.B;   // any valid row in this warp
      float acc[8][16];
      for (int c = 0; c < p.n_chunks; ++c) {
        const uint32_t cur = slot, cph = sph;
        if (++slot == 2u) { slot = 0; sph ^= 1u; }
        if (!failed && !mbar_wait(accf_bar(cur), cph, abort_flag, p.timeout_ns)) {
          failed = true;
          *abort_flag = 1;
        }
        if (failed) continue;
        tc_fence_after();
        if (warp_rows) {
          const uint32_t sbase = tmem_base + tlane + cur * static_cast<uint32_t>(kRowsN) +
                                 static_cast<uint32_t>(g * 128);
          // two groups of two 32-column loads, one wait each (a wait per
          // load left the drain latency-bound)
#pragma unroll
          for (int h4 = 0; h4 < 2; ++h4) {
            uint32_t rw[2][32];
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2) tmem_ld32(sbase + (h4 * 2 + b2) * 32, rw[b2]);
            tmem_wait_ld();
#pragma unroll
            for (int b4 = 0; b4 < 4; ++b4) {
              const int bb = h4 * 4 + b4;
              const uint32_t* rr = &rw[b4 >> 1][(b4 & 1) * 16];   // this block's 16 columns
              if (c == 0) {
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[bb][i] = __uint_as_float(rr[i]);
              } else {
#pragma unroll
                for (int i = 0; i < 16; i += 2)
                  add2_rn(acc[bb][i], acc[bb][i + 1], __uint_as_float(rr[i]),
                          __uint_as_float(rr[i + 1]));
              }
            }
          }
        }
        tc_fence_before();   // slot fully read: hand it back to the leader's MMA warp
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(acce_bar(cur));
          else mbar_arrive_remote(cluster_addr(acce_bar(cur), 0));
        }
      }
      if (epi_bar_or<256>(failed || *abort_flag)) {
        if (threadIdx.x == 128) { *abort_flag = 1; atomicOr(p.err, ERR_TIMEOUT); }
        break;
      }
      const int vb = vt * kRowsN + g * 128;      // first vocabulary entry of this half
      // ---- the half-row record: (max, sum exp(z - max)) in ascending v
      Lse ls{-INFINITY, 0.0f};
      if (row_ok) {
        // the target's logit, if it lies in this half: a select chain over
        // the 16-entry blocks, then over the block (no register is indexed
        // at run time); targets are vocabulary indices of the whole head,
        // this head's rows start at v_off
        const int tl = p.targets[n] - p.v_off - vb;
        if (tl >= 0 && tl < 128) {
          const int tb = tl >> 4, ti = tl & 15;
          float sel[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) sel[i] = acc[0][i];
#pragma unroll
          for (int bb = 1; bb < 8; ++bb)
#pragma unroll
            for (int i = 0; i < 16; ++i) sel[i] = bb == tb ? acc[bb][i] : sel[i];
          float z = sel[0];
#pragma unroll
          for (int i = 1; i < 16; ++i) z = i == ti ? sel[i] : z;
          p.zt[n] = z;
        }
        const int nv = min(128, p.V - vb);      // valid entries in this half
        // exp(z - m) = 2^(z log2(e) - m log2(e)): one fma and one ex2 per
        // entry (the rounding of m log2(e) scales the half's whole sum by
        // the same factor, within |m| 2^-24 in the log). The tail is bound
        // by instruction issue, so a full half (every tile but possibly the
        // last) runs without the per-entry bound test.
        float m = -INFINITY, sum = 0.0f;
        if (nv == 128) {
#pragma unroll
          for (int bb = 0; bb < 8; ++bb)
#pragma unroll
            for (int i = 0; i < 16; ++i) m = fmaxf(m, acc[bb][i]);
          const float ml = m * kLog2e;
#pragma unroll
          for (int bb = 0; bb < 8; ++bb)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              sum = __fadd_rn(sum, exp2_approx(fmaf(acc[bb][i], kLog2e, -ml)));
        } else {
#pragma unroll
          for (int bb = 0; bb < 8; ++bb)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (bb * 16 + i < nv) m = fmaxf(m, acc[bb][i]);
          const float ml = m * kLog2e;
#pragma unroll
          for (int bb = 0; bb < 8; ++bb)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (bb * 16 + i < nv) sum = __fadd_rn(sum, exp2_approx(fmaf(acc[bb][i], kLog2e, -ml)));
        }
        ls = Lse{m, sum};
      }
      // ---- the two halves of a row: the second hands its record to the first
      if (g == 1) {
        red[0 * kRowsHalf + r] = __float_as_uint(ls.m);
        red[1 * kRowsHalf + r] = __float_as_uint(ls.S);
      }
      named_bar_sync(1, 256);
      if (g == 0 && row_ok) {
        const size_t o = static_cast<size_t>(n) * p.n_vt + vt;   // records [B][n_vt]
        const Lse other{__uint_as_float(red[0 * kRowsHalf + r]), __uint_as_float(red[1 * kRowsHalf + r])};
        const Lse tot = lse_merge(ls, other);
        p.rec_m[o] = tot.m;
        p.rec_s[o] = tot.S;
      }
      named_bar_sync(1, 256);
    }
    if (failed && threadIdx.x == 128) atomicOr(p.err, ERR_TIMEOUT);
  }

  // neither CTA leaves (or frees its tensor memory) before the leader's MMAs
  // and both CTAs' remote arrivals are done
  tc_fence_before();
  cluster_sync();
  // the merge kernel may be scheduled now (at the end: waiting merge blocks
  // would share the SMs' issue slots with this kernel for its whole run)
  grid_dep_launch();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512u);
  }
}

}  // namespace detlm
