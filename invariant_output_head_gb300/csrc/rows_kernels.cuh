// rows_kernels.cuh -- the log-prob projection, with the hidden rows on the
// tensor core's M axis.
//
// Kernel 1b (head_rows_kernel): the same logits as head_gemm_kernel -- the
// same K chunks, the same fp32 round-to-nearest fold of the chunk sums --
// with the roles of the operands exchanged: a unit is 128 hidden rows (the
// MMA's M axis and TMEM lanes) x 256 vocabulary entries (N). The tensor
// core's result for one output element does not depend on which operand is
// A or on its position in the tile (checked bit for bit on GB300 with a
// standalone probe and against the swap-AB kernel over several shapes), so a
// row's logits are the same bits as in head_gemm_kernel. What changes is the
// epilogue: a thread holds 128 logits of its own row, so the log-sum-exp
// record is a thread-local fold over registers instead of a transpose across
// lanes, and the MMA no longer waits for a long end-of-tile reduction (the
// trainer's 8192-row call: 4.31 -> 3.11 ms on GB300).
//
// The record is per (row, 256-entry vocabulary tile): each 128-entry half
// takes its exact maximum, then adds exp(z - max) in ascending vocabulary
// order; the two halves merge in a fixed order. The log-prob call uses this
// kernel for every B, so the rounding tree never depends on B. (For the
// greedy calls the swap-AB kernel stays faster: at B = 256 one of its units
// covers every row, while here each W tile would be read once per 128 rows,
// and its stores of fp32 logits are coalesced along the vocabulary.)
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer, warps
// 2..3 idle (warpgroup 0 runs with 40 registers), warps 4..11 the epilogue
// (two warps per TMEM lane quarter, 128 vocabulary columns each, 232
// registers).
#pragma once
#include "head_kernels.cuh"

namespace detlm {

constexpr int kRowsM = 128;       // hidden rows per unit (MMA M)
constexpr int kRowsN = 256;       // vocabulary entries per unit (MMA N)
constexpr int kRowsThreads = 384;
constexpr int kRowsMaxStages = 6;
constexpr int kRowsScratch = 32 * 17;   // words per epilogue warp (one 16-column block)

struct RowsLayout {
  uint32_t a_bytes, b_bytes, stage_bytes, ctrl_off, red_off, scr_off, total;
};

// Stage s: the hidden-row box [128 rows x 128 B] then the W box [256 x 128 B],
// both 128-byte swizzled; then the barriers, the half-row records and the
// epilogue warps' scratch.
__host__ __device__ inline RowsLayout rows_layout(int stages) {
  RowsLayout L;
  L.a_bytes = kRowsM * kRowBytes;
  L.b_bytes = kRowsN * kRowBytes;
  L.stage_bytes = L.a_bytes + L.b_bytes;
  L.ctrl_off = static_cast<uint32_t>(stages) * L.stage_bytes;
  // full[S], empty[S], slot_full[2], slot_empty[2], never, drain; then the
  // TMEM address holder and the abort flag
  L.red_off = L.ctrl_off + (2u * stages + 6u) * 8u + 16u;
  L.scr_off = L.red_off + 4u * kRowsM * 4u;          // [128 rows] x 4 words
  L.total = L.scr_off + 8u * kRowsScratch * 4u;
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
  uint32_t* red = reinterpret_cast<uint32_t*>(smem + L.red_off);      // [2][128] used
  float* scratch = reinterpret_cast<float*>(smem + L.scr_off);
  const uint32_t smem_base = smem_u32(smem);
  auto sA = [&](int s) { return smem_base + static_cast<uint32_t>(s) * L.stage_bytes; };
  auto sB = [&](int s) { return sA(s) + L.a_bytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 8);
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
    tmem_alloc(smem_u32(tmem_holder), 512u);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int n_units = p.n_vt * p.n_nt;
  const int kElems = kRowBytes / 2;     // 16-bit elements per 128-byte box row
  const int spu = p.nk;                 // one K box per stage

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsWg0Wide));
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      // W is read-only for the head's life: the W boxes of the first S
      // stages are requested before waiting for the previous kernels on the
      // stream; the hidden rows (which a previous kernel may write) after.
      const int n_my = (n_units - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                       static_cast<int>(gridDim.x);
      const int pre = min(S, n_my > 0 ? n_my * spu : 0);
      for (int j = 0; j < pre; ++j) {
        const int u = blockIdx.x + (j / spu) * gridDim.x;
        const int vt = u / p.n_nt, kb = j - (j / spu) * spu;
        mbar_expect_tx(full_bar(j), L.stage_bytes);
        tma_load_2d(sB(j), &tmW, kb * kElems, vt * kRowsN, full_bar(j), pol_w);
      }
      grid_dep_wait();
      uint32_t stage = 0, phase = 0, outstanding = 0, out_par = 0;
      bool ok = true;
      int j = 0;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const int vt = u / p.n_nt, rt = u - (u / p.n_nt) * p.n_nt;
        for (int kb = 0; kb < spu; ++kb, ++j) {
          if (j < pre) {
            tma_load_2d(sA(stage), &tmH, kb * kElems, rt * kRowsM, full_bar(stage), pol_h);
            mbar_arrive(full_bar(stage));
          } else {
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
            mbar_arrive_expect_tx(full_bar(stage), L.stage_bytes);
            tma_load_2d(sB(stage), &tmW, kb * kElems, vt * kRowsN, full_bar(stage), pol_w);
            tma_load_2d(sA(stage), &tmH, kb * kElems, rt * kRowsM, full_bar(stage), pol_h);
          }
          outstanding |= 1u << stage;
          out_par = (out_par & ~(1u << stage)) | (phase << stage);
          if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, ERR_TIMEOUT);
        const int zero = 0;
        for (int s = 0; s < S; ++s)
          if ((outstanding >> s) & 1u) mbar_wait(full_bar(s), (out_par >> s) & 1u, &zero, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsWg0Wide));
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, slot = 0, sph = 0;
      bool ok = true;
      if (p.stall) ok = mbar_wait(never_bar, 0, abort_flag, p.timeout_ns);
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
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
              mma_f16(d_tmem, da + 2u * k, db + 2u * k, p.idesc, !(sc == 0 && k == 0));
            mma_commit(empty_bar(stage));
            if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          mma_commit(accf_bar(slot));
          if (++slot == 2u) { slot = 0; sph ^= 1u; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, ERR_TIMEOUT);
      }
      mma_commit(drain_bar);
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
    const int r = q * 32 + lane;               // hidden row within the unit
    const uint32_t tlane = static_cast<uint32_t>(q * 32) << 16;
    float* scr = scratch + (warp - 4) * kRowsScratch;
    uint32_t slot = 0, sph = 0;
    bool failed = false;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const int vt = u / p.n_nt, rt = u - (u / p.n_nt) * p.n_nt;
      const int n = rt * kRowsM + r;
      const bool row_ok = n < p.B;
      const bool warp_rows = rt * kRowsM + q * 32 < p.B;   // any valid row in this warp
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
#pragma unroll
          for (int bb = 0; bb < 8; ++bb) {
            uint32_t rr[16];
            tmem_ld16(sbase + bb * 16, rr);
            tmem_wait_ld();
            if (c == 0) {
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[bb][i] = __uint_as_float(rr[i]);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[bb][i] = __fadd_rn(acc[bb][i], __uint_as_float(rr[i]));
            }
          }
        }
        tc_fence_before();   // slot fully read: hand it back to the MMA warp
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(cur));
      }
      if (epi_bar_or<256>(failed || *abort_flag)) {
        if (threadIdx.x == 128) { *abort_flag = 1; atomicOr(p.err, ERR_TIMEOUT); }
        break;
      }
      const int vb = vt * kRowsN + g * 128;      // first vocabulary entry of this half
      // ---- the half-row record: (max, sum exp(z - max)) in ascending v
      Lse ls{-INFINITY, 0.0f};
      if (row_ok) {
        // the target's logit, if it lies in this half (its 16-entry block
        // through the lane's scratch row: no register indexed at run time)
        const int tl = p.targets[n] - vb;
        if (tl >= 0 && tl < 128) {
          const int tb = tl >> 4;
          float sel[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) sel[i] = acc[0][i];
#pragma unroll
          for (int bb = 1; bb < 8; ++bb)
#pragma unroll
            for (int i = 0; i < 16; ++i) sel[i] = bb == tb ? acc[bb][i] : sel[i];
#pragma unroll
          for (int i = 0; i < 16; ++i) scr[lane * 17 + i] = sel[i];
          p.zt[n] = scr[lane * 17 + (tl & 15)];
        }
        const int nv = min(128, p.V - vb);      // valid entries in this half
        float m = -INFINITY;
#pragma unroll
        for (int bb = 0; bb < 8; ++bb)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (bb * 16 + i < nv) m = fmaxf(m, acc[bb][i]);
        float sum = 0.0f;
#pragma unroll
        for (int bb = 0; bb < 8; ++bb)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (bb * 16 + i < nv) sum = __fadd_rn(sum, __expf(acc[bb][i] - m));
        ls = Lse{m, sum};
      }
      // ---- the two halves of a row: the second hands its record to the first
      if (g == 1) {
        red[0 * kRowsM + r] = __float_as_uint(ls.m);
        red[1 * kRowsM + r] = __float_as_uint(ls.S);
      }
      named_bar_sync(1, 256);
      if (g == 0 && row_ok) {
        const size_t o = static_cast<size_t>(n) * p.n_vt + vt;   // records [B][n_vt]
        const Lse other{__uint_as_float(red[0 * kRowsM + r]), __uint_as_float(red[1 * kRowsM + r])};
        const Lse tot = lse_merge(ls, other);
        p.rec_m[o] = tot.m;
        p.rec_s[o] = tot.S;
      }
      named_bar_sync(1, 256);
    }
    if (failed && threadIdx.x == 128) atomicOr(p.err, ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  // the merge kernel may be scheduled now (at the end: waiting merge blocks
  // would share the SMs' issue slots with this kernel for its whole run)
  grid_dep_launch();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512u);
  }
}

}  // namespace detlm
