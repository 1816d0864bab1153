// pair_kernels.cuh -- the wide greedy projection (more than 128 hidden rows)
// on CTA pairs.
//
// Kernel 1c (head_pair_kernel): the same logits as head_gemm_kernel -- the
// same K chunks, the same fp32 round-to-nearest (integer head: int32) fold
// of the chunk sums -- computed by clusters of two CTAs with
// tcgen05.mma.cta_group::2. A unit is 256 vocabulary rows x 256 hidden rows.
// Per 64-element K step each CTA loads 128 hidden rows (its half of the MMA's
// M = 256 operand) and 128 vocabulary rows (its half of the N = 256
// operand): 32 KB of shared memory written per CTA and step instead of the
// 48 KB a one-CTA 128 x 256 unit needs, and the tensor core reads half of the
// N operand from each CTA. On GB300 the one-CTA kernel at N = 256 is bound by
// shared-memory bandwidth (its TMA fill plus the MMA's operand reads run near
// 100 bytes per clock per SM, and the 128 x 256 x 16 MMAs take ~112 ns
// instead of 65), which the pair layout relieves.
//
// Here the hidden rows are the MMA's M axis: tensor-memory lane = hidden row,
// column = vocabulary row. Each epilogue thread therefore owns one hidden row
// and 128 consecutive vocabulary entries (one 128-row tile of W), and folds
// its tile record (max, lowest index, runner-up) in registers, in ascending
// vocabulary order, with no exchange between threads; the per-unit work after
// the last chunk overlaps the MMA filling both accumulator slots with the
// next unit's first chunks. fp32 logits go through per-warp staging buffers
// in shared memory and leave by TMA tensor stores, which run while the warp
// drains the next unit (plain stores of 64-byte row runs where the logits
// are not 16-byte aligned device memory). The tensor core's result for an
// element depends neither on the operand roles nor on the pair mode (checked
// bit for bit on GB300 with standalone probes), so the logits are
// head_gemm_kernel's bit for bit, and the greedy record is exact.
//
// The pair protocol is the log-prob kernel's (rows_kernels.cuh): the leader
// issues every MMA; both producers' loads complete on the leader's stage
// barrier; MMA commits arrive on both CTAs' barriers (multicast); a chunk's
// accumulator slot goes back to the MMA when the epilogue warps of both CTAs
// (eight each) have arrived on the leader's slot-empty barrier. Every wait is
// bounded.
#pragma once
#include "head_kernels.cuh"
#include "rows_kernels.cuh"

namespace detlm {

constexpr int kPairThreads = 384;
constexpr int kPairMaxStages = 7;
constexpr int kPairN = 256;         // hidden rows per unit (the pair's MMA M); also its N
constexpr int kPairWarps = 8;       // epilogue warps 4 .. 11, 128 columns each

// Logits staging: per epilogue warp two buffers of 32 hidden rows x 16
// logits (64-byte rows, 64-byte swizzle: 16-byte chunk c of row r sits at
// chunk c ^ ((r >> 1) & 3), so a warp's row-per-lane writes and the 8-row
// reads below are both free of bank conflicts).
constexpr uint32_t kPairStageBuf = 32 * 16 * 4;
constexpr uint32_t kPairXsBytes = 2 * kPairStageBuf;

struct PairLayout {
  uint32_t a_bytes, b_bytes, stage_bytes, ctrl_off, xs_off, total;
};

// Stage s: this CTA's 128 hidden rows [128 rows x 128 B] (operand A) then its
// 128 vocabulary rows [128 rows x 128 B] (its half of operand B), both
// 128-byte swizzled; then the barriers and the epilogue warps' logits
// staging buffers (1024-byte aligned: the swizzle pattern repeats every 512
// bytes).
__host__ __device__ inline PairLayout pair_layout(int stages) {
  PairLayout L;
  L.a_bytes = kRowsHalf * kRowBytes;
  L.b_bytes = kBM * kRowBytes;
  L.stage_bytes = L.a_bytes + L.b_bytes;
  L.ctrl_off = static_cast<uint32_t>(stages) * L.stage_bytes;
  // full[S], empty[S], slot_full[2], slot_empty[2], never, drain; then the
  // TMEM address holder and the abort flag
  L.xs_off = (L.ctrl_off + (2u * stages + 6u) * 8u + 16u + 1023u) & ~1023u;
  L.total = L.xs_off + kPairWarps * kPairXsBytes;
  return L;
}

// p.n_vt: 128-row vocabulary tiles (the records' tiles); a unit covers tiles
// 2 vp and 2 vp + 1 (the second may lie past V: its rows read as zeros and
// no record of it is written). p.n_nt: 256-row hidden tiles.
template <int MODE>
__global__ void __launch_bounds__(kPairThreads, 1)
head_pair_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                 const __grid_constant__ CUtensorMap tmL, const HeadParams p) {
  static_assert(MODE == MODE_GREEDY || MODE == MODE_INT, "mode");
  constexpr int N = kPairN;
  constexpr int WBLK = 8;                          // 16-column blocks per epilogue warp
  constexpr int ET = 32 * kPairWarps;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  const PairLayout L = pair_layout(S);
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
  uint8_t* xsall = smem + L.xs_off;
  const uint32_t smem_base = smem_u32(smem);
  auto sA = [&](int s) { return smem_base + static_cast<uint32_t>(s) * L.stage_bytes; };
  auto sB = [&](int s) { return sA(s) + L.a_bytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);       // the leader's arrival (+ both CTAs' loads)
      mbar_init(empty_bar(s), 1);      // the leader's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);       // the leader's MMA commit
      mbar_init(acce_bar(b), 2 * kPairWarps);   // eight epilogue warps of each CTA
    }
    mbar_init(never_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmH);
    if (p.tma_logits) tma_prefetch_desc(&tmL);
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
  const int n_vp = (p.n_vt + 1) >> 1;   // 256-row vocabulary units
  const int n_units = n_vp * p.n_nt;
  const int kElems = kRowBytes / 2;     // 16-bit elements per 128-byte box row
  const int spu = p.nk;                 // one K box per stage
  const int half = static_cast<int>(rank) * kRowsHalf;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsWg0Wide));
    if (lane == 0) {
      // W streams through once (evict first) unless several hidden-row tiles
      // share each W tile: their units run on neighbouring pairs at about
      // the same time, and the second reads it from L2
      const uint64_t pol_w = p.n_nt > 1 ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      const bool leader = rank == 0;
      // W is read-only for the head's life: the W boxes of the first S
      // stages are requested before waiting for the previous kernels on the
      // stream; the hidden rows (which a previous kernel may write) after.
      const int n_my = (n_units - pair + n_pairs - 1) / n_pairs;
      const int pre = min(S, n_my > 0 ? n_my * spu : 0);
      for (int j = 0; j < pre; ++j) {
        const int u = pair + (j / spu) * n_pairs;
        const int vp = u / p.n_nt, kb = j - (j / spu) * spu;
        if (leader) mbar_expect_tx(full_bar(j), 2u * L.stage_bytes);
        tma_load_2d_pair(sB(j), &tmW, kb * kElems, vp * (2 * kBM) + half,
                         cluster_addr(full_bar(j), 0), pol_w);
      }
      grid_dep_wait();
      uint32_t stage = 0, phase = 0, outstanding = 0, out_par = 0;
      bool ok = true;
      int j = 0;
      for (int u = pair; u < n_units && ok; u += n_pairs) {
        const int vp = u / p.n_nt, nt = u - (u / p.n_nt) * p.n_nt;
        for (int kb = 0; kb < spu; ++kb, ++j) {
          const uint32_t fb = cluster_addr(full_bar(stage), 0);
          if (j < pre) {
            tma_load_2d_pair(sA(stage), &tmH, kb * kElems, nt * N + half, fb, pol_h);
            if (leader) mbar_arrive(full_bar(stage));
          } else {
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
            if (leader) mbar_arrive_expect_tx(full_bar(stage), 2u * L.stage_bytes);
            tma_load_2d_pair(sB(stage), &tmW, kb * kElems, vp * (2 * kBM) + half, fb, pol_w);
            tma_load_2d_pair(sA(stage), &tmH, kb * kElems, nt * N + half, fb, pol_h);
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
          const uint32_t d_tmem = tmem_base + slot * static_cast<uint32_t>(N);
#pragma unroll
          for (int sc = 0; sc < kBlocksPerChunk; ++sc) {
            const int kb = c * kBlocksPerChunk + sc;
            if (kb >= p.nk) break;
            // each stage's MMAs go out as soon as its loads have landed
            // (waiting for both stages of a chunk first measured slower)
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
    const int q = warp & 3;                    // TMEM lane quarter: hidden rows 32 q ..
    const int g = (warp - 4) >> 2;             // column half: the unit's tile 2 vp + g
    const int et = threadIdx.x - 128;          // 0 .. ET-1
    const uint32_t tlane = static_cast<uint32_t>(q * 32) << 16;
    uint8_t* xs = xsall + (warp - 4) * kPairXsBytes;
    const uint32_t xs_u32 = smem_u32(xs);
    const bool tma_lg = p.tma_logits != 0;
    // without the tensor map (rows not 16-byte aligned): plain stores
    const bool vec = (p.V & 3) == 0 && (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0;
    uint32_t nbuf = 0;                         // staging buffers used so far
    uint32_t slot = 0, sph = 0;
    bool failed = false;
    using Acc = typename std::conditional<MODE == MODE_INT, int32_t, float>::type;
    for (int u = pair; u < n_units; u += n_pairs) {
      const int vp = u / p.n_nt, nt = u - (u / p.n_nt) * p.n_nt;
      Acc acc[WBLK][16];
      for (int c = 0; c < p.n_chunks; ++c) {
        const uint32_t cur = slot, cph = sph;
        if (++slot == 2u) { slot = 0; sph ^= 1u; }
        if (!failed && !mbar_wait(accf_bar(cur), cph, abort_flag, p.timeout_ns)) {
          failed = true;
          *abort_flag = 1;
        }
        if (failed) continue;
        tc_fence_after();
        const uint32_t sbase = tmem_base + tlane + cur * static_cast<uint32_t>(N) +
                               static_cast<uint32_t>(g * WBLK * 16);
        // two groups of two 32-column loads, one wait each (a wait per
        // load leaves the drain latency-bound)
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
            if constexpr (MODE == MODE_INT) {
              // exact integer chunk sums (|sum| <= 128 * 2^14 = 2^21): adding
              // 1.5 * 2^23 is exact and leaves the integer in the low
              // mantissa bits; int32 fold
#pragma unroll
              for (int i = 0; i < 16; i += 2) {
                float f0 = __uint_as_float(rr[i]), f1 = __uint_as_float(rr[i + 1]);
                add2_rn(f0, f1, 12582912.0f, 12582912.0f);
                const int32_t x0 = __float_as_int(f0) - 0x4B400000;
                const int32_t x1 = __float_as_int(f1) - 0x4B400000;
                acc[bb][i] = (c == 0) ? x0 : acc[bb][i] + x0;
                acc[bb][i + 1] = (c == 0) ? x1 : acc[bb][i + 1] + x1;
              }
            } else if (c == 0) {
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
        tc_fence_before();   // slot fully read: hand it back to the leader's MMA warp
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(acce_bar(cur));
          else mbar_arrive_remote(cluster_addr(acce_bar(cur), 0));
        }
      }
      if (epi_bar_or<ET>(failed || *abort_flag)) {
        if (et == 0) { *abort_flag = 1; atomicOr(p.err, ERR_TIMEOUT); }
        break;
      }
      const int tile = 2 * vp + g;                     // this warp's 128-row vocabulary tile
      const int vt0 = tile * kBM;                      // its first vocabulary row (this head)
      const int lim = p.V - vt0;                       // its rows below V (<= 0: none)
      const int nw0 = nt * N + static_cast<int>(rank) * kRowsHalf + q * 32;   // warp's row 0
      const int n = nw0 + lane;                        // this thread's hidden row
      if (p.logits != nullptr && lim > 0) {
        // per 16-column block the warp's 32 rows x 16 logits go to a staging
        // buffer (row = lane); the tensor map's store (clipped at B and V)
        // then runs asynchronously while the warp drains the next unit, or,
        // without it, each store instruction writes 8 rows x 64 bytes
        const int rl = lane & 7, cc = lane >> 3;
#pragma unroll
        for (int bb = 0; bb < WBLK; ++bb) {
          // blocks wholly past V or B store nothing (warp-uniform)
          if (vt0 + bb * 16 >= p.V || nw0 >= p.B) continue;
          const uint32_t buf = nbuf & 1u;
          if (tma_lg && nbuf >= 2) {
            if (lane == 0) bulk_wait_group_read<1>();   // this buffer's previous store has read it
            __syncwarp();
          }
          uint8_t* sb = xs + buf * kPairStageBuf;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 w;
            if constexpr (MODE == MODE_INT) {
              w = make_uint4(acc[bb][4 * k], acc[bb][4 * k + 1], acc[bb][4 * k + 2], acc[bb][4 * k + 3]);
            } else {
              w = make_uint4(__float_as_uint(acc[bb][4 * k]), __float_as_uint(acc[bb][4 * k + 1]),
                             __float_as_uint(acc[bb][4 * k + 2]), __float_as_uint(acc[bb][4 * k + 3]));
            }
            *reinterpret_cast<uint4*>(sb + lane * 64 + 16 * (k ^ ((lane >> 1) & 3))) = w;
          }
          if (tma_lg) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmL, xs_u32 + buf * kPairStageBuf, vt0 + bb * 16, nw0);
              bulk_commit_group();
            }
            ++nbuf;
          } else {
            __syncwarp();
            uint32_t* lg = reinterpret_cast<uint32_t*>(p.logits);
            const int v = vt0 + bb * 16 + 4 * cc;        // first of this lane's four columns
#pragma unroll
            for (int r8 = 0; r8 < 4; ++r8) {
              const int r = r8 * 8 + rl;
              const uint4 w =
                  *reinterpret_cast<const uint4*>(sb + r * 64 + 16 * (cc ^ ((r >> 1) & 3)));
              const int nr = nw0 + r;
              if (nr < p.B) {
                uint32_t* dst = lg + static_cast<size_t>(nr) * p.V + v;
                if (vec && v + 3 < p.V) {
                  *reinterpret_cast<uint4*>(dst) = w;
                } else {
                  if (v < p.V) dst[0] = w.x;
                  if (v + 1 < p.V) dst[1] = w.y;
                  if (v + 2 < p.V) dst[2] = w.z;
                  if (v + 3 < p.V) dst[3] = w.w;
                }
              }
            }
            __syncwarp();
          }
        }
      }
      if (lim > 0 && n < p.B) {
        // this row's record of the tile: ascending vocabulary order, a strict
        // comparison keeps the lowest index of the maximum; rows at or past V
        // (only in the last tile) count as -inf / INT32_MIN
        const int vg0 = p.v_off + vt0;
        const size_t o = static_cast<size_t>(n) * p.n_vt + tile;   // records [B][n_vt]
        auto fold = [&](auto ragged) {
          constexpr bool kRagged = decltype(ragged)::value;
          if constexpr (MODE == MODE_INT) {
            ITop2 t{INT32_MIN, INT32_MAX, INT32_MIN};
#pragma unroll
            for (int bb = 0; bb < WBLK; ++bb)
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int j = bb * 16 + i;
                const int32_t x = (!kRagged || j < lim) ? acc[bb][i] : INT32_MIN;
                const bool gt = x > t.m;
                t.s = gt ? t.m : max(t.s, x);
                t.i = gt ? vg0 + j : t.i;
                t.m = gt ? x : t.m;
              }
            reinterpret_cast<int32_t*>(p.rec_m)[o] = t.m;
            p.rec_i[o] = t.i;
            reinterpret_cast<int32_t*>(p.rec_s)[o] = t.s;
          } else {
            Top2 t{-INFINITY, INT32_MAX, -INFINITY};
#pragma unroll
            for (int bb = 0; bb < WBLK; ++bb)
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int j = bb * 16 + i;
                const float x = (!kRagged || j < lim) ? acc[bb][i] : -INFINITY;
                const bool gt = x > t.m;
                t.s = gt ? t.m : fmaxf(t.s, x);
                t.i = gt ? vg0 + j : t.i;
                t.m = gt ? x : t.m;
              }
            p.rec_m[o] = t.m;
            p.rec_i[o] = t.i;
            p.rec_s[o] = t.s;
          }
        };
        if (lim >= kBM) fold(std::false_type{});
        else fold(std::true_type{});
      }
    }
    if (failed && et == 0) atomicOr(p.err, ERR_TIMEOUT);
    // the logits stores are complete before the CTA (and its shared memory)
    // goes away
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
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
