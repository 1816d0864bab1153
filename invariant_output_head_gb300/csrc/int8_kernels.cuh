// int8_kernels.cuh -- the exact integer head (int8 x int8 -> int32) on sm_103a.
//
// "Eliminating Nondeterminism in LLM Inference with Integer-Only Arithmetic",
// section "DetLLM": the only hardware-dispatched operation is the int8 x int8
// -> int32 matmul, and argmax breaks ties toward the lowest token id; section
// "What if we don't use floats at all?": integer sums are exact in any order
// while they cannot overflow, and the overflow can be bounded in advance.
//
// sm_103a has no tcgen05 integer MMA (kind::i8 does not assemble for this
// target), so the integer product runs on the kind::f16 tensor-core path with
// exact arithmetic:
//   * every int8 value is converted to IEEE fp16, where -128..127 are exact;
//   * each product of two such values is an integer of magnitude <= 2^14,
//     exact in the fp32 accumulator;
//   * the K axis is cut into chunks of 1024 elements, each accumulated in its
//     own TMEM accumulator, so every partial sum is an integer of magnitude
//     <= 1024 * 2^14 = 2^24 and exact in fp32 (footnote 3 of the same page:
//     2^24 is where fp32 runs out of integer precision);
//   * the chunk sums are converted to int32 and added in int32; with
//     d <= 16384 every logit is bounded by 16384 * 2^14 = 2^28 < 2^31.
//
// The conversion int8 -> fp16 is exact bit arithmetic: flipping the sign bit
// gives u = x + 128 in 0..255; the half with bits 0x6400 | u is 1024 + u;
// subtracting 1152 (exact) leaves x.
//
// Warp roles (480 threads): warp 0 TMA of int8 tiles (W and the hidden rows)
// into an S-stage ring, warps 6..13 converters, warps 1 and 14 MMA issuers
// (even and odd K boxes, each into its own accumulator: one thread's
// tcgen05.mma issue rate would bound the kernel), warps 2..5 epilogue. The converters write each W box, as fp16, straight into a
// ring of tensor-memory slots (tcgen05.st; the MMA takes its A operand from
// tensor memory), and the small hidden-row box into fp16 shared memory in the
// same stage (the MMA's B operand). Keeping the fp16 copy of W out of shared
// memory leaves it to the int8 ring. Each issuer's chunk sums go to a ring
// of two tensor-memory accumulators that the epilogue drains into int32
// registers as they finish; the two issuers' sums of a chunk are integers
// below 2^24, exact in fp32, so the split changes no bit of the result.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>
#include "ptx.cuh"
#include "head_kernels.cuh"

namespace detlm {

constexpr int kI8Chunk = 1024;            // K elements per exact fp32 chunk
constexpr int kI8BoxesPerChunk = kI8Chunk / kRowBytes;   // 8 int8 K boxes
constexpr int kI8ConvWarps = 8;            // converter warps (warps 6 .. 13)
constexpr int kI8Threads = 192 + 32 * kI8ConvWarps + 32;   // + warp 14: second MMA issuer
constexpr int kI8MaxD = 16384;            // keeps |logit| <= 16384 * 2^14 = 2^28
constexpr int kI8MaxStages = 12;
constexpr int kI8MaxN = 64;
constexpr int kI8AccCols = 256;           // 2 chunk slots x 2 issuers x N <= 64 columns
constexpr int kI8ASlots = 4;              // fp16 W boxes in tensor memory, 64 columns each
static_assert(kI8AccCols + 64 * kI8ASlots <= 512, "tensor memory");

__host__ __device__ inline int int8_chunks(int64_t d) {
  return static_cast<int>((d + kI8Chunk - 1) / kI8Chunk);
}

// Hidden rows per MMA for the integer head (B below the wide-batch path):
// B rounded up to 16, at most 64 (more rows: several column tiles).
__host__ __device__ inline int int8_cols_for(int64_t B, int64_t /*d*/) {
  int n = static_cast<int>((B + 15) / 16) * 16;
  if (n < 16) n = 16;
  return n < kI8MaxN ? n : kI8MaxN;
}

struct Int8Params {
  int32_t V, d, B;           // V: vocabulary rows of this head's W
  int32_t N, n_vt, n_nt, nk, n_chunks;
  int32_t stages;            // int8 ring depth
  uint32_t idesc;
  int32_t* logits;           // optional int32 [B, V]
  int32_t* rec_m;            // [B, n_vt]
  int32_t* rec_i;
  int32_t* rec_s;
  int* err;
  int32_t stall;
  uint64_t timeout_ns;
  int32_t v_off;             // vocabulary index of this head's first W row
};
static_assert(sizeof(Int8Params) <= 128, "kernel parameter struct above 128 bytes");

// One stage: the int8 W box [128 rows x 128 B], the int8 hidden-row box
// [N x 128 B], then the hidden rows as fp16 in two 64-element sub-tiles
// [N x 128 B each, 128-byte swizzle]. With N a multiple of 16 every part
// starts on a 1024-byte boundary.
struct Int8Layout {
  uint32_t h8, h16, stage, tx, ctrl, red, xp, total;
};

__host__ __device__ inline Int8Layout int8_layout(int N, int stages) {
  Int8Layout L;
  L.h8 = kBM * kRowBytes;
  L.h16 = L.h8 + static_cast<uint32_t>(N) * kRowBytes;
  L.stage = L.h16 + 2u * static_cast<uint32_t>(N) * kRowBytes;
  L.tx = L.h16;                                   // bytes the TMA brings per stage
  L.ctrl = static_cast<uint32_t>(stages) * L.stage;
  // full[S], empty[S], conv[S], a_empty[kI8ASlots], accf[2], acce[2], never,
  // drain; then the TMEM address holder and the abort flag
  L.red = L.ctrl + (3u * stages + kI8ASlots + 6u) * 8u + 16u;
  L.xp = L.red + 3u * 4u * static_cast<uint32_t>(N) * 4u;
  L.total = L.xp + 4u * kXpWords * 4u;
  return L;
}

// four int8 in one word -> two half2 holding the same integers exactly
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;             // bytes x + 128
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  const __half2 k = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), k);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), k);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

// Elementwise int8 -> fp16 (exact) for the wide-batch integer path: n is a
// multiple of 16 (rows of d % 16 == 0 elements).
__global__ void i8_to_f16_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, size_t n16) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 w = in[i];
    uint4 o0, o1;
    i8x4_to_h2x2(w.x, o0.x, o0.y);
    i8x4_to_h2x2(w.y, o0.z, o0.w);
    i8x4_to_h2x2(w.z, o1.x, o1.y);
    i8x4_to_h2x2(w.w, o1.z, o1.w);
    out[2 * i] = o0;
    out[2 * i + 1] = o1;
  }
}

// Convert ROWS rows of a swizzled int8 tile (128 B per row) into the two
// swizzled fp16 sub-tiles (each 128 B per row) at dst (sub-tile 1 at
// dst + ROWS * 128). The converter threads share the 16-byte chunks; the
// trip count is a compile-time constant so all loads are issued before the
// conversions (the loop was latency-bound otherwise).
template <int ROWS>
__device__ __forceinline__ void convert_tile(const uint8_t* src, uint8_t* dst, int ct) {
  constexpr int kNT = 32 * kI8ConvWarps;
  constexpr int kIters = (ROWS * 8 + kNT - 1) / kNT;
  uint4 w[kIters];
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int q = ct + it * kNT;
    const int r = q >> 3, c = q & 7;                       // row, logical 16-byte chunk
    if (q < ROWS * 8)
      w[it] = *reinterpret_cast<const uint4*>(src + r * 128 + ((c ^ (r & 7)) << 4));
  }
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int q = ct + it * kNT;
    if (q >= ROWS * 8) continue;
    const int r = q >> 3, c = q & 7;
    uint4 o0, o1;
    i8x4_to_h2x2(w[it].x, o0.x, o0.y);
    i8x4_to_h2x2(w[it].y, o0.z, o0.w);
    i8x4_to_h2x2(w[it].z, o1.x, o1.y);
    i8x4_to_h2x2(w[it].w, o1.z, o1.w);
    // int8 elements 16c .. 16c+15 -> fp16 sub-tile c/4, chunks 2(c%4), 2(c%4)+1
    uint8_t* sub = dst + (c >> 2) * ROWS * 128 + r * 128;
    const int cc = (c & 3) * 2;
    *reinterpret_cast<uint4*>(sub + ((cc ^ (r & 7)) << 4)) = o0;
    *reinterpret_cast<uint4*>(sub + (((cc + 1) ^ (r & 7)) << 4)) = o1;
  }
}

// tcgen05 helpers used only here: 32 consecutive 32-bit columns stored per
// thread (thread i -> lane base + i), the wait for them, and an MMA whose A
// operand is read from tensor memory (row m of A in lane m, two fp16 of K
// per 32-bit column, eight columns per K = 16 step).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
         "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
         "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
         "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
         "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int N_>
__global__ void __launch_bounds__(kI8Threads, 1)
int8_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                 const Int8Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  constexpr int N = N_;
  static_assert(N % 16 == 0 && N <= kI8MaxN && 4 * N <= kI8AccCols, "shape");
  const Int8Layout L = int8_layout(N, S);

  const uint32_t bar0 = smem_u32(smem + L.ctrl);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto conv = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto a_empty = [&](int a) { return bar0 + 8u * (3 * S + a); };
  auto accf = [&](int b) { return bar0 + 8u * (3 * S + kI8ASlots + b); };
  auto acce = [&](int b) { return bar0 + 8u * (3 * S + kI8ASlots + 2 + b); };
  const uint32_t never_bar = bar0 + 8u * (3 * S + kI8ASlots + 4);
  const uint32_t drain_bar = bar0 + 8u * (3 * S + kI8ASlots + 5);
  uint32_t* tmem_holder =
      reinterpret_cast<uint32_t*>(smem + L.ctrl + (3 * S + kI8ASlots + 6) * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* red_m = reinterpret_cast<int32_t*>(smem + L.red);
  int32_t* red_i = red_m + 4 * N;
  int32_t* red_s = red_i + 4 * N;
  int32_t* xpose = reinterpret_cast<int32_t*>(smem + L.xp);
  const uint32_t base = smem_u32(smem);
  // stages whose W boxes the producer requests before the previous kernels
  // on the stream have finished (at most the ring, at most this CTA's work)
  auto pre_stages = [&]() {
    const int units = p.n_vt * p.n_nt;
    const int n_my = (units - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                     static_cast<int>(gridDim.x);
    return min(S, n_my > 0 ? n_my * p.nk : 0);
  };

  if (threadIdx.x == 0) {
    // this thread is the TMA producer: W is read-only for the head's life,
    // so the W boxes of the first S stages are requested first -- right
    // after their full barriers exist, before the other barriers, the
    // tensor-memory allocation and the wait for the previous kernels on the
    // stream; the hidden rows (which a previous kernel may write) only after
    // that wait
    for (int s = 0; s < S; ++s) mbar_init(full(s), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    const uint64_t pol_w = policy_evict_first();
    const int pre = pre_stages();
    for (int j = 0; j < pre; ++j) {
      const int u = blockIdx.x + (j / p.nk) * gridDim.x;
      const int vt = u / p.n_nt, kb = j - (j / p.nk) * p.nk;
      mbar_expect_tx(full(j), L.tx);
      tma_load_2d(base + j * L.stage, &tmW, kb * kRowBytes, vt * kBM, full(j), pol_w);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(empty(s), 1);
      mbar_init(conv(s), kI8ConvWarps);
    }
    for (int a = 0; a < kI8ASlots; ++a) mbar_init(a_empty(a), 1);
    for (int b = 0; b < 2; ++b) { mbar_init(accf(b), 2); mbar_init(acce(b), 4); }
    mbar_init(never_bar, 1);
    mbar_init(drain_bar, 2);
    *abort_flag = 0;
    fence_mbar_init();
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
  const uint32_t tmem_a = tmem_base + static_cast<uint32_t>(kI8AccCols);   // A slots
  const int n_units = p.n_vt * p.n_nt;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      // (the W boxes of the first `pre` stages were requested in the set-up)
      const int pre = pre_stages();
      grid_dep_wait();
      uint32_t stage = 0, phase = 0, outstanding = 0, out_par = 0;
      bool ok = true;
      int j = 0;                     // stages issued by this CTA
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const int vt = u / p.n_nt, nt = u - (u / p.n_nt) * p.n_nt;
        for (int kb = 0; kb < p.nk; ++kb, ++j) {
          const uint32_t a = base + stage * L.stage;
          if (j < pre) {             // W already requested: add the hidden rows
            tma_load_2d(a + L.h8, &tmH, kb * kRowBytes, nt * N, full(stage), pol_h);
            mbar_arrive(full(stage));
          } else {
            if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
            outstanding &= ~(1u << stage);
            mbar_arrive_expect_tx(full(stage), L.tx);
            tma_load_2d(a, &tmW, kb * kRowBytes, vt * kBM, full(stage), pol_w);
            tma_load_2d(a + L.h8, &tmH, kb * kRowBytes, nt * N, full(stage), pol_h);
          }
          outstanding |= 1u << stage;
          out_par = (out_par & ~(1u << stage)) | (phase << stage);
          if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, ERR_TIMEOUT);
        // let this thread's loads still in flight land before the CTA exits
        const int zero = 0;
        for (int s = 0; s < S; ++s)
          if ((outstanding >> s) & 1u) mbar_wait(full(s), (out_par >> s) & 1u, &zero, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 14) {
    // ------------------------------------------------------- MMA issuers
    // issuer `which` takes the K boxes kb % 2 == which of every chunk into
    // accumulator (slot, which); both commit every chunk's accf (count 2)
    if (lane == 0) {
      const int which = warp == 1 ? 0 : 1;
      uint32_t cslot = 0, cph = 0;
      bool ok = true;
      if (p.stall) ok = mbar_wait(never_bar, 0, abort_flag, p.timeout_ns);
      int gb = 0;                                   // boxes seen by this CTA (all issuers)
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        for (int c0 = 0; c0 < p.nk && ok; c0 += kI8BoxesPerChunk) {
          if (!mbar_wait(acce(cslot), cph ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
          const uint32_t d_tmem = tmem_base + (cslot * 2u + which) * static_cast<uint32_t>(N);
          const int nb = min(kI8BoxesPerChunk, p.nk - c0);
          for (int kin = which; kin < nb; kin += 2) {
            const int g = gb + kin;                   // this box's ring positions
            const uint32_t stage = static_cast<uint32_t>(g % S);
            const uint32_t phase = static_cast<uint32_t>((g / S) & 1);
            const uint32_t aslot = static_cast<uint32_t>(g % kI8ASlots);
            if (!mbar_wait(conv(stage), phase, abort_flag, p.timeout_ns)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a_tmem = tmem_a + aslot * 64u;
            const uint32_t h16 = base + stage * L.stage + L.h16;
            const uint64_t db0 = sdesc_sw128(h16);
            const uint64_t db1 = sdesc_sw128(h16 + N * kRowBytes);
#pragma unroll
            for (int k = 0; k < 8; ++k)   // K = 16 per MMA: 8 TMEM columns of A, 32 bytes of B
              mma_f16_tmem_a(d_tmem, a_tmem + 8u * k, (k < 4 ? db0 : db1) + 2u * (k & 3), p.idesc,
                             (kin != which) || k != 0);
            mma_commit(empty(stage));
            mma_commit(a_empty(aslot));
          }
          if (!ok) break;
          // every chunk: an arrival from each issuer (after its MMAs, if any)
          mma_commit(accf(cslot));
          if (++cslot == 2u) { cslot = 0; cph ^= 1u; }
          gb += nb;
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
  } else if (warp >= 6 && warp < 6 + kI8ConvWarps) {
    // ------------------------------------------------------- converters
    // Warp w converts rows 32*(w%4) .. +31 (its tensor-memory lane quarter)
    // of the W box, K half (w-6)/4; all converter threads share the hidden
    // rows.
    const int ct = threadIdx.x - 192;   // 0 .. 32 * kI8ConvWarps - 1
    const int q = warp & 3, hk = (warp - 6) >> 2;
    const int r = q * 32 + lane;
    const uint32_t tl = static_cast<uint32_t>(q * 32) << 16;
    uint32_t stage = 0, phase = 0, aslot = 0, aph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      for (int kb = 0; kb < p.nk; ++kb) {
        const bool g1 = mbar_wait(full(stage), phase, abort_flag, p.timeout_ns);
        const bool g2 = g1 && mbar_wait(a_empty(aslot), aph ^ 1u, abort_flag, p.timeout_ns);
        if (!g2) { ok = false; break; }
        tc_fence_after();
        const uint8_t* st = smem + stage * L.stage;
        uint4 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = hk * 4 + i;                  // logical 16-byte chunk of the row
          w[i] = *reinterpret_cast<const uint4*>(st + r * kRowBytes + ((c ^ (r & 7)) << 4));
        }
        uint32_t o[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          i8x4_to_h2x2(w[i].x, o[8 * i + 0], o[8 * i + 1]);
          i8x4_to_h2x2(w[i].y, o[8 * i + 2], o[8 * i + 3]);
          i8x4_to_h2x2(w[i].z, o[8 * i + 4], o[8 * i + 5]);
          i8x4_to_h2x2(w[i].w, o[8 * i + 6], o[8 * i + 7]);
        }
        tmem_st32(tmem_a + tl + aslot * 64u + static_cast<uint32_t>(hk * 32), o);
        convert_tile<N>(st + L.h8, smem + stage * L.stage + L.h16, ct);
        tmem_wait_st();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(conv(stage));
        if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
        if (++aslot == static_cast<uint32_t>(kI8ASlots)) { aslot = 0; aph ^= 1u; }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.err, ERR_TIMEOUT);
    }
  } else {
    // --------------------------------------------------------- epilogue
    grid_dep_wait();          // logits and records: only after the previous kernels
    const int q = warp & 3;
    const int et = threadIdx.x - 64;
    const int row = q * 32 + lane;
    const uint32_t tlane = static_cast<uint32_t>(q * 32) << 16;
    uint32_t cslot = 0, cph = 0;
    bool failed = false;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const int vt = u / p.n_nt, nt = u - (u / p.n_nt) * p.n_nt;
      int32_t acc[N / 16][16];
#pragma unroll
      for (int bb = 0; bb < N / 16; ++bb)
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[bb][i] = 0;
      for (int ch = 0; ch < p.n_chunks; ++ch) {
        const uint32_t cur = cslot, ph = cph;
        if (++cslot == 2u) { cslot = 0; cph ^= 1u; }
        if (!failed && !mbar_wait(accf(cur), ph, abort_flag, p.timeout_ns)) {
          failed = true;
          *abort_flag = 1;
        }
        if (failed) continue;
        tc_fence_after();
        // issuer 1 has boxes in this chunk unless the chunk is a single box
        const int nb = min(kI8BoxesPerChunk, p.nk - ch * kI8BoxesPerChunk);
#pragma unroll
        for (int bb = 0; bb < N / 16; ++bb) {
          uint32_t r0[16], r1[16];
          tmem_ld16(tmem_base + tlane + (cur * 2u) * static_cast<uint32_t>(N) + bb * 16, r0);
          tmem_ld16(tmem_base + tlane + (cur * 2u + 1u) * static_cast<uint32_t>(N) + bb * 16, r1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            acc[bb][i] += __float2int_rn(__uint_as_float(r0[i])) +
                          (nb > 1 ? __float2int_rn(__uint_as_float(r1[i])) : 0);
        }
        tc_fence_before();   // accumulator fully read: hand it back to the MMA warp
        __syncwarp();
        if (lane == 0) mbar_arrive(acce(cur));
      }
      if (epi_bar_or<128>(failed || *abort_flag)) {
        if (et == 0) { *abort_flag = 1; atomicOr(p.err, ERR_TIMEOUT); }
        break;
      }
      const int v = vt * kBM + row;
      const bool vok = v < p.V;
      const int n0 = nt * N;
#pragma unroll
      for (int bb = 0; bb < N / 16; ++bb) {
        const int c0 = bb * 16;
        if (p.logits != nullptr && vok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = n0 + c0 + i;
            if (n < p.B) p.logits[static_cast<size_t>(n) * p.V + v] = acc[bb][i];
          }
        }
        int32_t* xp = xpose + q * kXpWords;
#pragma unroll
        for (int i = 0; i < 16; ++i) xp[lane * kXpStride + i] = vok ? acc[bb][i] : INT32_MIN;
        __syncwarp();
        const ITop2 t = xp_itop2(xp, lane, p.v_off + vt * kBM + q * 32);
        if (lane < 16) {
          red_m[q * N + c0 + lane] = t.m;
          red_i[q * N + c0 + lane] = t.i;
          red_s[q * N + c0 + lane] = t.s;
        }
        __syncwarp();
      }
      named_bar_sync(1, 128);
      for (int c = et; c < N; c += 128) {
        const int n = n0 + c;
        if (n >= p.B) continue;
        ITop2 t[4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) t[qq] = ITop2{red_m[qq * N + c], red_i[qq * N + c], red_s[qq * N + c]};
        const ITop2 rr = itop2_merge(itop2_merge(t[0], t[1]), itop2_merge(t[2], t[3]));
        const size_t o = static_cast<size_t>(n) * p.n_vt + vt;   // records [B][n_vt]
        p.rec_m[o] = rr.m;
        p.rec_i[o] = rr.i;
        p.rec_s[o] = rr.s;
      }
      named_bar_sync(1, 128);
    }
    if (failed && et == 0) atomicOr(p.err, ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  // the merge kernel may be scheduled now (at the end: waiting merge blocks
  // would take issue slots from the converter warps)
  grid_dep_launch();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512u);
  }
}

struct Int8MergeParams {
  int32_t B, n_vt;
  const int32_t* rec_m;
  const int32_t* rec_i;
  const int32_t* rec_s;
  int32_t* token;
  int32_t* gap;
  AcceptArgs acc;
};

__global__ void __launch_bounds__(kMergeThreads) int8_merge_kernel(const Int8MergeParams p) {
  grid_dep_launch();  // the next call's kernel 1 may start (it prefetches only W)
  grid_dep_wait();
  const int n = blockIdx.x;
  const int g = threadIdx.x;
  const size_t base = static_cast<size_t>(n) * p.n_vt;
  __shared__ ITop2 part[4];
  ITop2 acc{INT32_MIN, INT32_MAX, INT32_MIN};
  for (int t0 = g; t0 < p.n_vt; t0 += kMergeThreads * kMergeBatch) {
    ITop2 r[kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      const int t = t0 + j * kMergeThreads;
      r[j] = t < p.n_vt ? ITop2{p.rec_m[base + t], p.rec_i[base + t], p.rec_s[base + t]}
                        : ITop2{INT32_MIN, INT32_MAX, INT32_MIN};
    }
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) acc = itop2_merge(acc, r[j]);
  }
  const ITop2 tot = block_tree128(acc, itop2_merge, part);
  if (g == 0) {
    p.token[n] = tot.i;
    p.gap[n] = tot.s == INT32_MIN ? INT32_MAX : tot.m - tot.s;
    accept_fold(p.acc, n, tot.i);
  }
}

}  // namespace detlm
