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
// Warp roles (448 threads): warp 0 TMA of int8 tiles, warp 1 MMA issuer,
// warps 2..5 epilogue, warps 6..13 converters (int8 ring -> fp16 ring in the
// 128-byte swizzle layout the MMA descriptors expect).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>
#include "ptx.cuh"
#include "head_kernels.cuh"

namespace detlm {

constexpr int kI8Chunk = 1024;            // K elements per exact fp32 chunk
constexpr int kI8ConvWarps = 8;            // converter warps (warps 6 .. 13)
constexpr int kI8Threads = 192 + 32 * kI8ConvWarps;
constexpr int kI8MaxD = 16384;            // 16 chunks; keeps |logit| <= 2^28
constexpr int kI8MaxStages8 = 8;
constexpr int kI8MaxN = 64;               // keeps >= 5 int8 stages in shared memory

__host__ __device__ inline int int8_chunks(int64_t d) {
  return static_cast<int>((d + kI8Chunk - 1) / kI8Chunk);
}

// Hidden rows per MMA for the integer head: two TMEM buffers of n_chunks
// accumulators each must fit 512 columns, and the int8 and fp16 rings must
// fit shared memory.
__host__ __device__ inline int int8_cols_for(int64_t B, int64_t d) {
  const int nc = int8_chunks(d);
  int cap = (256 / nc) / 16 * 16;
  if (cap < 16) cap = 16;
  if (cap > kI8MaxN) cap = kI8MaxN;
  int n = static_cast<int>((B + 15) / 16) * 16;
  if (n < 16) n = 16;
  return n < cap ? n : cap;
}

struct Int8Params {
  int32_t V, d, B;
  int32_t N, n_vt, n_nt, nk, n_chunks;
  int32_t s8, s16;           // int8 ring and fp16 ring depths
  uint32_t tmem_cols;
  uint32_t idesc;
  int32_t* logits;           // optional int32 [B, V]
  int32_t* rec_m;            // [n_vt, B]
  int32_t* rec_i;
  int32_t* rec_s;
  int* err;
  int32_t stall;
  uint64_t timeout_ns;
};

struct Int8Layout {
  uint32_t a8, b8, st8, a16, b16, st16, off16, ctrl, red, xp, total;
};

__host__ __device__ inline Int8Layout int8_layout(int N, int s8, int s16) {
  Int8Layout L;
  L.a8 = kBM * kRowBytes;                       // int8 W tile: 128 rows x 128 B
  L.b8 = static_cast<uint32_t>(N) * kRowBytes;  // int8 h tile
  L.st8 = L.a8 + L.b8;
  L.a16 = 2u * kBM * kRowBytes;                 // fp16 W: two 64-element sub-tiles
  L.b16 = 2u * static_cast<uint32_t>(N) * kRowBytes;
  L.st16 = L.a16 + L.b16;
  L.off16 = static_cast<uint32_t>(s8) * L.st8;
  L.ctrl = L.off16 + static_cast<uint32_t>(s16) * L.st16;
  // f8full[s8], f8empty[s8], f16full[s16], f16empty[s16], accf[2], acce[2],
  // never, drain; then TMEM holder and abort flag
  L.red = L.ctrl + (2u * s8 + 2u * s16 + 6u) * 8u + 16u;
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

template <int N_>
__global__ void __launch_bounds__(kI8Threads, 1)
int8_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                 const Int8Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S8 = p.s8, S16 = p.s16;
  constexpr int N = N_;
  const Int8Layout L = int8_layout(N, S8, S16);

  const uint32_t bar0 = smem_u32(smem + L.ctrl);
  auto f8full = [&](int s) { return bar0 + 8u * s; };
  auto f8empty = [&](int s) { return bar0 + 8u * (S8 + s); };
  auto f16full = [&](int s) { return bar0 + 8u * (2 * S8 + s); };
  auto f16empty = [&](int s) { return bar0 + 8u * (2 * S8 + S16 + s); };
  auto accf = [&](int b) { return bar0 + 8u * (2 * S8 + 2 * S16 + b); };
  auto acce = [&](int b) { return bar0 + 8u * (2 * S8 + 2 * S16 + 2 + b); };
  const uint32_t never_bar = bar0 + 8u * (2 * S8 + 2 * S16 + 4);
  const uint32_t drain_bar = bar0 + 8u * (2 * S8 + 2 * S16 + 5);
  uint32_t* tmem_holder =
      reinterpret_cast<uint32_t*>(smem + L.ctrl + (2 * S8 + 2 * S16 + 6) * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* red_m = reinterpret_cast<int32_t*>(smem + L.red);
  int32_t* red_i = red_m + 4 * N;
  int32_t* red_s = red_i + 4 * N;
  int32_t* xpose = reinterpret_cast<int32_t*>(smem + L.xp);
  const uint32_t base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S8; ++s) { mbar_init(f8full(s), 1); mbar_init(f8empty(s), kI8ConvWarps); }
    for (int s = 0; s < S16; ++s) { mbar_init(f16full(s), kI8ConvWarps); mbar_init(f16empty(s), 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(accf(b), 1); mbar_init(acce(b), 4); }
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
    tmem_alloc(smem_u32(tmem_holder), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int n_units = p.n_vt * p.n_nt;
  const int kb_per_chunk = kI8Chunk / kRowBytes;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      // W is read-only for the head's life: the W boxes of the first S8
      // stages are requested before waiting for the previous kernels on the
      // stream; the hidden rows (which a previous kernel may write) after.
      const int n_my = (n_units - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                       static_cast<int>(gridDim.x);
      const int pre = min(S8, n_my > 0 ? n_my * p.nk : 0);
      for (int j = 0; j < pre; ++j) {
        const int u = blockIdx.x + (j / p.nk) * gridDim.x;
        const int vt = u / p.n_nt, kb = j - (j / p.nk) * p.nk;
        mbar_expect_tx(f8full(j), L.st8);
        tma_load_2d(base + j * L.st8, &tmW, kb * kRowBytes, vt * kBM, f8full(j), pol_w);
      }
      grid_dep_wait();
      uint32_t stage = 0, phase = 0, outstanding = 0, out_par = 0;
      bool ok = true;
      int j = 0;                     // stages issued by this CTA
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const int vt = u / p.n_nt, nt = u - (u / p.n_nt) * p.n_nt;
        for (int kb = 0; kb < p.nk; ++kb, ++j) {
          const uint32_t a = base + stage * L.st8;
          if (j < pre) {             // W already requested: add the hidden rows
            tma_load_2d(a + L.a8, &tmH, kb * kRowBytes, nt * N, f8full(stage), pol_h);
            mbar_arrive(f8full(stage));
          } else {
            if (!mbar_wait(f8empty(stage), phase ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
            outstanding &= ~(1u << stage);
            mbar_arrive_expect_tx(f8full(stage), L.st8);
            tma_load_2d(a, &tmW, kb * kRowBytes, vt * kBM, f8full(stage), pol_w);
            tma_load_2d(a + L.a8, &tmH, kb * kRowBytes, nt * N, f8full(stage), pol_h);
          }
          outstanding |= 1u << stage;
          out_par = (out_par & ~(1u << stage)) | (phase << stage);
          if (++stage == static_cast<uint32_t>(S8)) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, ERR_TIMEOUT);
        const int zero = 0;
        for (int s = 0; s < S8; ++s)
          if ((outstanding >> s) & 1u) mbar_wait(f8full(s), (out_par >> s) & 1u, &zero, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      if (p.stall) ok = mbar_wait(never_bar, 0, abort_flag, p.timeout_ns);
      int j = 0;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++j) {
        const uint32_t buf = j & 1, aph = (j >> 1) & 1;
        if (!mbar_wait(acce(buf), aph ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < p.nk; ++kb) {
          if (!mbar_wait(f16full(stage), phase, abort_flag, p.timeout_ns)) { ok = false; break; }
          tc_fence_after();
          const int ch = kb / kb_per_chunk;
          const uint32_t d_tmem =
              tmem_base + (buf * static_cast<uint32_t>(p.n_chunks) + ch) * static_cast<uint32_t>(N);
          const uint32_t a16 = base + L.off16 + stage * L.st16;
          const uint32_t b16 = a16 + L.a16;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint64_t da = sdesc_sw128(a16 + t * (kBM * kRowBytes));
            const uint64_t db = sdesc_sw128(b16 + t * (N * kRowBytes));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f16(d_tmem, da + 2u * k, db + 2u * k, p.idesc,
                      ((kb % kb_per_chunk) | t | k) != 0);
          }
          mma_commit(f16empty(stage));
          if (++stage == static_cast<uint32_t>(S16)) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(accf(buf));
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
  } else if (warp >= 6) {
    // ------------------------------------------------------- converters
    const int ct = threadIdx.x - 192;   // 0 .. 32 * kI8ConvWarps - 1
    uint32_t s8 = 0, ph8 = 0, s16 = 0, ph16 = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      for (int kb = 0; kb < p.nk; ++kb) {
        const bool g1 = mbar_wait(f8full(s8), ph8, abort_flag, p.timeout_ns);
        const bool g2 = g1 && mbar_wait(f16empty(s16), ph16 ^ 1u, abort_flag, p.timeout_ns);
        if (!g2) { ok = false; break; }
        const uint8_t* src = smem + s8 * L.st8;
        uint8_t* dst = smem + L.off16 + s16 * L.st16;
        convert_tile<kBM>(src, dst, ct);
        convert_tile<N>(src + L.a8, dst + L.a16, ct);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(f8empty(s8));
          mbar_arrive(f16full(s16));
        }
        if (++s8 == static_cast<uint32_t>(S8)) { s8 = 0; ph8 ^= 1u; }
        if (++s16 == static_cast<uint32_t>(S16)) { s16 = 0; ph16 ^= 1u; }
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
    int j = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++j) {
      const int vt = u / p.n_nt, nt = u - (u / p.n_nt) * p.n_nt;
      const uint32_t buf = j & 1, aph = (j >> 1) & 1;
      const bool got = mbar_wait(accf(buf), aph, abort_flag, p.timeout_ns);
      if (epi_bar_or<128>(!got || *abort_flag)) {
        if (et == 0) { *abort_flag = 1; atomicOr(p.err, ERR_TIMEOUT); }
        break;
      }
      tc_fence_after();
      const uint32_t tlane = static_cast<uint32_t>(q * 32) << 16;
      const int v = vt * kBM + row;
      const bool vok = v < p.V;
      const int n0 = nt * N;
      for (int c0 = 0; c0 < N; c0 += 16) {
        int32_t x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = 0;
        for (int ch = 0; ch < p.n_chunks; ++ch) {
          uint32_t r[16];
          tmem_ld16(tmem_base + tlane +
                        (buf * static_cast<uint32_t>(p.n_chunks) + ch) * static_cast<uint32_t>(N) + c0,
                    r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] += __float2int_rn(__uint_as_float(r[i]));
        }
        if (c0 + 16 >= N) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce(buf));
        }
        if (p.logits != nullptr && vok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = n0 + c0 + i;
            if (n < p.B) p.logits[static_cast<size_t>(n) * p.V + v] = x[i];
          }
        }
        int32_t* xp = xpose + q * kXpWords;
#pragma unroll
        for (int i = 0; i < 16; ++i) xp[lane * kXpStride + i] = vok ? x[i] : INT32_MIN;
        __syncwarp();
        const ITop2 t = xp_itop2(xp, lane, vt * kBM + q * 32);
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
        const ITop2 r = itop2_merge(itop2_merge(t[0], t[1]), itop2_merge(t[2], t[3]));
        const size_t o = static_cast<size_t>(n) * p.n_vt + vt;   // records [B][n_vt]
        p.rec_m[o] = r.m;
        p.rec_i[o] = r.i;
        p.rec_s[o] = r.s;
      }
      named_bar_sync(1, 128);
    }
  }

  tc_fence_before();
  __syncthreads();
  // the merge kernel may be scheduled now (at the end: waiting merge blocks
  // would take issue slots from the converter warps)
  grid_dep_launch();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
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
