// head_kernels.cuh -- the output-head kernels for GB300 (sm_103a).
//
// Kernel 1 (head_gemm_kernel): a persistent, warp-specialised projection
//   z[n, v] = sum_k h[n, k] * W[v, k]
// with W as the 128-row M operand of tcgen05.mma ("swap-AB": the vocabulary
// runs along the tensor core's M axis and TMEM lanes, the hidden rows along
// N). A unit of work is one 128-row vocabulary tile x N hidden rows, N a
// multiple of 16 (the hidden rows padded with zeros). The K loop walks d in
// ascending 128-byte blocks, four MMAs of K=16 each, always the same steps
// for a given d: the reduction order of every logit is fixed by the weight's
// shape, never by the row count ("TandemLLM docs, 12 Exactness", section
// 12.2).
//
// Accumulation in K chunks: the tensor core's fp32 accumulation rounds each
// K=16 step toward zero-ish, so a long K loop in one accumulator drifts by
// about half an ulp per step when all products share a sign. K is therefore
// cut into chunks of kChunkK elements (a function of d only); each chunk is
// accumulated from zero in one of up to kMaxSlots TMEM slots (a ring), and the
// epilogue adds the chunk sums in fp32 registers with round-to-nearest, in
// ascending chunk order. This keeps every logit within 1e-6 * sum|w h| and
// is the same arithmetic for every B.
//
// Warp 0 issues TMA loads into an S-stage ring; warp 1 (and, up to N = 128,
// warps 6 and 7, round robin over K chunks) issues the MMAs into the chunk
// slot ring; the epilogue warps (2..5, or eight warps 4..11 at N = 256) drain
// each slot into running sums (one thread per vocabulary row and up to 128
// hidden-row columns), then write the optional fp32 logits and the per-tile
// record of each hidden row:
//   greedy : (m, i, s) = tile maximum, lowest index attaining it, runner-up
//            value of the tile's multiset (gated: also the lowest index of
//            the maximum of the logits rounded to 16 bits; sampling: the
//            same record over the scores z/T + G).
// The log-prob call has its own projection kernel (head_rows_kernel, in
// rows_kernels.cuh) with the same K chunks and fold, hence the same logits;
// its record per (row, 256-entry vocabulary tile) is (m, S) = the tile's
// maximum and sum_v exp(z_v - m), plus z[target].
//
// Kernel 2 (merge_kernel): one 128-thread block per hidden row folds the
// n_vt tile records in a fixed order that depends on V only: thread g folds
// its leaf of the tree -- the greedy records g, g+128, g+256, ... (an exact
// fold, any order gives the same bits), the log-sum-exp records of the
// contiguous tiles [g n_vt / 128, (g+1) n_vt / 128) -- in ascending order,
// then the 128 partial results combine in a balanced binary tree over g
// (pairs g^1, g^2, ..., g^64). No atomics take part in any logit, token, gap
// or log-probability (the speculative-verify fold's atomicMin is order-free).
//
// Both reductions are written so that a row's bits do not depend on its
// position in the tile or on B: the greedy record is exact (a function of
// the multiset of values), and every floating-point sum of the log-sum-exp
// runs in an order fixed by V alone, the same for every row, with operators
// that are commutative bit for bit.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <cmath>
#include <type_traits>
#include "ptx.cuh"

namespace detlm {

constexpr int kBM = 128;          // vocabulary rows per tile = MMA M = TMEM lanes
constexpr int kRowBytes = 128;    // bytes of K per stage and tile row (one swizzle row)
constexpr int kMaxN = 256;        // largest MMA N
constexpr int kChunkK = 128;      // K elements per accumulation chunk
constexpr int kBlocksPerChunk = kChunkK / 64;   // 128-byte K blocks of 16-bit data
constexpr int kMaxStages = 12;
constexpr int kMaxSlots = 8;
constexpr int kSmemLimit = 232448;  // 227 KB dynamic shared memory per CTA

// MODE_INT: the integer head's wide-batch path. The int8 values of W and h
// are held as fp16 (exact), every 128-element chunk sum is an integer below
// 2^21 (exact in the fp32 accumulator) and the chunk sums are added in
// int32; logits, records and the decision are int32.
// MODE_GATED: the greedy call plus the margin gate of "Greedy Decoding Has a
// Precision Clause" (section on correcting the vulnerable token decisions):
// the record also carries, for the logits rounded to the head's 16-bit
// format, the lowest index of their maximum.
// MODE_SAMPLE: seeded Gumbel-max sampling ("TandemLLM docs, 12 Exactness",
// 12.5): the record is the greedy record of the scores z / T + G, G the
// Gumbel noise of the row's (seed, position) at each vocabulary entry.
enum : int { MODE_GREEDY = 0, MODE_LOGPROB = 1, MODE_INT = 2, MODE_GATED = 3, MODE_SAMPLE = 4 };
enum : int { ERR_TIMEOUT = 1, ERR_TARGET = 2 };

// Kept at 128 bytes or less: with the parameter struct above 128 bytes the
// N = 256 log-prob kernel ran 12 % slower on GB300 (same registers and code
// otherwise). Mode-specific pointers share storage.
struct HeadParams {
  int32_t V, d, B;          // V: vocabulary rows of this head's W
  int32_t N;            // hidden rows per unit (MMA N), multiple of 16, <= kMaxN
  int32_t n_vt, n_nt;   // vocabulary tiles, hidden-row tiles
  int32_t nk;           // K blocks of 128 bytes
  int32_t n_chunks;     // K chunks of kChunkK elements (= pipeline stages per unit)
  int32_t n_slots;      // TMEM chunk slots (ring), N columns each
  int32_t stages;
  uint32_t tmem_cols;
  uint32_t idesc;
  int32_t stall;            // test hook: MMA issuer waits on a dead barrier
  int32_t n_issuers;        // MMA-issuing threads: 1 .. 3 (N <= 128, ring lengths multiples of it)
  float* logits;            // optional fp32 [B, V]
  float* rec_m;             // [B, n_vt] tile maximum
  int32_t* rec_i;           // [B, n_vt] greedy: lowest index of the maximum
  float* rec_s;             // [B, n_vt] greedy: runner-up; logprob: sum exp
  int* err;                 // device error word
  uint64_t timeout_ns;
  union {
    const int32_t* targets;   // logprob: [B]
    int32_t* rec_b;           // gated: [B, n_vt] lowest index of the rounded maximum
    const uint64_t* seeds;    // sample: [B] generator key of each row
  };
  union {
    float* zt;                // logprob: [B] target logit
    const uint64_t* positions;  // sample: [B] position t of each row
  };
  union {
    int32_t round_fp16;       // gated: 1 rounds logits to fp16, 0 to bf16
    float temperature;        // sample: T > 0
    int32_t tma_logits;       // pair kernel: 1 = logits leave through the logits tensor map
  };
  int32_t v_off;            // vocabulary index of this head's first W row
};
static_assert(sizeof(HeadParams) <= 128, "kernel parameter struct above 128 bytes");

// Greedy speculative verify, folded into the merge ("Inference and Decoding",
// section 6: the target scores every drafted position in one pass and keeps
// the drafts while they agree; "TandemLLM docs, 12 Exactness", 12.1: at
// temperature 0 that means equality with the greedy token). Rows are
// request-major, P per request. The block that merges row n = r*P + j lowers
// first_miss[r] to j when its token differs from the draft; the last of the
// request's P blocks to arrive writes accepted[r] = min(first_miss[r], P)
// and puts both workspace words back to their idle values. atomicMin is
// order-free, so the result does not depend on which block finishes last.
struct AcceptArgs {
  int32_t P;
  int32_t R;                // requests (length of each workspace half)
  const int32_t* drafts;    // [R, P]; nullptr: plain greedy call
  int32_t* words;           // workspace: first_miss [R] (kMissNone between calls),
                            // then arrived [R] (0 between calls)
  int32_t* accepted;        // [R] output
};
constexpr int32_t kMissNone = 0x7f7f7f7f;   // what a 0x7f byte fill leaves

__device__ __forceinline__ void accept_fold(const AcceptArgs& a, int n, int32_t tok) {
  if (a.drafts == nullptr) return;
  const int r = n / a.P;
  const int j = n - r * a.P;
  int32_t* first_miss = a.words + r;
  int32_t* arrived = a.words + a.R + r;
  if (tok != a.drafts[n]) atomicMin(first_miss, j);
  __threadfence();
  if (atomicAdd(arrived, 1) == a.P - 1) {
    __threadfence();
    const int32_t f = atomicExch(first_miss, kMissNone);
    *arrived = 0;
    a.accepted[r] = f < a.P ? f : a.P;
  }
}

// 128 bytes or less, like the projection kernel's parameters; the members
// of one mode share storage with another mode's.
struct MergeParams {
  int32_t V, B, n_vt;
  int32_t round_fp16;       // gated: 1 rounds logits to fp16, 0 to bf16
  float tau;                // gated: threshold of the margin
  const float* rec_m;
  const int32_t* rec_i;
  const float* rec_s;
  int32_t* token;
  float* gap;
  int* err;
  union {
    const float* zt;          // logprob: [B] target logit
    const int32_t* rec_b;     // gated: [B, n_vt]
  };
  union {
    const int32_t* targets;   // logprob: [B]
    int32_t* base_token;      // gated: optional [B]
  };
  union {
    float* logp;              // logprob: [B]
    float* margin;            // gated: optional [B]
    float* score_gap;         // sample: optional [B], best minus runner-up score
  };
  AcceptArgs acc;
};
static_assert(sizeof(MergeParams) <= 128, "kernel parameter struct above 128 bytes");

// ------------------------------------------------------------ merge rules
struct Top2 { float m; int32_t i; float s; };   // max, its lowest index, runner-up
struct ITop2 { int32_t m; int32_t i; int32_t s; };  // the same for int32 logits
struct Lse { float m; float S; };               // max, sum exp(z - max)

// Top-2 of a multiset with index tie-break: exact, associative, commutative.
__device__ __forceinline__ Top2 top2_merge(const Top2& a, const Top2& b) {
  const bool aw = (a.m > b.m) || (a.m == b.m && a.i < b.i);
  Top2 r;
  r.m = aw ? a.m : b.m;
  r.i = aw ? a.i : b.i;
  r.s = fmaxf(aw ? a.s : b.s, aw ? b.m : a.m);
  return r;
}

__device__ __forceinline__ ITop2 itop2_merge(const ITop2& a, const ITop2& b) {
  const bool aw = (a.m > b.m) || (a.m == b.m && a.i < b.i);
  ITop2 r;
  r.m = aw ? a.m : b.m;
  r.i = aw ? a.i : b.i;
  r.s = max(aw ? a.s : b.s, aw ? b.m : a.m);
  return r;
}

// (m, S) pairs of log-sum-exp: commutative bit for bit (equal maxima add the
// two sums with one rounding; otherwise the smaller side is scaled).
__device__ __forceinline__ Lse lse_merge(const Lse& a, const Lse& b) {
  Lse hi = a, lo = b;
  if (a.m < b.m) { hi = b; lo = a; }
  if (lo.m == -INFINITY) return hi;
  const float e = (lo.m == hi.m) ? 1.0f : __expf(lo.m - hi.m);
  return Lse{hi.m, fmaf(lo.S, e, hi.S)};
}

__device__ __forceinline__ Top2 shfl_xor(const Top2& x, int b) {
  return Top2{__shfl_xor_sync(0xffffffffu, x.m, b), __shfl_xor_sync(0xffffffffu, x.i, b),
              __shfl_xor_sync(0xffffffffu, x.s, b)};
}
__device__ __forceinline__ ITop2 shfl_xor(const ITop2& x, int b) {
  return ITop2{__shfl_xor_sync(0xffffffffu, x.m, b), __shfl_xor_sync(0xffffffffu, x.i, b),
               __shfl_xor_sync(0xffffffffu, x.s, b)};
}
__device__ __forceinline__ Lse shfl_xor(const Lse& x, int b) {
  return Lse{__shfl_xor_sync(0xffffffffu, x.m, b), __shfl_xor_sync(0xffffffffu, x.S, b)};
}
// Order-preserving 32-bit keys of finite floats (larger float, larger
// unsigned key); key 0 is below every finite value and marks "no value".
__device__ __forceinline__ uint32_t fkey(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float funkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Per-column reduction of one 16-column block over a warp's 32 vocabulary
// rows, through a shared-memory transpose (warp-collective shuffles and
// reductions serialise on this part, a 16-element fold from shared memory
// does not). Lane l ends with column (l & 15) folded over rows 16*(l >> 4) ..
// 16*(l >> 4) + 15 in ascending order; one exchange with lane l ^ 16 then
// covers all 32 rows. The fold order is the same for every column.
constexpr int kXpStride = 17;             // padded row stride (no bank conflicts)
constexpr int kXpWords = 32 * kXpStride;  // per warp

// greedy: exact (max, lowest row index of it, runner-up); invalid rows are -inf
__device__ __forceinline__ Top2 xp_top2(const float* xp, int lane, int v_row0) {
  const int c = lane & 15, h = lane >> 4;
  Top2 t{-INFINITY, INT32_MAX, -INFINITY};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int r = h * 16 + j;
    const float x = xp[r * kXpStride + c];
    if (x > t.m) {              // strictly greater: on a tie the lower row stays
      t.s = t.m;
      t.m = x;
      t.i = v_row0 + r;
    } else {
      t.s = fmaxf(t.s, x);
    }
  }
  return top2_merge(t, shfl_xor(t, 16));
}

// A logit rounded once (to nearest, ties to even) into the head's 16-bit
// format: the value an ordinary bf16 / fp16 projection returns. Rounding is
// monotone, so the rounded maximum of any subset is the rounding of its
// maximum and the rounded runner-up that of its runner-up.
__device__ __forceinline__ float round16(float x, bool fp16) {
  return fp16 ? __half2float(__float2half_rn(x)) : __bfloat162float(__float2bfloat16_rn(x));
}

// Lowest index attaining the maximum of the rounded logits; the value is
// carried only during a fold (elsewhere it is round16 of the record's m).
struct Low16 { float m; int32_t i; };
__device__ __forceinline__ Low16 low16_merge(const Low16& a, const Low16& b) {
  const bool aw = (a.m > b.m) || (a.m == b.m && a.i < b.i);
  return aw ? a : b;
}
__device__ __forceinline__ Low16 shfl_xor(const Low16& x, int b) {
  return Low16{__shfl_xor_sync(0xffffffffu, x.m, b), __shfl_xor_sync(0xffffffffu, x.i, b)};
}

// gated: the greedy fold plus the lowest row index of the rounded maximum
__device__ __forceinline__ Top2 xp_gated(const float* xp, int lane, int v_row0, bool fp16,
                                         int32_t& i16) {
  const int c = lane & 15, h = lane >> 4;
  Top2 t{-INFINITY, INT32_MAX, -INFINITY};
  Low16 b{-INFINITY, INT32_MAX};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int r = h * 16 + j;
    const float x = xp[r * kXpStride + c];
    if (x > t.m) {
      t.s = t.m;
      t.m = x;
      t.i = v_row0 + r;
    } else {
      t.s = fmaxf(t.s, x);
    }
    const float x16 = round16(x, fp16);
    if (x16 > b.m) {            // strictly greater: on a tie the lower row stays
      b.m = x16;
      b.i = v_row0 + r;
    }
  }
  i16 = low16_merge(b, shfl_xor(b, 16)).i;
  return top2_merge(t, shfl_xor(t, 16));
}

// integer head: exact (max, lowest row, runner-up); INT32_MIN marks rows
// outside the vocabulary (|z| is far below 2^31)
__device__ __forceinline__ ITop2 xp_itop2(const int32_t* xp, int lane, int v_row0) {
  const int c = lane & 15, h = lane >> 4;
  ITop2 t{INT32_MIN, INT32_MAX, INT32_MIN};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int r = h * 16 + j;
    const int32_t x = xp[r * kXpStride + c];
    if (x > t.m) {
      t.s = t.m;
      t.m = x;
      t.i = v_row0 + r;
    } else {
      t.s = max(t.s, x);
    }
  }
  return itop2_merge(t, shfl_xor(t, 16));
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplications
// (multipliers 0xD2511F53, 0xCD9E8D57) mixed with the key, which advances by
// the Weyl increments 0x9E3779B9, 0xBB67AE85 between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Sampling score of vocabulary entry v for the row keyed by (seed, t):
// z / T + G, G = -log(-log U), U = (2 (x >> 9) + 1) 2^-24 (exact in fp32,
// strictly inside (0, 1)), x = word (v mod 4) of the Philox block with
// counter (v div 4, t low, t high, 0) and key (seed low, seed high).
__device__ __forceinline__ float sample_score(float z, float T, uint32_t k0, uint32_t k1,
                                              uint32_t t_lo, uint32_t t_hi, uint32_t v) {
  const uint4 w = philox4x32_10(make_uint4(v >> 2, t_lo, t_hi, 0u), k0, k1);
  const uint32_t j = v & 3u;
  const uint32_t x = j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w;
  const float U = __uint2float_rn(((x >> 9) << 1) | 1u) * 5.9604644775390625e-8f;   // 2^-24
  const float G = -logf(-logf(U));
  return __fadd_rn(__fdiv_rn(z, T), G);
}

__device__ __forceinline__ int brev4(int l) {
  return ((l & 1) << 3) | ((l & 2) << 1) | ((l & 4) >> 1) | ((l & 8) >> 3);
}

// ----------------------------------------------------------- shared layout
// Up to N = 128 a pipeline stage holds one whole K chunk (two 128-byte K
// boxes) and four epilogue warps (warps 2..5) hold the running sums. At
// N = 256 a stage holds one K box (so that four stages still fit) and eight
// epilogue warps (warpgroups 1 and 2, two warps per TMEM lane quadrant) hold
// 128 columns each; warpgroup 0 (producer, MMA issuer, two idle warps) gives
// registers to them: launched at 168 per thread, 40 for warpgroup 0 and 232
// for the epilogue (128 * 40 + 256 * 232 = 384 * 168).
__host__ __device__ constexpr int epi_warps_for(int N) { return N > 128 ? 8 : 4; }
__host__ __device__ constexpr int epi_first_warp(int N) { return N > 128 ? 4 : 2; }
__host__ __device__ constexpr int kblocks_per_stage(int N) { return N > 128 ? 1 : 2; }
// Up to N = 128 warps 6 and 7 can issue MMAs too, every second or third K
// chunk round robin: one thread's tcgen05.mma issue rate holds back the TMA
// ring at small N. Each chunk keeps its own MMAs in K order, so the
// arithmetic does not change. The host uses k issuers only when both rings
// the issuers wait on (stages, chunk slots) have lengths that are multiples
// of k: then a chunk and the one a ring length earlier belong to the same
// issuer and every parity wait is unambiguous (the kernel refuses other
// combinations).
__host__ __device__ constexpr int max_mma_issuers(int N) { return N > 128 ? 1 : 3; }
__host__ __device__ constexpr int threads_for(int N) { return N > 128 ? 384 : 256; }
constexpr int kRegsLaunchWide = 168;   // registers per thread at launch, N = 256
constexpr int kRegsWg0Wide = 40;
constexpr int kRegsEpiWide = 232;
static_assert(128 * kRegsWg0Wide + 256 * kRegsEpiWide == 384 * kRegsLaunchWide,
              "register split must equal the launch budget");

struct SmemLayout {
  uint32_t a_bytes, b_bytes, stage_bytes, ctrl_off, red_off, xp_off, total;
};

// Stage s: kblocks_per_stage 128-byte K boxes of the W tile (each [128 rows x
// 128 B], swizzled) followed by as many boxes of the hidden-row tile
// ([N rows x 128 B] each).
__host__ __device__ inline SmemLayout smem_layout(int N, int stages, bool gated = false) {
  SmemLayout L;
  const uint32_t kps = static_cast<uint32_t>(kblocks_per_stage(N));
  L.a_bytes = kps * kBM * kRowBytes;
  L.b_bytes = kps * static_cast<uint32_t>(N) * kRowBytes;
  L.stage_bytes = L.a_bytes + L.b_bytes;
  L.ctrl_off = static_cast<uint32_t>(stages) * L.stage_bytes;
  // barriers: full[S], empty[S], slot_full[kMaxSlots], slot_empty[kMaxSlots],
  // never, drain; then the TMEM address holder and the abort flag
  L.red_off = L.ctrl_off + (2u * stages + 2u * kMaxSlots + 2u) * 8u + 16u;
  // per-quadrant column results: 3 words x 4 quadrants x N columns (gated and
  // sampling: 4 x N more words, the quadrants' lowest indices of the rounded
  // maximum or the columns' sampling keys), then the epilogue warps'
  // transpose areas
  L.xp_off = L.red_off + 3u * 4u * static_cast<uint32_t>(N) * 4u +
             (gated ? 4u * static_cast<uint32_t>(N) * 4u : 0u);
  L.total = L.xp_off + static_cast<uint32_t>(epi_warps_for(N)) * kXpWords * 4u;
  return L;
}

// Barrier over the epilogue threads (barrier 1) that also ORs a predicate, so
// every thread takes the same branch afterwards.
template <int COUNT>
__device__ __forceinline__ bool epi_bar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r) : "r"(static_cast<uint32_t>(pred)), "n"(COUNT) : "memory");
  return r != 0;
}

// ----------------------------------------------------------------- kernel 1
template <int MODE, int NBLK>
__global__ void __launch_bounds__(threads_for(16 * NBLK), 1)
head_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                 const __grid_constant__ CUtensorMap tmH, const HeadParams p) {
  static_assert(MODE == MODE_GREEDY || MODE == MODE_GATED || MODE == MODE_SAMPLE,
                "log-prob runs on head_rows_kernel, the integer wide path on head_pair_kernel");
  constexpr int N = 16 * NBLK;
  constexpr int EW = epi_warps_for(N);          // epilogue warps
  constexpr int ET = 32 * EW;                   // epilogue threads
  constexpr int KPS = kblocks_per_stage(N);     // K boxes per stage
  constexpr int WBLK = NBLK / (EW / 4);         // 16-column blocks per epilogue warp
  constexpr int E0 = epi_first_warp(N);         // first epilogue warp
  const int NWAY = p.n_issuers;                 // MMA-issuing threads (1 .. 3)
  static_assert(N <= kMaxN && NBLK % (EW / 4) == 0 && kBlocksPerChunk % KPS == 0, "shape");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  const SmemLayout L = smem_layout(N, S, MODE == MODE_GATED || MODE == MODE_SAMPLE);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.ctrl_off);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * S + kMaxSlots + b); };
  const uint32_t never_bar = bar0 + 8u * (2 * S + 2 * kMaxSlots);
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 2 * kMaxSlots + 1);
  uint32_t* tmem_holder =
      reinterpret_cast<uint32_t*>(smem + L.ctrl_off + (2 * S + 2 * kMaxSlots + 2) * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* red_m = reinterpret_cast<float*>(smem + L.red_off);
  int32_t* red_i = reinterpret_cast<int32_t*>(red_m + 4 * N);
  float* red_s = reinterpret_cast<float*>(red_i + 4 * N);
  int32_t* red_b = reinterpret_cast<int32_t*>(red_s + 4 * N);   // gated: [4][N]
  uint32_t* skey = reinterpret_cast<uint32_t*>(red_b);     // sample: [4][N] seed lo/hi, t lo/hi
  float* xpose = reinterpret_cast<float*>(smem + L.xp_off);
  const uint32_t smem_base = smem_u32(smem);
  auto sA = [&](int s) { return smem_base + static_cast<uint32_t>(s) * L.stage_bytes; };
  auto sB = [&](int s) { return sA(s) + L.a_bytes; };

  const int kElems = kRowBytes / 2;     // 16-bit elements per 128-byte row
  // stages whose W boxes the producer requests before the previous kernels
  // on the stream have finished (at most the ring, at most this CTA's work)
  auto pre_stages = [&]() {
    const int units = p.n_vt * p.n_nt, per_unit = (p.nk + KPS - 1) / KPS;
    const int n_my = (units - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                     static_cast<int>(gridDim.x);
    return min(S, n_my > 0 ? n_my * per_unit : 0);
  };

  if (threadIdx.x == 0) {
    // this thread is the TMA producer: W is read-only for the life of the
    // head, so the W boxes of the first S stages are requested first --
    // right after their full barriers exist, before the other barriers, the
    // tensor-memory allocation and the wait for the previous kernels on the
    // stream; the hidden rows (which a previous kernel may write) only after
    // that wait
    for (int s = 0; s < S; ++s) mbar_init(full_bar(s), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    const uint64_t pol_w = policy_evict_first();
    const int pre = pre_stages(), spu = (p.nk + KPS - 1) / KPS;
    for (int j = 0; j < pre; ++j) {
      const int u = blockIdx.x + (j / spu) * gridDim.x;
      const int vt = u / p.n_nt, st = j - (j / spu) * spu;
      const int kb0 = st * KPS;
      const int nb = min(KPS, p.nk - kb0);
      mbar_expect_tx(full_bar(j), static_cast<uint32_t>(nb) * (kBM + N) * kRowBytes);
      for (int b = 0; b < nb; ++b)
        tma_load_2d(sA(j) + b * kBM * kRowBytes, &tmW, (kb0 + b) * kElems, vt * kBM,
                    full_bar(j), pol_w);
    }
    for (int s = 0; s < S; ++s) mbar_init(empty_bar(s), 1);
    for (int b = 0; b < p.n_slots; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), EW);
    }
    mbar_init(never_bar, 1);
    mbar_init(drain_bar, static_cast<uint32_t>(NWAY));
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmH);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Launched as a dependent grid: the set-up above overlapped the previous
  // kernels on the stream.
  const uint32_t tmem_base = *tmem_holder;
  const int n_units = p.n_vt * p.n_nt;
  const int spu = (p.nk + KPS - 1) / KPS;   // stages per unit

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if constexpr (EW == 8) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsWg0Wide));
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
        for (int st = 0; st < spu; ++st, ++j) {
          const int kb0 = st * KPS;
          const int nb = min(KPS, p.nk - kb0);
          if (j < pre) {             // W already requested: add the hidden rows
            for (int b = 0; b < nb; ++b)
              tma_load_2d(sB(stage) + b * N * kRowBytes, &tmH, (kb0 + b) * kElems, nt * N,
                          full_bar(stage), pol_h);
            mbar_arrive(full_bar(stage));
          } else {
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full_bar(stage), static_cast<uint32_t>(nb) *
                                                       (kBM + N) * kRowBytes);
            for (int b = 0; b < nb; ++b) {
              tma_load_2d(sA(stage) + b * kBM * kRowBytes, &tmW, (kb0 + b) * kElems, vt * kBM,
                          full_bar(stage), pol_w);
              tma_load_2d(sB(stage) + b * N * kRowBytes, &tmH, (kb0 + b) * kElems, nt * N,
                          full_bar(stage), pol_h);
            }
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
          if ((outstanding >> s) & 1u)
            mbar_wait(full_bar(s), (out_par >> s) & 1u, &zero, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1 || (max_mma_issuers(N) > 1 && warp >= E0 + EW)) {
    // ------------------------------------------------------- MMA issuer
    if constexpr (EW == 8) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsWg0Wide));
    const int which = warp == 1 ? 0 : warp - (E0 + EW) + 1;   // chunks which, which + NWAY, ...
    if (lane == 0 && which < NWAY) {
      constexpr int SPC = kBlocksPerChunk / KPS;     // pipeline stages per chunk
      // ring lengths must be multiples of NWAY (the host only enables two
      // issuers then)
      bool ok = S % NWAY == 0 && p.n_slots % NWAY == 0 && NWAY <= S && NWAY <= p.n_slots;
      if (p.stall) ok = ok && mbar_wait(never_bar, 0, abort_flag, p.timeout_ns);
      if constexpr (max_mma_issuers(N) == 1) {
        // one issuer (N = 256, 40 registers): ring positions by increments
        uint32_t stage = 0, phase = 0, slot = 0, sph = 0;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
          for (int c = 0; c < p.n_chunks && ok; ++c) {
            if (!mbar_wait(acce_bar(slot), sph ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + slot * static_cast<uint32_t>(N);
#pragma unroll
            for (int sc = 0; sc < SPC; ++sc) {
              const int kb0 = c * kBlocksPerChunk + sc * KPS;
              if (kb0 >= p.nk) break;
              if (!mbar_wait(full_bar(stage), phase, abort_flag, p.timeout_ns)) { ok = false; break; }
              tc_fence_after();
              const int nb = min(KPS, p.nk - kb0);
              for (int b = 0; b < nb; ++b) {
                const uint64_t da = sdesc_sw128(sA(stage) + b * kBM * kRowBytes);
                const uint64_t db = sdesc_sw128(sB(stage) + b * N * kRowBytes);
                const bool first = (kb0 + b) == c * kBlocksPerChunk;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  mma_f16(d_tmem, da + 2u * k, db + 2u * k, p.idesc, !(first && k == 0));
              }
              mma_commit(empty_bar(stage));
              if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            mma_commit(accf_bar(slot));
            if (++slot == static_cast<uint32_t>(p.n_slots)) { slot = 0; sph ^= 1u; }
          }
        }
      } else {
        // N <= 128: one stage per chunk; issuer `which` takes chunks which,
        // which + NWAY, ... and its ring positions advance by NWAY (both
        // ring lengths are multiples of NWAY, so no position is shared
        // with the other issuer in between)
        static_assert(SPC == 1, "one pipeline stage per chunk");
        uint32_t stage = which, phase = 0, slot = which, sph = 0;
        int turn = 0;                                // this chunk's issuer
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
          for (int c = 0; c < p.n_chunks && ok; ++c) {
            if (turn == which) {
              if (!mbar_wait(acce_bar(slot), sph ^ 1u, abort_flag, p.timeout_ns)) { ok = false; break; }
              if (!mbar_wait(full_bar(stage), phase, abort_flag, p.timeout_ns)) { ok = false; break; }
              tc_fence_after();
              const uint32_t d_tmem = tmem_base + slot * static_cast<uint32_t>(N);
              const int kb0 = c * kBlocksPerChunk;
              const int nb = min(KPS, p.nk - kb0);
              for (int b = 0; b < nb; ++b) {
                const uint64_t da = sdesc_sw128(sA(stage) + b * kBM * kRowBytes);
                const uint64_t db = sdesc_sw128(sB(stage) + b * N * kRowBytes);
#pragma unroll
                for (int k = 0; k < 4; ++k)   // K = 16 per MMA: 32 bytes = 2 descriptor units
                  mma_f16(d_tmem, da + 2u * k, db + 2u * k, p.idesc, !(b == 0 && k == 0));
              }
              mma_commit(empty_bar(stage));
              mma_commit(accf_bar(slot));
              stage += static_cast<uint32_t>(NWAY);
              if (stage >= static_cast<uint32_t>(S)) { stage -= static_cast<uint32_t>(S); phase ^= 1u; }
              slot += static_cast<uint32_t>(NWAY);
              if (slot >= static_cast<uint32_t>(p.n_slots)) { slot -= static_cast<uint32_t>(p.n_slots); sph ^= 1u; }
            }
            if (++turn == NWAY) turn = 0;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, ERR_TIMEOUT);
      }
      // every MMA this thread issued has finished before TMEM is released
      mma_commit(drain_bar);
      const int zero = 0;
      mbar_wait(drain_bar, 0, &zero, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= E0 && warp < E0 + EW) {
    // --------------------------------------------------------- epilogue
    if constexpr (EW == 8) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kRegsEpiWide));
    grid_dep_wait();          // outputs and records: only after the previous kernels
    const int q = warp & 3;                    // TMEM lane quadrant of this warp
    const int g = (warp - E0) >> 2;            // column half (eight epilogue warps)
    const int et = threadIdx.x - 32 * E0;      // 0 .. ET-1
    const int row = q * 32 + lane;             // vocabulary row within the tile
    const uint32_t tlane = static_cast<uint32_t>(q * 32) << 16;
    float* xp = xpose + (warp - E0) * kXpWords;
    uint32_t slot = 0, sph = 0;
    bool failed = false;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const int vt = u / p.n_nt, nt = u - (u / p.n_nt) * p.n_nt;
      float acc[WBLK][16];
      for (int c = 0; c < p.n_chunks; ++c) {
        const uint32_t cur = slot, cph = sph;
        if (++slot == static_cast<uint32_t>(p.n_slots)) { slot = 0; sph ^= 1u; }
        if (!failed && !mbar_wait(accf_bar(cur), cph, abort_flag, p.timeout_ns)) {
          failed = true;
          *abort_flag = 1;
        }
        if (failed) continue;
        tc_fence_after();
        const uint32_t sbase = tmem_base + tlane + cur * static_cast<uint32_t>(N) +
                               static_cast<uint32_t>(g * WBLK * 16);
        // groups of up to four 16-column loads, one wait each; the chunk
        // sums are added with packed round-to-nearest fp32 adds
        constexpr int kG = WBLK < 4 ? WBLK : 4;
#pragma unroll
        for (int b0 = 0; b0 < WBLK; b0 += kG) {
          uint32_t r[kG][16];
#pragma unroll
          for (int k = 0; k < kG; ++k) tmem_ld16(sbase + (b0 + k) * 16, r[k]);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < kG; ++k) {
            const int bb = b0 + k;
            if (c == 0) {
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[bb][i] = __uint_as_float(r[k][i]);
            } else {
#pragma unroll
              for (int i = 0; i < 16; i += 2)
                add2_rn(acc[bb][i], acc[bb][i + 1], __uint_as_float(r[k][i]),
                        __uint_as_float(r[k][i + 1]));
            }
          }
        }
        tc_fence_before();   // slot fully read: hand it back to the MMA warp
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(cur));
      }
      if (epi_bar_or<ET>(failed || *abort_flag)) {
        if (et == 0) { *abort_flag = 1; atomicOr(p.err, ERR_TIMEOUT); }
        break;
      }
      const int v = vt * kBM + row;
      const bool vok = v < p.V;
      const int n0 = nt * N;
      const int vg0 = p.v_off + vt * kBM + q * 32;   // vocabulary index of this warp's row 0
      if constexpr (MODE == MODE_SAMPLE) {
        // the unit's column keys, once per unit (ordered before the reads by
        // this barrier, after the previous unit's reads by the one above)
        for (int c = et; c < N; c += ET) {
          const int n = n0 + c;
          const uint64_t sd = n < p.B ? p.seeds[n] : 0ull;
          const uint64_t tp = n < p.B ? p.positions[n] : 0ull;
          skey[c] = static_cast<uint32_t>(sd);
          skey[N + c] = static_cast<uint32_t>(sd >> 32);
          skey[2 * N + c] = static_cast<uint32_t>(tp);
          skey[3 * N + c] = static_cast<uint32_t>(tp >> 32);
        }
        named_bar_sync(1, ET);
      }
#pragma unroll
      for (int bb = 0; bb < WBLK; ++bb) {
        const int c0 = (g * WBLK + bb) * 16;
        if (p.logits != nullptr && vok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = n0 + c0 + i;
            if (n < p.B) p.logits[static_cast<size_t>(n) * p.V + v] = acc[bb][i];
          }
        }
        if constexpr (MODE == MODE_SAMPLE) {
          // logits to this lane's transpose row first, then the scores in
          // place (a rolled loop: the noise is long code)
#pragma unroll
          for (int i = 0; i < 16; ++i) xp[lane * kXpStride + i] = acc[bb][i];
#pragma unroll 1
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            float x = -INFINITY;
            if (vok && n0 + c < p.B)
              x = sample_score(xp[lane * kXpStride + i], p.temperature, skey[c], skey[N + c],
                               skey[2 * N + c], skey[3 * N + c],
                               static_cast<uint32_t>(p.v_off + v));
            xp[lane * kXpStride + i] = x;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) xp[lane * kXpStride + i] = vok ? acc[bb][i] : -INFINITY;
        }
        __syncwarp();
        if constexpr (MODE == MODE_GREEDY || MODE == MODE_SAMPLE) {
          const Top2 t = xp_top2(xp, lane, vg0);
          if (lane < 16) {
            red_m[q * N + c0 + lane] = t.m;
            red_i[q * N + c0 + lane] = t.i;
            red_s[q * N + c0 + lane] = t.s;
          }
        } else {
          static_assert(MODE == MODE_GATED, "the log-prob call runs on head_rows_kernel");
          int32_t i16;
          const Top2 t = xp_gated(xp, lane, vg0, p.round_fp16 != 0, i16);
          if (lane < 16) {
            red_m[q * N + c0 + lane] = t.m;
            red_i[q * N + c0 + lane] = t.i;
            red_s[q * N + c0 + lane] = t.s;
            red_b[q * N + c0 + lane] = i16;
          }
        }
        __syncwarp();
      }
      named_bar_sync(1, ET);
      // fixed combination of the four 32-row quadrants: (q0 . q1) . (q2 . q3)
      for (int c = et; c < N; c += ET) {
        const int n = n0 + c;
        if (n >= p.B) continue;
        const size_t o = static_cast<size_t>(n) * p.n_vt + vt;   // records [B][n_vt]
        {
          Top2 t[4];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            t[qq] = Top2{red_m[qq * N + c], red_i[qq * N + c], red_s[qq * N + c]};
          const Top2 r = top2_merge(top2_merge(t[0], t[1]), top2_merge(t[2], t[3]));
          p.rec_m[o] = r.m;
          p.rec_i[o] = r.i;
          p.rec_s[o] = r.s;
          if constexpr (MODE == MODE_GATED) {
            const bool f16 = p.round_fp16 != 0;
            Low16 b[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) b[qq] = Low16{round16(t[qq].m, f16), red_b[qq * N + c]};
            p.rec_b[o] = low16_merge(low16_merge(b[0], b[1]), low16_merge(b[2], b[3])).i;
          }
        }
      }
      named_bar_sync(1, ET);
    }
    if (failed && et == 0) atomicOr(p.err, ERR_TIMEOUT);
  } else {
    // warps 2 and 3 of warpgroup 0 (N = 256 only): no role, fewer registers
    if constexpr (EW == 8) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsWg0Wide));
  }

  tc_fence_before();
  __syncthreads();
  // the merge kernel may be scheduled now: triggered at the end, not after
  // the set-up, because B waiting merge blocks would share the SMs' issue
  // slots with this kernel for its whole run
  grid_dep_launch();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// ----------------------------------------------------------------- kernel 2
// gap in bf16 ulps of the winner: (m - s) * 2^(7 - E), E = floor(log2|m|)
// clamped at -126, evaluated in double (exact difference of two floats,
// exact power-of-two scaling) and rounded once to float.
__device__ __forceinline__ float gap_ulp_bf16(float m, float s) {
  const uint32_t eb = (__float_as_uint(m) >> 23) & 0xFFu;
  const int E = static_cast<int>(eb > 1u ? eb : 1u) - 127;
  const double scale = __longlong_as_double(static_cast<long long>(1023 + 7 - E) << 52);
  return static_cast<float>((static_cast<double>(m) - static_cast<double>(s)) * scale);
}

// Balanced-tree combination of one value per thread over a 128-thread block
// (levels g^1 .. g^16 by shuffles, then (w0 . w1) . (w2 . w3) across warps);
// the result is valid in thread 0.
template <typename T, typename M>
__device__ __forceinline__ T block_tree128(T x, M merge_fn, T* smem4) {
#pragma unroll
  for (int b = 1; b < 32; b <<= 1) x = merge_fn(x, shfl_xor(x, b));
  if ((threadIdx.x & 31) == 0) smem4[threadIdx.x >> 5] = x;
  __syncthreads();
  return merge_fn(merge_fn(smem4[0], smem4[1]), merge_fn(smem4[2], smem4[3]));
}

constexpr int kMergeThreads = 128;
constexpr int kMergeBatch = 8;     // records loaded per thread before folding

// The log-sum-exp tree over a row's tile records: 128 leaves, leaf g holding
// the tiles [leaf_lo(g, n), leaf_lo(g + 1, n)) of the n tiles, folded in
// ascending order; the leaves combine in a balanced binary tree (block_tree128).
// The shape is a function of n alone. A run of whole leaves is a run of whole
// tiles, so a head cut into P = 2, 4, ..., 128 vocabulary shards on leaf
// boundaries (shard r: leaves [128 r / P, 128 (r + 1) / P)) computes subtrees
// of this very tree, and combining the shards' roots in a balanced tree gives
// the same bits (shard_kernels.cuh).
constexpr int kLeaves = kMergeThreads;
__host__ __device__ inline int leaf_lo(int g, int n) {
  return static_cast<int>((static_cast<int64_t>(g) * n) / kLeaves);
}

// Fold of tiles [t0, t1) of one row's (m, S) records, in ascending order,
// starting from the identity (a no-op of lse_merge, bit for bit).
__device__ __forceinline__ Lse lse_fold_range(const float* rm, const float* rs, int t0, int t1) {
  Lse acc{-INFINITY, 0.0f};
  for (int t = t0; t < t1; t += kMergeBatch) {
    Lse r[kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)
      r[j] = t + j < t1 ? Lse{rm[t + j], rs[t + j]} : Lse{-INFINITY, 0.0f};
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) acc = lse_merge(acc, r[j]);
  }
  return acc;
}

template <int MODE>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  grid_dep_launch(); // the next call's kernel 1 may start (it prefetches only W)
  grid_dep_wait();   // records of kernel 1 are complete and visible
  const int n = blockIdx.x;
  const int g = threadIdx.x;
  const size_t base = static_cast<size_t>(n) * p.n_vt;
  if constexpr (MODE == MODE_GREEDY || MODE == MODE_SAMPLE) {
    __shared__ Top2 part[4];
    Top2 acc{-INFINITY, INT32_MAX, -INFINITY};
    for (int t0 = g; t0 < p.n_vt; t0 += kMergeThreads * kMergeBatch) {
      Top2 r[kMergeBatch];
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        const int t = t0 + j * kMergeThreads;
        r[j] = t < p.n_vt ? Top2{p.rec_m[base + t], p.rec_i[base + t], p.rec_s[base + t]}
                          : Top2{-INFINITY, INT32_MAX, -INFINITY};
      }
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) acc = top2_merge(acc, r[j]);
    }
    const Top2 tot = block_tree128(acc, top2_merge, part);
    if (g == 0) {
      p.token[n] = tot.i;
      if constexpr (MODE == MODE_GREEDY) {
        p.gap[n] = gap_ulp_bf16(tot.m, tot.s);
      } else {
        if (p.score_gap != nullptr) p.score_gap[n] = __fsub_rn(tot.m, tot.s);
      }
      accept_fold(p.acc, n, tot.i);
    }
  } else if constexpr (MODE == MODE_GATED) {
    // the greedy fold and, beside it, the lowest index of the rounded maximum
    __shared__ Top2 part[4];
    __shared__ Low16 partb[4];
    const bool f16 = p.round_fp16 != 0;
    Top2 acc{-INFINITY, INT32_MAX, -INFINITY};
    Low16 accb{-INFINITY, INT32_MAX};
    for (int t0 = g; t0 < p.n_vt; t0 += kMergeThreads * kMergeBatch) {
      Top2 r[kMergeBatch];
      Low16 rb[kMergeBatch];
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        const int t = t0 + j * kMergeThreads;
        r[j] = t < p.n_vt ? Top2{p.rec_m[base + t], p.rec_i[base + t], p.rec_s[base + t]}
                          : Top2{-INFINITY, INT32_MAX, -INFINITY};
        rb[j] = t < p.n_vt ? Low16{round16(r[j].m, f16), p.rec_b[base + t]}
                           : Low16{-INFINITY, INT32_MAX};
      }
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        acc = top2_merge(acc, r[j]);
        accb = low16_merge(accb, rb[j]);
      }
    }
    const Top2 tot = block_tree128(acc, top2_merge, part);
    const Low16 totb = block_tree128(accb, low16_merge, partb);
    if (g == 0) {
      // margin of the rounded logits: round16 of the top two values
      const float margin = __fsub_rn(round16(tot.m, f16), round16(tot.s, f16));
      const bool fired = margin < p.tau;
      const int32_t tok = fired ? tot.i : totb.i;
      p.token[n] = tok;
      p.gap[n] = gap_ulp_bf16(tot.m, tot.s);
      if (p.base_token != nullptr) p.base_token[n] = totb.i;
      if (p.margin != nullptr) p.margin[n] = margin;
      accept_fold(p.acc, n, tok);
    }
  } else {
    __shared__ Lse part[4];
    const Lse acc = lse_fold_range(p.rec_m + base, p.rec_s + base, leaf_lo(g, p.n_vt),
                                   leaf_lo(g + 1, p.n_vt));
    const Lse tot = block_tree128(acc, lse_merge, part);
    if (g == 0) {
      const int tg = p.targets[n];
      if (tg < 0 || tg >= p.V) {
        p.logp[n] = __int_as_float(0x7fc00000);
        atomicOr(p.err, ERR_TARGET);
      } else {
        p.logp[n] = p.zt[n] - (tot.m + logf(tot.S));
      }
    }
  }
}

}  // namespace detlm
