// quant_kernels.cuh -- the integer front end of the int8 head.
//
// A float row x (bf16, fp16 or fp32) becomes int8 with a per-row dyadic
// multiplier, computed from that row's own values only ("Eliminating
// Nondeterminism in LLM Inference with Integer-Only Arithmetic", section
// DetLLM: every tensor carries a scale made of an integer multiplier and a
// shift with one fixed rounding rule; each token is quantized from its own
// values, so its bits cannot depend on the batch):
//   amax = max |x|, E = floor(log2 amax), S = E + 8,
//   M = floor(127 * 2^S / amax)          (15 bits, in [16256, 32512]),
//   q = round-half-even(x * M / 2^S)      (in [-127, 127]; amax -> +-127).
// Every step is integer arithmetic on the exact significand and exponent of
// the input: |x| = X * 2^e with X < 2^24, so X * M < 2^39 and the rounding
// shift is exact. An all-zero row gives q = 0, M = 0, S = 0.
#pragma once
#include <cstdint>
#include "ptx.cuh"

namespace detlm {

constexpr int kQThreads = 256;
enum : int { QF_BF16 = 0, QF_FP16 = 1, QF_FP32 = 3 };   // the header's dtype values

struct QuantParams {
  const void* x;
  int32_t fmt;
  int64_t d;
  int8_t* q;          // [B, d]
  int32_t* mult;      // [B] M
  int32_t* shift;     // [B] S
};

// magnitude bits (sign cleared) of element k of a row
__device__ __forceinline__ uint32_t q_load_bits(const void* row, int fmt, int64_t k) {
  if (fmt == QF_FP32) return reinterpret_cast<const uint32_t*>(row)[k];
  return reinterpret_cast<const uint16_t*>(row)[k];
}
__device__ __forceinline__ uint32_t q_sign_mask(int fmt) {
  return fmt == QF_FP32 ? 0x80000000u : 0x8000u;
}

// |x| = X * 2^e from the magnitude bits (finite values; subnormals included)
__device__ __forceinline__ void q_decode(uint32_t mag, int fmt, uint32_t& X, int& e) {
  uint32_t ex, man;
  int mbits, bias;
  if (fmt == QF_BF16) {
    ex = mag >> 7; man = mag & 0x7Fu; mbits = 7; bias = 127;
  } else if (fmt == QF_FP16) {
    ex = mag >> 10; man = mag & 0x3FFu; mbits = 10; bias = 15;
  } else {
    ex = mag >> 23; man = mag & 0x7FFFFFu; mbits = 23; bias = 127;
  }
  X = ex ? (man | (1u << mbits)) : man;
  e = static_cast<int>(ex ? ex : 1u) - bias - mbits;
}

__global__ void __launch_bounds__(kQThreads) quantize_rows_kernel(const QuantParams p) {
  // launched as a dependent grid: the int8 projection that follows may
  // start at once (it prefetches only W before waiting for this grid); x and
  // q may be in use by the previous kernels on the stream until they complete
  grid_dep_launch();
  grid_dep_wait();
  const int64_t n = blockIdx.x;
  const int fmt = p.fmt;
  const size_t eb = fmt == QF_FP32 ? 4 : 2;
  const void* row = static_cast<const uint8_t*>(p.x) + static_cast<size_t>(n) * p.d * eb;
  const uint32_t smask = q_sign_mask(fmt);
  // pass 1: the largest magnitude (integer max of the magnitude bits, which
  // orders finite values of one format; order-free)
  uint32_t mx = 0;
  for (int64_t k = threadIdx.x; k < p.d; k += kQThreads)
    mx = max(mx, q_load_bits(row, fmt, k) & ~smask);
  mx = __reduce_max_sync(0xffffffffu, mx);
  __shared__ uint32_t wmax[kQThreads / 32];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
  __syncthreads();
  uint32_t amax = 0;
#pragma unroll
  for (int w = 0; w < kQThreads / 32; ++w) amax = max(amax, wmax[w]);
  int8_t* qrow = p.q + static_cast<size_t>(n) * p.d;
  if (amax == 0) {
    for (int64_t k = threadIdx.x; k < p.d; k += kQThreads) qrow[k] = 0;
    if (threadIdx.x == 0) { p.mult[n] = 0; p.shift[n] = 0; }
    return;
  }
  uint32_t A;
  int ea;
  q_decode(amax, fmt, A, ea);
  const int bl = 32 - __clz(A);                     // bit length of A
  const int S = ea + bl - 1 + 8;                    // E + 8
  const uint64_t M = (uint64_t{127} << (bl + 7)) / A;
  if (threadIdx.x == 0) { p.mult[n] = static_cast<int32_t>(M); p.shift[n] = S; }
  // pass 2: q = RNE(X * M * 2^(e - S)) with the sign of x
  for (int64_t k = threadIdx.x; k < p.d; k += kQThreads) {
    const uint32_t bits = q_load_bits(row, fmt, k);
    uint32_t X;
    int e;
    q_decode(bits & ~smask, fmt, X, e);
    const uint64_t P = static_cast<uint64_t>(X) * M;
    const int sh = S - e;
    uint32_t qm;
    if (P == 0 || sh >= 64) {
      qm = 0;                                        // below half a step
    } else if (sh <= 0) {
      qm = static_cast<uint32_t>(P << (-sh));       // at most 127, so -sh <= 6
    } else {
      const uint64_t q0 = P >> sh;
      const uint64_t rem = P & ((uint64_t{1} << sh) - 1);
      const uint64_t half = uint64_t{1} << (sh - 1);
      qm = static_cast<uint32_t>(q0 + ((rem > half || (rem == half && (q0 & 1))) ? 1 : 0));
    }
    const int32_t qv = (bits & smask) ? -static_cast<int32_t>(qm) : static_cast<int32_t>(qm);
    qrow[k] = static_cast<int8_t>(qv);
  }
}

}  // namespace detlm
