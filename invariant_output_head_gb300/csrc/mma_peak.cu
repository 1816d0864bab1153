// mma_peak.cu -- dense throughput of the tensor-core instruction the heads
// run on (tcgen05.mma.cta_group::1.kind::f16, fp16 operands from shared
// memory, fp32 accumulator in tensor memory, M = 128, N = 256, K = 16): the
// roofline denominator of the integer head's wide path, which computes its
// exact int8 products on this instruction (sm_103a has no tcgen05 integer
// MMA). A measurement aid for the benchmark, not part of the head's C ABI.
//
// One CTA per SM; one thread issues `iters` x 4 MMAs back to back on operands
// already in shared memory (no loads), into one 256-column accumulator, then
// waits (bounded) for them to complete. Timed with CUDA events by the caller.
#include <cuda_runtime.h>
#include <cstdint>
#include <cstring>

#include "ptx.cuh"

namespace {

using namespace detlm;

constexpr int kM = 128, kN = 256;
constexpr uint32_t kABytes = kM * 128;   // one 64-element K box of A (fp16)
constexpr uint32_t kBBytes = kN * 128;   // one 64-element K box of B
constexpr uint64_t kLimitNs = 2000000000ull;

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kABytes + kBBytes);
  uint32_t* holder = reinterpret_cast<uint32_t*>(bar + 1);
  // operands: small fp16 integers (their values do not change the rate)
  for (uint32_t i = threadIdx.x; i < (kABytes + kBBytes) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(smem)[i] = 0x3C003C00u ^ ((i & 7u) << 10);   // 1.0, 2.0, ...
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(bar), 1);
    fence_mbar_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(holder), 256u);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_f16(0u, kM, kN);
    const uint64_t da = sdesc_sw128(smem_u32(smem));
    const uint64_t db = sdesc_sw128(smem_u32(smem + kABytes));
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int k = 0; k < 4; ++k) mma_f16(tmem, da + 2u * k, db + 2u * k, idesc, (it | k) != 0);
    }
    mma_commit(smem_u32(bar));
    const int zero = 0;
    if (!mbar_wait(smem_u32(bar), 0, &zero, kLimitNs)) atomicOr(err, 1);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem, 256u);
  }
}

}  // namespace

// Run the probe on `ctas` CTAs (one per SM) with `iters` K = 64 steps each,
// timed by CUDA events on the default stream. Returns 0 and the rate in
// TFLOP/s (2 M N K per MMA) in *tflops; -1 on a CUDA error or a wait that ran
// out.
extern "C" int detlm_mma_f16_peak(int ctas, int iters, double* tflops) {
  if (ctas < 1 || iters < 1 || tflops == nullptr) return -1;
  const size_t smem = kABytes + kBBytes + 64 + 1024;
  if (cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return -1;
  int* err = nullptr;
  if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return -1;
  cudaMemset(err, 0, sizeof(int));
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  mma_peak_kernel<<<ctas, 128, smem>>>(iters / 8 + 1, err);   // warm-up
  cudaEventRecord(a);
  mma_peak_kernel<<<ctas, 128, smem>>>(iters, err);
  cudaEventRecord(b);
  cudaError_t e = cudaEventSynchronize(b);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
  int h_err = 1;
  if (e == cudaSuccess) e = cudaMemcpy(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  cudaFree(err);
  if (e != cudaSuccess || h_err != 0 || ms <= 0.0f) return -1;
  const double flops = 2.0 * kM * kN * 16.0 * 4.0 * iters * ctas;
  *tflops = flops / (ms * 1e-3) / 1e12;
  return 0;
}
