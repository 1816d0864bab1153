// detlm_head.cu -- the C ABI of the output-head library (host side).
//
// Validates every argument on the host before any GPU work, owns the TMA
// descriptor of W, the split-V record workspace and the device error word,
// encodes the TMA descriptor of h per call (a pure host computation), and
// launches kernel 1 (projection + per-tile records) and kernel 2 (fixed-order
// merge, launched with programmatic dependent launch so that its launch
// overlaps kernel 1's tail).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "detlm_head.h"
#include "head_kernels.cuh"
#include "int8_kernels.cuh"
#include "quant_kernels.cuh"
#include "rows_kernels.cuh"
#include "pair_kernels.cuh"
#include "shard_kernels.cuh"

using namespace detlm;

struct detlm_head {
  int device = 0;
  int dtype = 0;
  int64_t V = 0, d = 0;      // V: rows of this head's W
  // vocabulary shard r of P: this head's rows are [v_off, v_off + V) of a
  // vocabulary of V_total (P = 1: the whole head)
  int64_t v_off = 0, V_total = 0;
  int P = 1, rank = 0;
  const void* W = nullptr;
  CUtensorMap tmW;
  int n_vt = 0, nk = 0, num_sms = 0;
  int rows_pairs = 0;        // CTA pairs of the rows kernel that fit at once (0: not asked yet)
  int wide_pairs = 0;        // the same for the wide greedy kernel
  int* d_err = nullptr;
  int* err_host = nullptr;   // pinned word the error word is read into
  // where the GPU has native atomics on host memory (Grace with NVLink-C2C),
  // the error word itself is a mapped pinned host word: d_err is its device
  // address and the check reads it without a copy
  int* err_mapped = nullptr;
  // split-V record workspace
  void* ws = nullptr;
  int64_t ws_B = 0;
  // device staging for the *_host calls
  void* stage = nullptr;
  size_t stage_bytes = 0;
  // the *_host_async calls: the hidden rows staged on the call's stream, the
  // outputs in two alternating slots copied to the host on the handle's own
  // copy stream (so a call's device-to-host copy overlaps the next call's
  // kernels); done[k]: slot k's kernels finished, freed[k]: its copy did
  void* a_in = nullptr;
  size_t a_in_bytes = 0;
  void* a_out[2] = {nullptr, nullptr};
  size_t a_out_bytes = 0;
  int a_next = 0;
  cudaStream_t a_copy = nullptr;
  cudaEvent_t a_done[2] = {nullptr, nullptr}, a_freed[2] = {nullptr, nullptr};
  // integer head, wide batches: fp16 copy of W (made at the first such call)
  // and the call's hidden rows in fp16
  void* W16 = nullptr;
  CUtensorMap tmW16;
  void* h16 = nullptr;
  size_t h16_bytes = 0;
  // verify: per-request workspace (first_miss, arrived) and the arguments of
  // the call in progress (drafts == nullptr outside detlm_head_verify)
  int32_t* vws = nullptr;
  int64_t vws_R = 0;
  AcceptArgs acc{};
  // integer front end: the quantized rows and their multipliers and shifts
  void* q8 = nullptr;
  size_t q8_bytes = 0;
  // test hook and timing hook
  int stall = 0;
  uint64_t timeout_ns = 2000000000ull;
  cudaEvent_t t_start = nullptr, t_stop = nullptr;
};

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

size_t elem_bytes(int dtype) { return dtype == DETLM_INT8 ? 1 : 2; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 2-D K-major tensor map: dims {d, rows}, box {128 bytes of K, box_rows},
// 128-byte swizzle, zero fill outside the tensor.
bool encode_2d(CUtensorMap* m, int dtype, const void* base, int64_t d, int64_t rows,
               uint32_t box_rows) {
  const CUtensorMapDataType t = dtype == DETLM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                : dtype == DETLM_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const size_t eb = elem_bytes(dtype);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * eb};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / eb), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, t, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Hidden rows per MMA (N): B rounded up to 16 up to 128; above that 256
// (several column tiles past 256). The result of a row does not depend on N.
int cols_for(int64_t B) {
  if (B > 128) return 256;
  const int n = static_cast<int>((B + 15) / 16) * 16;
  return n < 16 ? 16 : n;
}

uint32_t tmem_cols_for(int ncols) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(ncols)) c <<= 1;
  return c;
}

// Chunk slots: as many as fit 512 TMEM columns, at most kMaxSlots. The
// slot count changes no arithmetic (every chunk starts from zero).
int slots_for(int N) {
  int s = 512 / N;
  return s > kMaxSlots ? kMaxSlots : s;
}

int stages_for(int N, bool gated = false) {
  const SmemLayout L1 = smem_layout(N, 1, gated);
  const uint32_t fixed = L1.total - L1.stage_bytes + 2u * kMaxStages * 8u + 1024u;
  int s = static_cast<int>((kSmemLimit - fixed) / L1.stage_bytes);
  if (s > kMaxStages) s = kMaxStages;
  return s;
}

// MMA-issuing threads: the most the kernel allows (N <= 128: 3) that divides
// the stage ring's length and leaves at least that many chunk slots; the slot
// ring is then cut to a multiple of it (the kernel's parity waits rely on
// both).
int issuers_for(int N, int stages, int* slots) {
  for (int k = max_mma_issuers(N); k > 1; --k) {
    if (stages % k == 0 && *slots >= k) {
      *slots -= *slots % k;
      return k;
    }
  }
  return 1;
}

int status_from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return DETLM_OK;
  if (e == cudaErrorMemoryAllocation) return DETLM_ENOMEM;
  return DETLM_ECUDA;
}

// workspace: rec_m, rec_i, rec_s, rec_b [B, n_vt] and zt [B], 256-byte
// aligned parts, laid out for the allocated row count
size_t ws_part(int64_t n) { return (static_cast<size_t>(n) * 4 + 255) & ~static_cast<size_t>(255); }
size_t ws_bytes_for(const detlm_head* h, int64_t B) {
  return 4 * ws_part(static_cast<int64_t>(h->n_vt) * B) + ws_part(B);
}

int ensure_ws(detlm_head* h, int64_t B, cudaStream_t stream) {
  if (B <= h->ws_B) return DETLM_OK;
  if (h->ws != nullptr) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return status_from_cuda(e);
    cudaFree(h->ws);
    h->ws = nullptr;
    h->ws_B = 0;
  }
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, ws_bytes_for(h, B));
  if (e != cudaSuccess) return status_from_cuda(e);
  h->ws = p;
  h->ws_B = B;
  return DETLM_OK;
}

struct WsView { float* m; int32_t* i; float* s; int32_t* b; float* zt; };
WsView ws_view(const detlm_head* h) {
  uint8_t* b = static_cast<uint8_t*>(h->ws);
  const size_t part = ws_part(static_cast<int64_t>(h->n_vt) * h->ws_B);
  WsView w;
  w.m = reinterpret_cast<float*>(b);
  w.i = reinterpret_cast<int32_t*>(b + part);
  w.s = reinterpret_cast<float*>(b + 2 * part);
  w.b = reinterpret_cast<int32_t*>(b + 3 * part);
  w.zt = reinterpret_cast<float*>(b + 4 * part);
  return w;
}

// verify workspace for R requests: first_miss [R] filled with kMissNone
// bytes, arrived [R] zero; the merge puts both back after every call
int ensure_vws(detlm_head* h, int64_t R, cudaStream_t stream) {
  if (R <= h->vws_R) return DETLM_OK;
  if (h->vws != nullptr) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return status_from_cuda(e);
    cudaFree(h->vws);
    h->vws = nullptr;
    h->vws_R = 0;
  }
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, static_cast<size_t>(R) * 8);
  if (e != cudaSuccess) return status_from_cuda(e);
  e = cudaMemsetAsync(p, 0x7f, static_cast<size_t>(R) * 4, stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(static_cast<int32_t*>(p) + R, 0, static_cast<size_t>(R) * 4, stream);
  if (e != cudaSuccess) {
    cudaFree(p);
    return status_from_cuda(e);
  }
  h->vws = static_cast<int32_t*>(p);
  h->vws_R = R;
  return DETLM_OK;
}

// One-time set-up of a kernel on the current device: its opt-in dynamic
// shared memory (the most any launch asks for) and, where want_regs > 0, a
// check of the register count its register split assumes. Later launches on
// the device skip these runtime calls (a bit per device; up to 64 devices,
// beyond that the set-up runs on every launch).
template <auto KERN>
cudaError_t prepare_kernel(int want_regs) {
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 64;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (ready.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  if (want_regs > 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, KERN);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != want_regs) return cudaErrorInvalidConfiguration;
  }
  cudaError_t e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemLimit);
  if (e != cudaSuccess) return e;
  ready.fetch_or(bit, std::memory_order_release);
  return cudaSuccess;
}

// Launch kernel 1 for N = 16 * nblk as a programmatic dependent of the
// previous kernel on the stream (its prologue overlaps that kernel's tail).
template <int MODE, int NBLK>
cudaError_t launch_gemm_n(const CUtensorMap& tmW, const CUtensorMap& tmH, const HeadParams& p,
                          int grid, size_t smem, cudaStream_t stream) {
  auto kern = head_gemm_kernel<MODE, NBLK>;
  // the wide kernel's register split assumes exactly its launch budget
  cudaError_t e = prepare_kernel<head_gemm_kernel<MODE, NBLK>>(
      threads_for(16 * NBLK) == 384 ? kRegsLaunchWide : 0);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(threads_for(16 * NBLK));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmW, tmH, p);
}

template <int MODE>
cudaError_t launch_gemm(const CUtensorMap& tmW, const CUtensorMap& tmH, const HeadParams& p,
                        int grid, size_t smem, cudaStream_t stream) {
  switch (p.N / 16) {
    case 1: return launch_gemm_n<MODE, 1>(tmW, tmH, p, grid, smem, stream);
    case 2: return launch_gemm_n<MODE, 2>(tmW, tmH, p, grid, smem, stream);
    case 3: return launch_gemm_n<MODE, 3>(tmW, tmH, p, grid, smem, stream);
    case 4: return launch_gemm_n<MODE, 4>(tmW, tmH, p, grid, smem, stream);
    case 5: return launch_gemm_n<MODE, 5>(tmW, tmH, p, grid, smem, stream);
    case 6: return launch_gemm_n<MODE, 6>(tmW, tmH, p, grid, smem, stream);
    case 7: return launch_gemm_n<MODE, 7>(tmW, tmH, p, grid, smem, stream);
    case 8: return launch_gemm_n<MODE, 8>(tmW, tmH, p, grid, smem, stream);
    case 16: return launch_gemm_n<MODE, 16>(tmW, tmH, p, grid, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

// arguments of the gated greedy call and of the sampling call
struct ModeArgs {
  float tau = 0.0f;
  int32_t* base_token = nullptr;
  float* margin = nullptr;
  const uint64_t* seeds = nullptr;
  const uint64_t* positions = nullptr;
  float temperature = 1.0f;
  float* score_gap = nullptr;
};

// Stages of the rows kernel: as many 32 KB stages as shared memory holds.
int rows_stages() {
  const RowsLayout L1 = rows_layout(1);
  const uint32_t fixed = L1.total - L1.stage_bytes + 2u * kRowsMaxStages * 8u + 1024u;
  int s = static_cast<int>((kSmemLimit - fixed) / L1.stage_bytes);
  return s > kRowsMaxStages ? kRowsMaxStages : s;
}

// The rows kernel's launch: clusters of two CTAs (384 threads each, the
// register split of the wide swap-AB kernel), as many pairs as fit on the
// GPU at once up to one per unit, a programmatic dependent of the previous
// kernel.
cudaError_t launch_rows_kernel(detlm_head* h, const CUtensorMap& tmH, const HeadParams& p,
                               int64_t units, size_t smem, cudaStream_t stream) {
  auto kern = head_rows_kernel;
  cudaError_t e = prepare_kernel<head_rows_kernel>(kRegsLaunchWide);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.blockDim = dim3(kRowsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  if (h->rows_pairs == 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(h->num_sms & ~1));
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    h->rows_pairs = clusters < h->num_sms / 2 ? clusters : h->num_sms / 2;
  }
  const int64_t pairs = units < h->rows_pairs ? units : h->rows_pairs;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, h->tmW, tmH, p);
}

// Stages of the wide greedy pair kernel: as many 32 KB stages as shared
// memory holds.
int pair_stages() {
  int s = kPairMaxStages;
  while (s > 2 && pair_layout(s).total + 1024u > kSmemLimit) --s;
  return s;
}

// The pair kernel's logits tensor map: [B][V] 4-byte elements, box 16 x 32
// (a warp's staging buffer), 64-byte swizzle. Used for logits in device
// memory with 16-byte aligned rows (V a multiple of 4, a 16-byte aligned
// base); otherwise (host memory the kernel writes through its mapping, such
// as the asynchronous host-buffer calls' pinned buffers) the kernel stores
// the logits with plain stores (returns false).
bool encode_logits(CUtensorMap* m, const void* logits, int64_t V, int64_t B, bool int32) {
  if (logits == nullptr || (V & 3) != 0 || !aligned(logits, 16)) return false;
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, logits) != cudaSuccess) {
    cudaGetLastError();   // clear the error the query recorded
    return false;
  }
  if (pa.type != cudaMemoryTypeDevice) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 4u};
  cuuint32_t box[2] = {16u, 32u};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, int32 ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(logits), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The wide greedy pair kernel's launch: clusters of two CTAs, as many pairs
// as fit on the GPU at once up to one per unit, a programmatic dependent of
// the previous kernel.
template <int MODE>
cudaError_t launch_pair_kernel(detlm_head* h, const CUtensorMap& tmW, const CUtensorMap& tmH,
                               const CUtensorMap& tmL, const HeadParams& p, int64_t units,
                               size_t smem, cudaStream_t stream) {
  auto kern = head_pair_kernel<MODE>;
  cudaError_t e = prepare_kernel<head_pair_kernel<MODE>>(kRegsLaunchWide);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  if (h->wide_pairs == 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(h->num_sms & ~1));
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    h->wide_pairs = clusters < h->num_sms / 2 ? clusters : h->num_sms / 2;
  }
  const int64_t pairs = units < h->wide_pairs ? units : h->wide_pairs;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmW, tmH, tmL, p);
}

// 256-entry tiles of a vocabulary of V (the log-sum-exp records' tiles, and
// the unit of the vocabulary shards)
int64_t tiles256(int64_t V) { return (V + kRowsN - 1) / kRowsN; }

// Rows [v_begin, v_end) of shard r of P: the 256-entry tiles of the leaves
// [128 r / P, 128 (r + 1) / P) of the log-sum-exp tree, i.e. tiles
// [floor(r n / P), floor((r + 1) n / P)) of the n = ceil(V / 256) tiles.
void shard_rows(int64_t V, int P, int r, int64_t* v_begin, int64_t* v_end) {
  const int64_t n = tiles256(V);
  const int64_t t0 = r * n / P, t1 = (r + 1) * n / P;
  *v_begin = t0 * kRowsN;
  *v_end = t1 * kRowsN < V ? t1 * kRowsN : V;
}

// Instead of the merge: one 16-byte record per row for this shard
// (shard_fold_kernel), launched as a dependent of the projection kernel.
cudaError_t launch_shard_fold(const detlm_head* h, int mode, int64_t B, int n_vt, const float* rec_m,
                              const int32_t* rec_i, const float* rec_s, const float* zt,
                              const int32_t* targets, ShardRec* out, cudaStream_t stream) {
  ShardFoldParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.B = static_cast<int32_t>(B);
  fp.n_vt = n_vt;
  fp.mode = mode;
  fp.n_tiles = static_cast<int32_t>(tiles256(h->V_total));
  fp.leaf0 = h->rank * (kLeaves / h->P);
  fp.n_leaves = kLeaves / h->P;
  fp.t0 = static_cast<int32_t>(h->v_off / kRowsN);
  fp.v_begin = static_cast<int32_t>(h->v_off);
  fp.v_end = static_cast<int32_t>(h->v_off + h->V);
  fp.rec_m = rec_m;
  fp.rec_i = rec_i;
  fp.rec_s = rec_s;
  fp.zt = zt;
  fp.targets = targets;
  fp.out = out;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, shard_fold_kernel, fp);
}

template <int MODE>
int launch_float(detlm_head* h, const void* h_dev, int64_t B, const int32_t* targets,
                 int32_t* token, float* gap, float* logits, float* logp, cudaStream_t stream,
                 const ModeArgs* gate = nullptr, ShardRec* shard_out = nullptr) {
  // the log-prob call runs on the rows kernel for every B (its records are
  // folded per row, in a fixed order, whatever B is)
  constexpr bool rows = MODE == MODE_LOGPROB;
  const int N = rows ? kRowsN : cols_for(B);
  // greedy calls of more than 128 rows: the pair kernel (CTA pairs, hidden
  // rows on the MMA's M axis; the same logits bit for bit)
  const bool wide = MODE == MODE_GREEDY && N == kPairN;
  CUtensorMap tmH;
  if (!encode_2d(&tmH, h->dtype, h_dev, h->d, B, (rows || wide) ? static_cast<uint32_t>(kRowsHalf)
                                                                 : static_cast<uint32_t>(N)))
    return DETLM_EINVAL;
  int st = ensure_ws(h, B, stream);
  if (st != DETLM_OK) return st;
  const WsView w = ws_view(h);

  HeadParams p;
  std::memset(&p, 0, sizeof(p));
  p.V = static_cast<int32_t>(h->V);
  p.d = static_cast<int32_t>(h->d);
  p.B = static_cast<int32_t>(B);
  p.N = N;
  p.nk = h->nk;
  p.n_chunks = static_cast<int32_t>((h->d + kChunkK - 1) / kChunkK);
  constexpr bool kExtraSmem = MODE == MODE_GATED || MODE == MODE_SAMPLE;
  if (rows) {
    // units: 256-entry vocabulary tiles x 256-row hidden tiles (one CTA pair)
    p.n_vt = static_cast<int32_t>((h->V + kRowsN - 1) / kRowsN);
    p.n_nt = static_cast<int32_t>((B + kRowsM - 1) / kRowsM);
    p.n_slots = 2;
    p.stages = rows_stages();
    p.n_issuers = 1;
    p.tmem_cols = 512;
    p.idesc = idesc_f16(h->dtype == DETLM_BF16 ? 1u : 0u, kRowsM, kRowsN);
  } else if (wide) {
    // units: two 128-row vocabulary tiles x 256 hidden rows (one CTA pair)
    p.n_vt = h->n_vt;
    p.n_nt = static_cast<int32_t>((B + kPairN - 1) / kPairN);
    p.n_slots = 2;
    p.stages = pair_stages();
    p.n_issuers = 1;
    p.tmem_cols = 512;
    p.idesc = idesc_f16(h->dtype == DETLM_BF16 ? 1u : 0u, 2 * kBM, kPairN);
  } else {
    p.n_vt = h->n_vt;
    p.n_nt = static_cast<int32_t>((B + N - 1) / N);
    p.n_slots = slots_for(N);
    p.stages = stages_for(N, kExtraSmem);
    p.n_issuers = issuers_for(N, p.stages, &p.n_slots);
    p.tmem_cols = tmem_cols_for(p.n_slots * N);
    p.idesc = idesc_f16(h->dtype == DETLM_BF16 ? 1u : 0u, kBM, static_cast<uint32_t>(N));
  }
  p.logits = logits;
  p.rec_m = w.m;
  p.rec_i = w.i;
  p.rec_s = w.s;
  p.err = h->d_err;
  p.stall = h->stall;
  p.timeout_ns = h->timeout_ns;
  p.v_off = static_cast<int32_t>(h->v_off);
  // the mode's own inputs (these members share storage)
  if constexpr (MODE == MODE_LOGPROB) {
    p.targets = targets;
    p.zt = w.zt;
  } else if constexpr (MODE == MODE_GATED) {
    p.rec_b = w.b;
    p.round_fp16 = h->dtype == DETLM_FP16 ? 1 : 0;
  } else if constexpr (MODE == MODE_SAMPLE) {
    p.seeds = gate->seeds;
    p.positions = gate->positions;
    p.temperature = gate->temperature;
  }

  const size_t smem = rows   ? rows_layout(p.stages).total + 1024
                     : wide ? pair_layout(p.stages).total + 1024
                            : smem_layout(N, p.stages, kExtraSmem).total + 1024;
  const int64_t units = wide ? static_cast<int64_t>((p.n_vt + 1) / 2) * p.n_nt
                             : static_cast<int64_t>(p.n_vt) * p.n_nt;
  const int grid = static_cast<int>(units < h->num_sms ? units : h->num_sms);
  CUtensorMap tmL = tmH;   // the pair kernel's logits map; not read unless valid
  if (wide) p.tma_logits = encode_logits(&tmL, logits, h->V, B, false) ? 1 : 0;
  if (h->t_start) cudaEventRecord(h->t_start, stream);
  cudaError_t e;
  if constexpr (rows) {
    e = launch_rows_kernel(h, tmH, p, units, smem, stream);
  } else if constexpr (MODE == MODE_GREEDY) {
    if (wide)
      e = launch_pair_kernel<MODE_GREEDY>(h, h->tmW, tmH, tmL, p, units, smem, stream);
    else
      e = launch_gemm<MODE>(h->tmW, tmH, p, grid, smem, stream);
  } else {
    e = launch_gemm<MODE>(h->tmW, tmH, p, grid, smem, stream);
  }
  if (h->t_stop) {
    cudaEventRecord(h->t_stop, stream);
    h->t_start = h->t_stop = nullptr;
  }
  if (e != cudaSuccess) return status_from_cuda(e);
  if (shard_out != nullptr)
    return status_from_cuda(launch_shard_fold(h, rows ? SHARD_LOGPROB : SHARD_GREEDY, B, p.n_vt,
                                              w.m, w.i, w.s, w.zt, targets, shard_out, stream));

  MergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  mp.V = p.V;
  mp.B = p.B;
  mp.n_vt = p.n_vt;
  mp.rec_m = w.m;
  mp.rec_i = w.i;
  mp.rec_s = w.s;
  mp.token = token;
  mp.gap = gap;
  mp.err = h->d_err;
  mp.acc = h->acc;
  if constexpr (MODE == MODE_LOGPROB) {
    mp.zt = w.zt;
    mp.targets = targets;
    mp.logp = logp;
  } else if constexpr (MODE == MODE_GATED) {
    mp.rec_b = w.b;
    mp.round_fp16 = h->dtype == DETLM_FP16 ? 1 : 0;
    mp.tau = gate->tau;
    mp.base_token = gate->base_token;
    mp.margin = gate->margin;
  } else if constexpr (MODE == MODE_SAMPLE) {
    mp.score_gap = gate->score_gap;
  }
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, merge_kernel<MODE>, mp);
  return status_from_cuda(e);
}

template <int N>
cudaError_t launch_int8_t(const CUtensorMap& tmW, const CUtensorMap& tmH, const Int8Params& p,
                          int grid, size_t smem, cudaStream_t stream) {
  cudaError_t e = prepare_kernel<int8_gemm_kernel<N>>(0);
  if (e != cudaSuccess) return e;
  // a programmatic dependent of the previous kernel on the stream (its
  // prologue and W prefetch overlap that kernel's tail)
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kI8Threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, int8_gemm_kernel<N>, tmW, tmH, p);
}

cudaError_t launch_int8_n(int N, const CUtensorMap& tmW, const CUtensorMap& tmH,
                          const Int8Params& p, int grid, size_t smem, cudaStream_t stream) {
  switch (N) {
    case 16: return launch_int8_t<16>(tmW, tmH, p, grid, smem, stream);
    case 32: return launch_int8_t<32>(tmW, tmH, p, grid, smem, stream);
    case 48: return launch_int8_t<48>(tmW, tmH, p, grid, smem, stream);
    case 64: return launch_int8_t<64>(tmW, tmH, p, grid, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Integer head, B >= kI8WideB: the projection kernel of the float heads on
// exact fp16 copies of the int8 values (MODE_INT), which is compute-bound
// there; the int8-streaming kernel serves smaller batches. Both are exact,
// so every B gives the same bits.
constexpr int64_t kI8WideB = 256;

cudaError_t i8_to_f16(const void* in, void* out, size_t n, cudaStream_t stream) {
  const size_t n16 = n / 16;
  size_t blocks = (n16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks == 0) blocks = 1;
  i8_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint4*>(in), static_cast<uint4*>(out), n16);
  return cudaGetLastError();
}

// The wide integer path's buffers: the fp16 copy of W (2 V d bytes, made
// once and kept until destroy) and the fp16 staging of B hidden rows. Made by
// detlm_head_reserve when max_B >= kI8WideB, else by the first such call.
int ensure_wide(detlm_head* h, int64_t B, cudaStream_t stream) {
  cudaError_t e;
  if (h->W16 == nullptr) {
    const size_t n = static_cast<size_t>(h->V) * h->d;
    void* w16 = nullptr;
    e = cudaMalloc(&w16, n * 2);
    if (e != cudaSuccess) return status_from_cuda(e);
    e = i8_to_f16(h->W, w16, n, stream);
    if (e != cudaSuccess || !encode_2d(&h->tmW16, DETLM_FP16, w16, h->d, h->V, kBM)) {
      cudaFree(w16);
      return e != cudaSuccess ? status_from_cuda(e) : DETLM_EINVAL;
    }
    h->W16 = w16;
  }
  const size_t hb = static_cast<size_t>(B) * h->d * 2;
  if (hb > h->h16_bytes) {
    if (h->h16 != nullptr) {
      e = cudaStreamSynchronize(stream);
      if (e != cudaSuccess) return status_from_cuda(e);
      cudaFree(h->h16);
      h->h16 = nullptr;
      h->h16_bytes = 0;
    }
    e = cudaMalloc(&h->h16, hb);
    if (e != cudaSuccess) return status_from_cuda(e);
    h->h16_bytes = hb;
  }
  return DETLM_OK;
}

int launch_int8_wide(detlm_head* h, const void* h_dev, int64_t B, int32_t* token, int32_t* gap,
                     int32_t* logits, cudaStream_t stream, ShardRec* shard_out = nullptr) {
  cudaError_t e;
  const int sw = ensure_wide(h, B, stream);
  if (sw != DETLM_OK) return sw;
  e = i8_to_f16(h_dev, h->h16, static_cast<size_t>(B) * h->d, stream);
  if (e != cudaSuccess) return status_from_cuda(e);
  // the pair kernel (CTA pairs, hidden rows on the MMA's M axis), as the
  // float heads' calls of more than 128 rows
  CUtensorMap tmH;
  if (!encode_2d(&tmH, DETLM_FP16, h->h16, h->d, B, static_cast<uint32_t>(kRowsHalf)))
    return DETLM_EINVAL;
  int st = ensure_ws(h, B, stream);
  if (st != DETLM_OK) return st;
  const WsView w = ws_view(h);

  HeadParams p;
  std::memset(&p, 0, sizeof(p));
  p.V = static_cast<int32_t>(h->V);
  p.d = static_cast<int32_t>(h->d);
  p.B = static_cast<int32_t>(B);
  p.N = kPairN;
  p.n_vt = h->n_vt;
  p.n_nt = static_cast<int32_t>((B + kPairN - 1) / kPairN);
  p.nk = static_cast<int32_t>((h->d * 2 + kRowBytes - 1) / kRowBytes);
  p.n_chunks = static_cast<int32_t>((h->d + kChunkK - 1) / kChunkK);
  p.n_slots = 2;
  p.stages = pair_stages();
  p.n_issuers = 1;
  p.tmem_cols = 512;
  p.idesc = idesc_f16(0u, 2 * kBM, kPairN);
  p.logits = reinterpret_cast<float*>(logits);
  p.rec_m = w.m;
  p.rec_i = w.i;
  p.rec_s = w.s;
  p.err = h->d_err;
  p.stall = h->stall;
  p.timeout_ns = h->timeout_ns;
  p.v_off = static_cast<int32_t>(h->v_off);
  const size_t smem = pair_layout(p.stages).total + 1024;
  const int64_t units = static_cast<int64_t>((p.n_vt + 1) / 2) * p.n_nt;
  CUtensorMap tmL = tmH;   // not read unless the logits map is valid
  p.tma_logits = encode_logits(&tmL, logits, h->V, B, true) ? 1 : 0;
  if (h->t_start) cudaEventRecord(h->t_start, stream);
  e = launch_pair_kernel<MODE_INT>(h, h->tmW16, tmH, tmL, p, units, smem, stream);
  if (h->t_stop) {
    cudaEventRecord(h->t_stop, stream);
    h->t_start = h->t_stop = nullptr;
  }
  if (e != cudaSuccess) return status_from_cuda(e);
  if (shard_out != nullptr)
    return status_from_cuda(launch_shard_fold(h, SHARD_GREEDY_INT, B, p.n_vt, w.m, w.i, w.s,
                                              nullptr, nullptr, shard_out, stream));

  Int8MergeParams mp;
  mp.B = p.B;
  mp.n_vt = p.n_vt;
  mp.rec_m = reinterpret_cast<const int32_t*>(w.m);
  mp.rec_i = w.i;
  mp.rec_s = reinterpret_cast<const int32_t*>(w.s);
  mp.token = token;
  mp.gap = gap;
  mp.acc = h->acc;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, int8_merge_kernel, mp);
  return status_from_cuda(e);
}

int launch_int8(detlm_head* h, const void* h_dev, int64_t B, int32_t* token, int32_t* gap,
                int32_t* logits, cudaStream_t stream, ShardRec* shard_out = nullptr) {
  if (B >= kI8WideB) return launch_int8_wide(h, h_dev, B, token, gap, logits, stream, shard_out);
  const int N = int8_cols_for(B, h->d);
  CUtensorMap tmH;
  if (!encode_2d(&tmH, DETLM_INT8, h_dev, h->d, B, static_cast<uint32_t>(N))) return DETLM_EINVAL;
  int st = ensure_ws(h, B, stream);
  if (st != DETLM_OK) return st;
  const WsView w = ws_view(h);

  Int8Params p;
  std::memset(&p, 0, sizeof(p));
  p.V = static_cast<int32_t>(h->V);
  p.d = static_cast<int32_t>(h->d);
  p.B = static_cast<int32_t>(B);
  p.N = N;
  p.n_vt = h->n_vt;
  p.n_nt = static_cast<int32_t>((B + N - 1) / N);
  p.nk = h->nk;
  p.n_chunks = int8_chunks(h->d);
  // as many int8 stages as shared memory holds (the W bytes in flight per SM
  // set the rate)
  const uint32_t fixed = int8_layout(N, 0).total + 3u * kI8MaxStages * 8u + 1024u;
  const uint32_t stage_bytes = int8_layout(N, 1).stage;
  p.stages = static_cast<int32_t>((kSmemLimit - fixed) / stage_bytes);
  if (p.stages > kI8MaxStages) p.stages = kI8MaxStages;
  if (p.stages < 2) return DETLM_EINVAL;   // cannot happen for N <= kI8MaxN
  p.idesc = idesc_f16(0u, kBM, static_cast<uint32_t>(N));
  p.logits = logits;
  p.rec_m = reinterpret_cast<int32_t*>(w.m);
  p.rec_i = w.i;
  p.rec_s = reinterpret_cast<int32_t*>(w.s);
  p.err = h->d_err;
  p.stall = h->stall;
  p.timeout_ns = h->timeout_ns;
  p.v_off = static_cast<int32_t>(h->v_off);

  const size_t smem = int8_layout(N, p.stages).total + 1024;
  const int64_t units = static_cast<int64_t>(p.n_vt) * p.n_nt;
  const int grid = static_cast<int>(units < h->num_sms ? units : h->num_sms);
  if (h->t_start) cudaEventRecord(h->t_start, stream);
  cudaError_t e = launch_int8_n(N, h->tmW, tmH, p, grid, smem, stream);
  if (h->t_stop) {
    cudaEventRecord(h->t_stop, stream);
    h->t_start = h->t_stop = nullptr;
  }
  if (e != cudaSuccess) return status_from_cuda(e);
  if (shard_out != nullptr)
    return status_from_cuda(launch_shard_fold(h, SHARD_GREEDY_INT, B, p.n_vt,
                                              reinterpret_cast<const float*>(p.rec_m), p.rec_i,
                                              reinterpret_cast<const float*>(p.rec_s), nullptr,
                                              nullptr, shard_out, stream));

  Int8MergeParams mp;
  mp.B = p.B;
  mp.n_vt = p.n_vt;
  mp.rec_m = p.rec_m;
  mp.rec_i = p.rec_i;
  mp.rec_s = p.rec_s;
  mp.token = token;
  mp.gap = gap;
  mp.acc = h->acc;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, int8_merge_kernel, mp);
  return status_from_cuda(e);
}

int read_err(detlm_head* h, cudaStream_t stream) {
  if (h->err_mapped != nullptr) {
    // the word lives in host memory: once the stream is idle no kernel of
    // this handle can write it, and the next ones see the host's clear
    const cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return status_from_cuda(e);
    volatile int* w = h->err_mapped;
    const int hv = *w;
    if (hv != 0) *w = 0;
    if (hv & ERR_TIMEOUT) return DETLM_ETIMEOUT;
    if (hv & ERR_TARGET) return DETLM_ETARGET;
    return DETLM_OK;
  }
  // into a pinned word: a copy to pageable memory costs an extra staging step
  cudaError_t e = cudaMemcpyAsync(h->err_host, h->d_err, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return status_from_cuda(e);
  const int hv = *h->err_host;
  if (hv != 0) {
    e = cudaMemsetAsync(h->d_err, 0, sizeof(int), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return status_from_cuda(e);
  }
  if (hv & ERR_TIMEOUT) return DETLM_ETIMEOUT;
  if (hv & ERR_TARGET) return DETLM_ETARGET;
  return DETLM_OK;
}

int ensure_stage(detlm_head* h, size_t bytes, cudaStream_t stream) {
  if (bytes <= h->stage_bytes) return DETLM_OK;
  if (h->stage != nullptr) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return status_from_cuda(e);
    cudaFree(h->stage);
    h->stage = nullptr;
    h->stage_bytes = 0;
  }
  cudaError_t e = cudaMalloc(&h->stage, bytes);
  if (e != cudaSuccess) return status_from_cuda(e);
  h->stage_bytes = bytes;
  return DETLM_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Copy n16 16-byte words of hidden rows from a buffer the device can read
// (pinned host memory) into the handle's staging, as a programmatic
// dependent of the previous call's merge: it waits for that kernel (and so
// for the previous projection, the last reader of the staging) before
// writing, and the next projection, launched as its dependent, requests its
// first W boxes while this copy runs.
__global__ void __launch_bounds__(256) stage_rows_kernel(const uint4* __restrict__ src,
                                                         uint4* __restrict__ dst, size_t n16) {
  grid_dep_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    dst[i] = src[i];
  __syncthreads();
  grid_dep_launch();
}

cudaError_t launch_stage_rows(const void* src_dev, void* dst, size_t bytes, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  size_t blocks = (n16 + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  if (blocks == 0) blocks = 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stage_rows_kernel, static_cast<const uint4*>(src_dev),
                            static_cast<uint4*>(dst), n16);
}

// The device address of a caller's buffer if kernels can write it directly
// (device or managed memory, or pinned host memory mapped into the device's
// address space, as cudaHostAlloc and cudaHostRegister give it), else null.
void* device_address(void* p) {
  if (p == nullptr) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();   // not a CUDA-known pointer: clear the sticky-free error
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) return a.devicePointer;
  return nullptr;
}

// Staging of the asynchronous host-buffer calls: the copy stream and its
// events on first use; the buffers grown to hold in_bytes of rows and
// out_bytes of outputs per slot (growth waits for every pending call).
int ensure_async(detlm_head* h, size_t in_bytes, size_t out_bytes, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (h->a_copy == nullptr) {
    e = cudaStreamCreateWithFlags(&h->a_copy, cudaStreamNonBlocking);
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
      e = cudaEventCreateWithFlags(&h->a_done[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->a_freed[k], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return status_from_cuda(e);
  }
  if (in_bytes > h->a_in_bytes || out_bytes > h->a_out_bytes) {
    e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->a_copy);
    if (e != cudaSuccess) return status_from_cuda(e);
  }
  if (in_bytes > h->a_in_bytes) {
    if (h->a_in) cudaFree(h->a_in);
    h->a_in = nullptr;
    h->a_in_bytes = 0;
    e = cudaMalloc(&h->a_in, in_bytes);
    if (e != cudaSuccess) return status_from_cuda(e);
    h->a_in_bytes = in_bytes;
  }
  if (out_bytes > h->a_out_bytes) {
    for (int k = 0; k < 2; ++k) {
      if (h->a_out[k]) cudaFree(h->a_out[k]);
      h->a_out[k] = nullptr;
    }
    h->a_out_bytes = 0;
    for (int k = 0; k < 2; ++k) {
      e = cudaMalloc(&h->a_out[k], out_bytes);
      if (e != cudaSuccess) return status_from_cuda(e);
    }
    h->a_out_bytes = out_bytes;
  }
  return DETLM_OK;
}

bool bad_B(int64_t B) { return B < 0 || B >= (int64_t{1} << 31); }

int launch_quantize(const void* x_dev, int dtype, int64_t B, int64_t d, int8_t* q, int32_t* mult,
                    int32_t* shift, cudaStream_t stream) {
  QuantParams qp;
  qp.x = x_dev;
  qp.fmt = dtype;
  qp.d = d;
  qp.q = q;
  qp.mult = mult;
  qp.shift = shift;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(kQThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return status_from_cuda(cudaLaunchKernelEx(&cfg, quantize_rows_kernel, qp));
}

}  // namespace

extern "C" {

const char* detlm_status_string(int status) {
  switch (status) {
    case DETLM_OK: return "ok";
    case DETLM_EINVAL: return "invalid argument";
    case DETLM_EUNSUPPORTED: return "operation not supported for this head's dtype";
    case DETLM_ECUDA: return "CUDA runtime error (no usable GPU, or a launch failed)";
    case DETLM_ETIMEOUT: return "a device-side bounded wait ran out";
    case DETLM_ENOMEM: return "out of memory";
    case DETLM_ETARGET: return "a target id was outside [0, V)";
    default: return "unknown status";
  }
}

int detlm_head_create(detlm_head_t** out, const void* W_dev, int64_t V, int64_t d, int dtype) {
  if (out == nullptr) return DETLM_EINVAL;
  *out = nullptr;
  if (W_dev == nullptr || !aligned(W_dev, 16)) return DETLM_EINVAL;
  if (dtype != DETLM_BF16 && dtype != DETLM_FP16 && dtype != DETLM_INT8) return DETLM_EINVAL;
  if (V < 1 || V >= (int64_t{1} << 31) || d < 1 || d >= (int64_t{1} << 31)) return DETLM_EINVAL;
  if ((d * static_cast<int64_t>(elem_bytes(dtype))) % 16 != 0) return DETLM_EINVAL;
  if (dtype == DETLM_INT8 && d > kI8MaxD) return DETLM_EINVAL;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return DETLM_ECUDA;
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || sms <= 0) return DETLM_ECUDA;   // built for sm_103a only
  if (!load_encode()) return DETLM_ECUDA;

  detlm_head* h = new (std::nothrow) detlm_head();
  if (h == nullptr) return DETLM_ENOMEM;
  h->device = dev;
  h->dtype = dtype;
  h->V = V;
  h->d = d;
  h->W = W_dev;
  h->num_sms = sms;
  h->n_vt = static_cast<int>((V + kBM - 1) / kBM);
  h->nk = static_cast<int>((d * static_cast<int64_t>(elem_bytes(dtype)) + kRowBytes - 1) / kRowBytes);
  h->timeout_ns = kDefaultTimeoutNs;
  h->V_total = V;
  if (!encode_2d(&h->tmW, dtype, W_dev, d, V, kBM)) {
    delete h;
    return DETLM_EINVAL;
  }
  int host_atomics = 0;
  cudaDeviceGetAttribute(&host_atomics, cudaDevAttrHostNativeAtomicSupported, dev);
  if (host_atomics) {
    e = cudaHostAlloc(reinterpret_cast<void**>(&h->err_mapped), sizeof(int), cudaHostAllocMapped);
    if (e == cudaSuccess) {
      *h->err_mapped = 0;
      e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->d_err), h->err_mapped, 0);
    }
  } else {
    e = cudaMalloc(&h->d_err, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(int));
  }
  if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&h->err_host), sizeof(int),
                                          cudaHostAllocDefault);
  if (e != cudaSuccess) {
    if (h->err_mapped) cudaFreeHost(h->err_mapped);
    else if (h->d_err) cudaFree(h->d_err);
    if (h->err_host) cudaFreeHost(h->err_host);
    delete h;
    return status_from_cuda(e);
  }
  *out = h;
  return DETLM_OK;
}

int detlm_shard_range(int64_t V, int P, int rank, int64_t* v_begin, int64_t* v_end) {
  if (v_begin == nullptr || v_end == nullptr) return DETLM_EINVAL;
  if (V < 1 || V >= (int64_t{1} << 31)) return DETLM_EINVAL;
  if (P < 1 || P > kLeaves || (P & (P - 1)) != 0 || rank < 0 || rank >= P) return DETLM_EINVAL;
  shard_rows(V, P, rank, v_begin, v_end);
  return DETLM_OK;
}

int detlm_head_create_shard(detlm_head_t** out, const void* W_shard_dev, int64_t V, int64_t d,
                            int dtype, int P, int rank) {
  if (out == nullptr) return DETLM_EINVAL;
  *out = nullptr;
  int64_t v0 = 0, v1 = 0;
  const int st = detlm_shard_range(V, P, rank, &v0, &v1);
  if (st != DETLM_OK) return st;
  if (v1 <= v0) return DETLM_EINVAL;             // fewer 256-entry tiles than shards
  detlm_head_t* h = nullptr;
  const int c = detlm_head_create(&h, W_shard_dev, v1 - v0, d, dtype);
  if (c != DETLM_OK) return c;
  h->v_off = v0;
  h->V_total = V;
  h->P = P;
  h->rank = rank;
  *out = h;
  return DETLM_OK;
}

int detlm_head_greedy_shard(detlm_head_t* h, const void* h_dev, int64_t B,
                            detlm_shard_rec_t* rec_dev, void* logits_dev, cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (B == 0) return DETLM_OK;
  if (h_dev == nullptr || !aligned(h_dev, 16)) return DETLM_EINVAL;
  if (rec_dev == nullptr || !aligned(rec_dev, 16)) return DETLM_EINVAL;
  if (logits_dev != nullptr && !aligned(logits_dev, 4)) return DETLM_EINVAL;
  ShardRec* out = reinterpret_cast<ShardRec*>(rec_dev);
  if (h->dtype == DETLM_INT8)
    return launch_int8(h, h_dev, B, nullptr, nullptr, static_cast<int32_t*>(logits_dev), stream,
                       out);
  return launch_float<MODE_GREEDY>(h, h_dev, B, nullptr, nullptr, nullptr,
                                   static_cast<float*>(logits_dev), nullptr, stream, nullptr, out);
}

int detlm_head_logprob_shard(detlm_head_t* h, const void* h_dev, const int32_t* targets_dev,
                             int64_t B, detlm_shard_rec_t* rec_dev, cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (h->dtype == DETLM_INT8) return DETLM_EUNSUPPORTED;
  if (B == 0) return DETLM_OK;
  if (h_dev == nullptr || !aligned(h_dev, 16)) return DETLM_EINVAL;
  if (targets_dev == nullptr || !aligned(targets_dev, 4)) return DETLM_EINVAL;
  if (rec_dev == nullptr || !aligned(rec_dev, 16)) return DETLM_EINVAL;
  return launch_float<MODE_LOGPROB>(h, h_dev, B, targets_dev, nullptr, nullptr, nullptr, nullptr,
                                    stream, nullptr, reinterpret_cast<ShardRec*>(rec_dev));
}

namespace {
cudaError_t launch_shard_merge(const ShardMergeParams& mp, int64_t B, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, shard_merge_kernel, mp);
}
bool bad_P(int P) { return P < 1 || P > kLeaves || (P & (P - 1)) != 0; }
}  // namespace

int detlm_merge_greedy_shards(const detlm_shard_rec_t* recs_dev, int P, int64_t B, int dtype,
                              int32_t* token_dev, void* gap_dev, cudaStream_t stream) {
  if (bad_P(P) || bad_B(B)) return DETLM_EINVAL;
  if (dtype != DETLM_BF16 && dtype != DETLM_FP16 && dtype != DETLM_INT8) return DETLM_EINVAL;
  if (static_cast<int64_t>(P) * B >= (int64_t{1} << 31)) return DETLM_EINVAL;
  if (B == 0) return DETLM_OK;
  if (recs_dev == nullptr || !aligned(recs_dev, 16)) return DETLM_EINVAL;
  if (token_dev == nullptr || !aligned(token_dev, 4)) return DETLM_EINVAL;
  if (gap_dev == nullptr || !aligned(gap_dev, 4)) return DETLM_EINVAL;
  ShardMergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  mp.P = P;
  mp.B = static_cast<int32_t>(B);
  mp.mode = dtype == DETLM_INT8 ? SHARD_GREEDY_INT : SHARD_GREEDY;
  mp.recs = reinterpret_cast<const ShardRec*>(recs_dev);
  mp.token = token_dev;
  mp.gap = gap_dev;
  return status_from_cuda(launch_shard_merge(mp, B, stream));
}

int detlm_merge_logprob_shards(const detlm_shard_rec_t* recs_dev, int P, int64_t B, int64_t V,
                               const int32_t* targets_dev, float* logp_dev, int* err_dev,
                               cudaStream_t stream) {
  if (bad_P(P) || bad_B(B)) return DETLM_EINVAL;
  if (V < 1 || V >= (int64_t{1} << 31)) return DETLM_EINVAL;
  if (static_cast<int64_t>(P) * B >= (int64_t{1} << 31)) return DETLM_EINVAL;
  if (B == 0) return DETLM_OK;
  if (recs_dev == nullptr || !aligned(recs_dev, 16)) return DETLM_EINVAL;
  if (targets_dev == nullptr || !aligned(targets_dev, 4)) return DETLM_EINVAL;
  if (logp_dev == nullptr || !aligned(logp_dev, 4)) return DETLM_EINVAL;
  if (err_dev != nullptr && !aligned(err_dev, 4)) return DETLM_EINVAL;
  ShardMergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  mp.P = P;
  mp.B = static_cast<int32_t>(B);
  mp.V = static_cast<int32_t>(V);
  mp.mode = SHARD_LOGPROB;
  mp.recs = reinterpret_cast<const ShardRec*>(recs_dev);
  mp.targets = targets_dev;
  mp.logp = logp_dev;
  mp.err = err_dev;
  return status_from_cuda(launch_shard_merge(mp, B, stream));
}

int detlm_head_reserve(detlm_head_t* h, int64_t max_B) {
  if (h == nullptr || bad_B(max_B)) return DETLM_EINVAL;
  int st = ensure_ws(h, max_B, nullptr);
  if (st == DETLM_OK && h->dtype == DETLM_INT8 && max_B >= kI8WideB) {
    st = ensure_wide(h, max_B, nullptr);
    if (st == DETLM_OK) st = status_from_cuda(cudaStreamSynchronize(nullptr));
  }
  return st;
}

int detlm_head_greedy(detlm_head_t* h, const void* h_dev, int64_t B, int32_t* token_dev,
                      void* gap_dev, void* logits_dev, cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (B == 0) return DETLM_OK;
  if (h_dev == nullptr || !aligned(h_dev, 16)) return DETLM_EINVAL;
  if (token_dev == nullptr || !aligned(token_dev, 4)) return DETLM_EINVAL;
  if (gap_dev == nullptr || !aligned(gap_dev, 4)) return DETLM_EINVAL;
  if (logits_dev != nullptr && !aligned(logits_dev, 4)) return DETLM_EINVAL;
  if (h->dtype == DETLM_INT8)
    return launch_int8(h, h_dev, B, token_dev, static_cast<int32_t*>(gap_dev),
                       static_cast<int32_t*>(logits_dev), stream);
  return launch_float<MODE_GREEDY>(h, h_dev, B, nullptr, token_dev, static_cast<float*>(gap_dev),
                                   static_cast<float*>(logits_dev), nullptr, stream);
}

int detlm_head_logprob(detlm_head_t* h, const void* h_dev, const int32_t* targets_dev, int64_t B,
                       float* logp_dev, cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (h->dtype == DETLM_INT8) return DETLM_EUNSUPPORTED;
  if (B == 0) return DETLM_OK;
  if (h_dev == nullptr || !aligned(h_dev, 16)) return DETLM_EINVAL;
  if (targets_dev == nullptr || !aligned(targets_dev, 4)) return DETLM_EINVAL;
  if (logp_dev == nullptr || !aligned(logp_dev, 4)) return DETLM_EINVAL;
  return launch_float<MODE_LOGPROB>(h, h_dev, B, targets_dev, nullptr, nullptr, nullptr, logp_dev,
                                    stream);
}

int detlm_head_greedy_gated(detlm_head_t* h, const void* h_dev, int64_t B, float tau,
                            int32_t* token_dev, float* gap_dev, float* logits_dev,
                            int32_t* base_token_dev, float* margin_dev, cudaStream_t stream) {
  if (h == nullptr || bad_B(B) || std::isnan(tau)) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (h->dtype == DETLM_INT8) return DETLM_EUNSUPPORTED;
  if (B == 0) return DETLM_OK;
  if (h_dev == nullptr || !aligned(h_dev, 16)) return DETLM_EINVAL;
  if (token_dev == nullptr || !aligned(token_dev, 4)) return DETLM_EINVAL;
  if (gap_dev == nullptr || !aligned(gap_dev, 4)) return DETLM_EINVAL;
  if (logits_dev != nullptr && !aligned(logits_dev, 4)) return DETLM_EINVAL;
  if (base_token_dev != nullptr && !aligned(base_token_dev, 4)) return DETLM_EINVAL;
  if (margin_dev != nullptr && !aligned(margin_dev, 4)) return DETLM_EINVAL;
  ModeArgs gate;
  gate.tau = tau;
  gate.base_token = base_token_dev;
  gate.margin = margin_dev;
  return launch_float<MODE_GATED>(h, h_dev, B, nullptr, token_dev, gap_dev, logits_dev, nullptr,
                                  stream, &gate);
}

int detlm_head_sample(detlm_head_t* h, const void* h_dev, int64_t B, float temperature,
                      const uint64_t* seeds_dev, const uint64_t* positions_dev, int32_t* token_dev,
                      float* score_gap_dev, float* logits_dev, cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return DETLM_EINVAL;
  if (h->dtype == DETLM_INT8) return DETLM_EUNSUPPORTED;
  if (B == 0) return DETLM_OK;
  if (h_dev == nullptr || !aligned(h_dev, 16)) return DETLM_EINVAL;
  if (seeds_dev == nullptr || !aligned(seeds_dev, 8)) return DETLM_EINVAL;
  if (positions_dev == nullptr || !aligned(positions_dev, 8)) return DETLM_EINVAL;
  if (token_dev == nullptr || !aligned(token_dev, 4)) return DETLM_EINVAL;
  if (score_gap_dev != nullptr && !aligned(score_gap_dev, 4)) return DETLM_EINVAL;
  if (logits_dev != nullptr && !aligned(logits_dev, 4)) return DETLM_EINVAL;
  ModeArgs a;
  a.seeds = seeds_dev;
  a.positions = positions_dev;
  a.temperature = temperature;
  a.score_gap = score_gap_dev;
  return launch_float<MODE_SAMPLE>(h, h_dev, B, nullptr, token_dev, nullptr, logits_dev, nullptr,
                                   stream, &a);
}

int detlm_quantize_rows(const void* x_dev, int dtype, int64_t B, int64_t d, int8_t* q_dev,
                        int32_t* mult_dev, int32_t* shift_dev, cudaStream_t stream) {
  if (dtype != DETLM_BF16 && dtype != DETLM_FP16 && dtype != DETLM_FP32) return DETLM_EINVAL;
  if (bad_B(B) || d < 1 || d >= (int64_t{1} << 31)) return DETLM_EINVAL;
  if (B == 0) return DETLM_OK;
  const size_t eb = dtype == DETLM_FP32 ? 4 : 2;
  if (x_dev == nullptr || !aligned(x_dev, eb)) return DETLM_EINVAL;
  if (q_dev == nullptr) return DETLM_EINVAL;
  if (mult_dev == nullptr || !aligned(mult_dev, 4)) return DETLM_EINVAL;
  if (shift_dev == nullptr || !aligned(shift_dev, 4)) return DETLM_EINVAL;
  return launch_quantize(x_dev, dtype, B, d, q_dev, mult_dev, shift_dev, stream);
}

int detlm_head_greedy_from_float(detlm_head_t* h, const void* x_dev, int x_dtype, int64_t B,
                                 int32_t* token_dev, int32_t* gap_dev, int32_t* logits_dev,
                                 int32_t* mult_dev, int32_t* shift_dev, cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (h->dtype != DETLM_INT8) return DETLM_EUNSUPPORTED;
  if (x_dtype != DETLM_BF16 && x_dtype != DETLM_FP16 && x_dtype != DETLM_FP32) return DETLM_EINVAL;
  if (B == 0) return DETLM_OK;
  const size_t eb = x_dtype == DETLM_FP32 ? 4 : 2;
  if (x_dev == nullptr || !aligned(x_dev, eb)) return DETLM_EINVAL;
  if (token_dev == nullptr || !aligned(token_dev, 4)) return DETLM_EINVAL;
  if (gap_dev == nullptr || !aligned(gap_dev, 4)) return DETLM_EINVAL;
  if (logits_dev != nullptr && !aligned(logits_dev, 4)) return DETLM_EINVAL;
  if (mult_dev != nullptr && !aligned(mult_dev, 4)) return DETLM_EINVAL;
  if (shift_dev != nullptr && !aligned(shift_dev, 4)) return DETLM_EINVAL;
  // handle buffer: q [B, d] (256-byte aligned, rows of d bytes, d % 16 == 0
  // for an int8 head) and, when the caller passes none, M and S [B]
  const size_t qb = round256(static_cast<size_t>(B) * h->d);
  const size_t need = qb + 2 * round256(static_cast<size_t>(B) * 4);
  if (need > h->q8_bytes) {
    if (h->q8 != nullptr) {
      cudaError_t e = cudaStreamSynchronize(stream);
      if (e != cudaSuccess) return status_from_cuda(e);
      cudaFree(h->q8);
      h->q8 = nullptr;
      h->q8_bytes = 0;
    }
    cudaError_t e = cudaMalloc(&h->q8, need);
    if (e != cudaSuccess) return status_from_cuda(e);
    h->q8_bytes = need;
  }
  uint8_t* base = static_cast<uint8_t*>(h->q8);
  int8_t* q = reinterpret_cast<int8_t*>(base);
  int32_t* m = mult_dev ? mult_dev : reinterpret_cast<int32_t*>(base + qb);
  int32_t* s = shift_dev ? shift_dev
                         : reinterpret_cast<int32_t*>(base + qb + round256(static_cast<size_t>(B) * 4));
  int st = launch_quantize(x_dev, x_dtype, B, h->d, q, m, s, stream);
  if (st != DETLM_OK) return st;
  return launch_int8(h, q, B, token_dev, gap_dev, logits_dev, stream);
}

int detlm_head_verify(detlm_head_t* h, const void* h_dev, int64_t n_req, int64_t P,
                      const int32_t* drafts_dev, int32_t* token_dev, void* gap_dev,
                      void* logits_dev, int32_t* accepted_dev, cudaStream_t stream) {
  if (h == nullptr || n_req < 0 || P < 1) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (n_req > 0 && P > (INT32_MAX - 1) / n_req) return DETLM_EINVAL;
  if (n_req == 0) return DETLM_OK;
  if (drafts_dev == nullptr || !aligned(drafts_dev, 4)) return DETLM_EINVAL;
  if (accepted_dev == nullptr || !aligned(accepted_dev, 4)) return DETLM_EINVAL;
  int st = ensure_vws(h, n_req, stream);
  if (st != DETLM_OK) return st;
  h->acc.P = static_cast<int32_t>(P);
  h->acc.drafts = drafts_dev;
  h->acc.R = static_cast<int32_t>(h->vws_R);
  h->acc.words = h->vws;
  h->acc.accepted = accepted_dev;
  st = detlm_head_greedy(h, h_dev, n_req * P, token_dev, gap_dev, logits_dev, stream);
  h->acc = AcceptArgs{};
  return st;
}

int detlm_head_greedy_host(detlm_head_t* h, const void* h_host, int64_t B, int32_t* token_host,
                           void* gap_host, void* logits_host, cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (B == 0) return DETLM_OK;
  if (h_host == nullptr || token_host == nullptr || gap_host == nullptr) return DETLM_EINVAL;
  const size_t hb = static_cast<size_t>(B) * h->d * elem_bytes(h->dtype);
  const size_t ob = static_cast<size_t>(B) * 4;
  const size_t lb = logits_host ? static_cast<size_t>(B) * h->V * 4 : 0;
  int st = ensure_stage(h, round256(hb) + 2 * round256(ob) + round256(lb), stream);
  if (st != DETLM_OK) return st;
  uint8_t* s = static_cast<uint8_t*>(h->stage);
  void* dh = s;
  int32_t* dtok = reinterpret_cast<int32_t*>(s + round256(hb));
  void* dgap = s + round256(hb) + round256(ob);
  void* dlog = logits_host ? s + round256(hb) + 2 * round256(ob) : nullptr;
  cudaError_t e = cudaMemcpyAsync(dh, h_host, hb, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return status_from_cuda(e);
  st = detlm_head_greedy(h, dh, B, dtok, dgap, dlog, stream);
  if (st != DETLM_OK) return st;
  e = cudaMemcpyAsync(token_host, dtok, ob, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(gap_host, dgap, ob, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess && logits_host)
    e = cudaMemcpyAsync(logits_host, dlog, lb, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return status_from_cuda(e);
  return read_err(h, stream);
}

int detlm_head_logprob_host(detlm_head_t* h, const void* h_host, const int32_t* targets_host,
                            int64_t B, float* logp_host, cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (h->dtype == DETLM_INT8) return DETLM_EUNSUPPORTED;
  if (B == 0) return DETLM_OK;
  if (h_host == nullptr || targets_host == nullptr || logp_host == nullptr) return DETLM_EINVAL;
  const size_t hb = static_cast<size_t>(B) * h->d * elem_bytes(h->dtype);
  const size_t ob = static_cast<size_t>(B) * 4;
  int st = ensure_stage(h, round256(hb) + 2 * round256(ob), stream);
  if (st != DETLM_OK) return st;
  uint8_t* s = static_cast<uint8_t*>(h->stage);
  void* dh = s;
  int32_t* dt = reinterpret_cast<int32_t*>(s + round256(hb));
  float* dlp = reinterpret_cast<float*>(s + round256(hb) + round256(ob));
  cudaError_t e = cudaMemcpyAsync(dh, h_host, hb, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(dt, targets_host, ob, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return status_from_cuda(e);
  st = detlm_head_logprob(h, dh, dt, B, dlp, stream);
  if (st != DETLM_OK) return st;
  e = cudaMemcpyAsync(logp_host, dlp, ob, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return status_from_cuda(e);
  return read_err(h, stream);
}

int detlm_head_greedy_host_async(detlm_head_t* h, const void* h_host, int64_t B,
                                 int32_t* token_host, void* gap_host, void* logits_host,
                                 cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (B == 0) return DETLM_OK;
  if (h_host == nullptr || token_host == nullptr || gap_host == nullptr) return DETLM_EINVAL;
  const size_t hb = static_cast<size_t>(B) * h->d * elem_bytes(h->dtype);
  const size_t ob = static_cast<size_t>(B) * 4;
  const size_t lb = logits_host ? static_cast<size_t>(B) * h->V * 4 : 0;
  // results straight into the caller's buffers where the device can write
  // them (pinned host memory): no staging, no copy back
  void* tok_d = device_address(token_host);
  void* gap_d = device_address(gap_host);
  void* log_d = device_address(logits_host);
  const bool direct = tok_d != nullptr && gap_d != nullptr &&
                      (logits_host == nullptr || log_d != nullptr) &&
                      aligned(tok_d, 4) && aligned(gap_d, 4) && (log_d == nullptr || aligned(log_d, 4));
  int st = ensure_async(h, round256(hb), direct ? 0 : 2 * round256(ob) + round256(lb), stream);
  if (st != DETLM_OK) return st;
  if (direct) {
    // rows the device can read (pinned, 16-byte aligned: row bytes are a
    // multiple of 16) are staged by a kernel that chains with the previous
    // call's kernels; other rows by a copy
    const void* in_d = aligned(h_host, 16) ? device_address(const_cast<void*>(h_host)) : nullptr;
    const cudaError_t e = in_d != nullptr
                              ? launch_stage_rows(in_d, h->a_in, hb, stream)
                              : cudaMemcpyAsync(h->a_in, h_host, hb, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return status_from_cuda(e);
    return detlm_head_greedy(h, h->a_in, B, static_cast<int32_t*>(tok_d), gap_d, log_d, stream);
  }
  const int k = h->a_next;
  uint8_t* o = static_cast<uint8_t*>(h->a_out[k]);
  int32_t* dtok = reinterpret_cast<int32_t*>(o);
  void* dgap = o + round256(ob);
  void* dlog = logits_host ? o + 2 * round256(ob) : nullptr;
  // the slot's previous copy to the host must be done before it is reused
  cudaError_t e = cudaStreamWaitEvent(stream, h->a_freed[k], 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h->a_in, h_host, hb, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return status_from_cuda(e);
  st = detlm_head_greedy(h, h->a_in, B, dtok, dgap, dlog, stream);
  if (st != DETLM_OK) return st;
  e = cudaEventRecord(h->a_done[k], stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->a_copy, h->a_done[k], 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(token_host, dtok, ob, cudaMemcpyDeviceToHost, h->a_copy);
  if (e == cudaSuccess) e = cudaMemcpyAsync(gap_host, dgap, ob, cudaMemcpyDeviceToHost, h->a_copy);
  if (e == cudaSuccess && logits_host)
    e = cudaMemcpyAsync(logits_host, dlog, lb, cudaMemcpyDeviceToHost, h->a_copy);
  if (e == cudaSuccess) e = cudaEventRecord(h->a_freed[k], h->a_copy);
  if (e != cudaSuccess) return status_from_cuda(e);
  h->a_next = k ^ 1;
  return DETLM_OK;
}

int detlm_head_logprob_host_async(detlm_head_t* h, const void* h_host, const int32_t* targets_host,
                                  int64_t B, float* logp_host, cudaStream_t stream) {
  if (h == nullptr || bad_B(B)) return DETLM_EINVAL;
  if (h->P > 1) return DETLM_EUNSUPPORTED;   // a vocabulary shard: the *_shard calls
  if (h->dtype == DETLM_INT8) return DETLM_EUNSUPPORTED;
  if (B == 0) return DETLM_OK;
  if (h_host == nullptr || targets_host == nullptr || logp_host == nullptr) return DETLM_EINVAL;
  const size_t hb = static_cast<size_t>(B) * h->d * elem_bytes(h->dtype);
  const size_t ob = static_cast<size_t>(B) * 4;
  void* lp_d = device_address(logp_host);
  const bool direct = lp_d != nullptr && aligned(lp_d, 4);
  int st = ensure_async(h, round256(hb) + round256(ob), direct ? 0 : round256(ob), stream);
  if (st != DETLM_OK) return st;
  if (direct) {
    uint8_t* in = static_cast<uint8_t*>(h->a_in);
    int32_t* dt = reinterpret_cast<int32_t*>(in + round256(hb));
    cudaError_t e = cudaMemcpyAsync(in, h_host, hb, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dt, targets_host, ob, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return status_from_cuda(e);
    return detlm_head_logprob(h, in, dt, B, static_cast<float*>(lp_d), stream);
  }
  const int k = h->a_next;
  float* dlp = static_cast<float*>(h->a_out[k]);
  uint8_t* in = static_cast<uint8_t*>(h->a_in);
  int32_t* dt = reinterpret_cast<int32_t*>(in + round256(hb));
  cudaError_t e = cudaStreamWaitEvent(stream, h->a_freed[k], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(in, h_host, hb, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(dt, targets_host, ob, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return status_from_cuda(e);
  st = detlm_head_logprob(h, in, dt, B, dlp, stream);
  if (st != DETLM_OK) return st;
  e = cudaEventRecord(h->a_done[k], stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->a_copy, h->a_done[k], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(logp_host, dlp, ob, cudaMemcpyDeviceToHost, h->a_copy);
  if (e == cudaSuccess) e = cudaEventRecord(h->a_freed[k], h->a_copy);
  if (e != cudaSuccess) return status_from_cuda(e);
  h->a_next = k ^ 1;
  return DETLM_OK;
}

int detlm_head_check(detlm_head_t* h, cudaStream_t stream) {
  if (h == nullptr) return DETLM_EINVAL;
  if (h->a_copy != nullptr) {
    // the asynchronous host-buffer calls' copies to the host
    const cudaError_t e = cudaStreamSynchronize(h->a_copy);
    if (e != cudaSuccess) return status_from_cuda(e);
  }
  return read_err(h, stream);
}

int detlm_head_time_next(detlm_head_t* h, cudaEvent_t start, cudaEvent_t stop) {
  if (h == nullptr || (start == nullptr) != (stop == nullptr)) return DETLM_EINVAL;
  h->t_start = start;
  h->t_stop = stop;
  return DETLM_OK;
}

int detlm_head_debug(detlm_head_t* h, int flags, uint64_t timeout_ns) {
  if (h == nullptr || (flags & ~DETLM_DEBUG_STALL) != 0) return DETLM_EINVAL;
  h->stall = (flags & DETLM_DEBUG_STALL) ? 1 : 0;
  h->timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
  return DETLM_OK;
}

int detlm_head_tiles(const detlm_head_t* h, int64_t B, int32_t* n_vtiles, int32_t* n_cols) {
  if (h == nullptr || bad_B(B) || n_vtiles == nullptr || n_cols == nullptr) return DETLM_EINVAL;
  *n_vtiles = h->n_vt;
  *n_cols = (h->dtype == DETLM_INT8 && B < kI8WideB) ? int8_cols_for(B, h->d) : cols_for(B);
  return DETLM_OK;
}

void detlm_head_destroy(detlm_head_t* h) {
  if (h == nullptr) return;
  // the handle's kernels and copies may still run on any stream: let them
  // finish before their memory (device, and mapped host memory that the
  // kernels write) is released
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  if (h->a_copy) {
    cudaStreamSynchronize(h->a_copy);
    cudaStreamDestroy(h->a_copy);
  }
  for (int k = 0; k < 2; ++k) {
    if (h->a_done[k]) cudaEventDestroy(h->a_done[k]);
    if (h->a_freed[k]) cudaEventDestroy(h->a_freed[k]);
    if (h->a_out[k]) cudaFree(h->a_out[k]);
  }
  if (h->a_in) cudaFree(h->a_in);
  if (h->ws) cudaFree(h->ws);
  if (h->vws) cudaFree(h->vws);
  if (h->q8) cudaFree(h->q8);
  if (h->W16) cudaFree(h->W16);
  if (h->h16) cudaFree(h->h16);
  if (h->stage) cudaFree(h->stage);
  if (h->err_mapped) cudaFreeHost(h->err_mapped);
  else if (h->d_err) cudaFree(h->d_err);
  if (h->err_host) cudaFreeHost(h->err_host);
  delete h;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Greedy call without any device allocation (see the header for who needs
// it). Its split-V records and error word live in this file-scope device
// array; host code obtains the array's device address once per device with
// cudaGetSymbolAddress (the host-side name is only a stand-in and must never
// be handed to a kernel).
static __device__ __align__(256) unsigned char detlm_noalloc_scratch[DETLM_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};
CUcontext g_noalloc_ctx[kNoAllocMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_once;

// The calling thread's current context (the one the symbol lookup is valid
// in), or nullptr when the driver entry point is unavailable.
CUcontext current_context() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  CUcontext c = nullptr;
  if (g_ctx_current == nullptr || g_ctx_current(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the scratch array on the current device, looked up with
// that device current the first time a context of it calls in; the cached
// address is keyed to the context, so a device reset (a new primary context)
// looks it up again.
int noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return DETLM_EUNSUPPORTED;
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr || ctx == nullptr || g_noalloc_ctx[dev] != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, detlm_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return DETLM_ECUDA;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = current_context();
  }
  *out = g_noalloc_ptr[dev];
  return DETLM_OK;
}

}  // namespace

extern "C" int detlm_greedy_noalloc(const void* W_dev, int64_t V, int64_t d, int dtype,
                                    const void* h_dev, int64_t B, int32_t* token_dev,
                                    float* gap_dev, float* logits_dev, int* err_dev,
                                    cudaStream_t stream) {
  if (dtype == DETLM_INT8) return DETLM_EUNSUPPORTED;
  if (dtype != DETLM_BF16 && dtype != DETLM_FP16) return DETLM_EINVAL;
  if (W_dev == nullptr || !aligned(W_dev, 16)) return DETLM_EINVAL;
  if (V < 1 || V >= (int64_t{1} << 31) || d < 1 || d >= (int64_t{1} << 31)) return DETLM_EINVAL;
  if ((d * 2) % 16 != 0) return DETLM_EINVAL;
  if (bad_B(B)) return DETLM_EINVAL;
  if (B == 0) return DETLM_OK;
  if (h_dev == nullptr || !aligned(h_dev, 16)) return DETLM_EINVAL;
  if (token_dev == nullptr || !aligned(token_dev, 4)) return DETLM_EINVAL;
  if (gap_dev == nullptr || !aligned(gap_dev, 4)) return DETLM_EINVAL;
  if (logits_dev != nullptr && !aligned(logits_dev, 4)) return DETLM_EINVAL;
  if (err_dev != nullptr && !aligned(err_dev, 4)) return DETLM_EINVAL;
  // scratch: error word (256 B), then rec_m, rec_i, rec_s [B, n_vt], each
  // part rounded up to 256 bytes
  const int n_vt = static_cast<int>((V + kBM - 1) / kBM);
  const size_t part = ws_part(static_cast<int64_t>(n_vt) * B);
  if (256 + 3 * part > DETLM_NOALLOC_SCRATCH_BYTES) return DETLM_EINVAL;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DETLM_ECUDA;
  int major = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || sms <= 0) return DETLM_ECUDA;
  if (!load_encode()) return DETLM_ECUDA;
  void* scratch = nullptr;
  int st = noalloc_scratch(dev, &scratch);
  if (st != DETLM_OK) return st;
  uint8_t* sb = static_cast<uint8_t*>(scratch);
  int* err = err_dev != nullptr ? err_dev : reinterpret_cast<int*>(sb);
  float* rec_m = reinterpret_cast<float*>(sb + 256);
  int32_t* rec_i = reinterpret_cast<int32_t*>(sb + 256 + part);
  float* rec_s = reinterpret_cast<float*>(sb + 256 + 2 * part);

  const int N = cols_for(B);
  CUtensorMap tmW, tmH;
  if (!encode_2d(&tmW, dtype, W_dev, d, V, kBM)) return DETLM_EINVAL;
  if (!encode_2d(&tmH, dtype, h_dev, d, B, static_cast<uint32_t>(N))) return DETLM_EINVAL;

  HeadParams p;
  std::memset(&p, 0, sizeof(p));
  p.V = static_cast<int32_t>(V);
  p.d = static_cast<int32_t>(d);
  p.B = static_cast<int32_t>(B);
  p.N = N;
  p.n_vt = n_vt;
  p.n_nt = static_cast<int32_t>((B + N - 1) / N);
  p.nk = static_cast<int32_t>((d * 2 + kRowBytes - 1) / kRowBytes);
  p.n_chunks = static_cast<int32_t>((d + kChunkK - 1) / kChunkK);
  p.n_slots = slots_for(N);
  p.stages = stages_for(N);
  p.n_issuers = issuers_for(N, p.stages, &p.n_slots);
  p.tmem_cols = tmem_cols_for(p.n_slots * N);
  p.idesc = idesc_f16(dtype == DETLM_BF16 ? 1u : 0u, kBM, static_cast<uint32_t>(N));
  p.logits = logits_dev;
  p.rec_m = rec_m;
  p.rec_i = rec_i;
  p.rec_s = rec_s;
  p.err = err;
  p.timeout_ns = kDefaultTimeoutNs;

  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), stream);   // must start at zero
  if (e != cudaSuccess) return status_from_cuda(e);
  const size_t smem = smem_layout(N, p.stages).total + 1024;
  const int64_t units = static_cast<int64_t>(p.n_vt) * p.n_nt;
  const int grid = static_cast<int>(units < sms ? units : sms);
  e = launch_gemm<MODE_GREEDY>(tmW, tmH, p, grid, smem, stream);
  if (e != cudaSuccess) return status_from_cuda(e);

  MergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  mp.V = p.V;
  mp.B = p.B;
  mp.n_vt = p.n_vt;
  mp.rec_m = rec_m;
  mp.rec_i = rec_i;
  mp.rec_s = rec_s;
  mp.token = token_dev;
  mp.gap = gap_dev;
  mp.err = err;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, merge_kernel<MODE_GREEDY>, mp);
  return status_from_cuda(e);
}
