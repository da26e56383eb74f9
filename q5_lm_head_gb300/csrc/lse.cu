// Logprobs over the capped logits: softmax and logprobs are taken over the
// logits after scale and cap ("Chapter 20 — Final norm, LM head, and the soft
// cap", §20.7), logprob_i = logit_i - lse with lse = log sum_j exp(logit_j)
// per batch row.
//
// Two small kernels over finished logits [batch][n_rows]:
//   lse_parts_kernel     one CTA per (chunk, row): the chunk's online (max, sum exp)
//                        pair.  The batch-1 kernel writes one such pair per CTA
//                        from its row epilogue instead, so it needs no extra pass.
//                        Launched as a programmatic dependent of the kernel that
//                        wrote the logits, like the apply kernel below.
//   logprob_apply_kernel every CTA combines the row's pairs in a fixed order
//                        (all CTAs get the same lse bit for bit), CTA 0 stores
//                        lse, and each CTA subtracts it from its chunk in place.
//                        Launched as a programmatic dependent of the kernel
//                        that wrote logits and pairs: its launch overlaps that
//                        kernel and griddepcontrol.wait orders the reads.
#include "common.cuh"
#include "internal.h"

namespace muse {
namespace {

constexpr int kLseThreads = 256;
constexpr int64_t kPartChunk = 2048;    // logits per (max, sum exp) pair of lse_parts_kernel, at least
constexpr int64_t kApplyChunk = 8192;   // logits per CTA of the apply kernel

__device__ __forceinline__ MaxSum block_combine(MaxSum a, MaxSum *s_part) {
  a = ms_warp_combine(a);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_part[warp] = a;
  __syncthreads();
  MaxSum r = ms_empty();
  for (int w = 0; w < kLseThreads / 32; ++w) r = ms_combine(r, s_part[w]);
  return r;
}

__global__ void __launch_bounds__(kLseThreads)
    lse_parts_kernel(const float *__restrict__ logits, int64_t n_rows, int64_t chunk, float2 *__restrict__ parts) {
  __shared__ MaxSum s_part[kLseThreads / 32];
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the logits are complete
  const int b = blockIdx.y;
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * chunk;
  const int64_t hi = lo + chunk < n_rows ? lo + chunk : n_rows;
  const float *row = logits + static_cast<int64_t>(b) * n_rows;
  MaxSum a = ms_empty();
  for (int64_t i = lo + threadIdx.x; i < hi; i += kLseThreads) a = ms_add(a, row[i]);
  a = block_combine(a, s_part);
  if (threadIdx.x == 0) parts[static_cast<int64_t>(b) * kMaxLseParts + blockIdx.x] = make_float2(a.m, a.s);
}

__global__ void __launch_bounds__(kLseThreads)
    logprob_apply_kernel(float *__restrict__ logits, int64_t n_rows, const float2 *__restrict__ parts,
                         int n_parts, float *__restrict__ lse) {
  __shared__ float s_lse;
  asm volatile("griddepcontrol.wait;" ::: "memory");   // logits and pairs are complete
  const int b = blockIdx.y;
  if (threadIdx.x < 32) {                               // fixed order: lane l folds pairs l, l+32, ...
    MaxSum a = ms_empty();
    for (int p = threadIdx.x; p < n_parts; p += 32) {
      const float2 v = parts[static_cast<int64_t>(b) * kMaxLseParts + p];
      a = ms_combine(a, {v.x, v.y});
    }
    a = ms_warp_combine(a);
    if (threadIdx.x == 0) {
      s_lse = a.m + logf(a.s);
      if (lse && blockIdx.x == 0) lse[b] = s_lse;
    }
  }
  __syncthreads();
  const float l = s_lse;
  float *row = logits + static_cast<int64_t>(b) * n_rows;
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * kApplyChunk;
  const int64_t hi = lo + kApplyChunk < n_rows ? lo + kApplyChunk : n_rows;
  for (int64_t i = lo + threadIdx.x; i < hi; i += kLseThreads) row[i] -= l;
}

}  // namespace

int lse_parts_for(int64_t n_rows) {
  const int64_t n = (n_rows + kPartChunk - 1) / kPartChunk;
  return static_cast<int>(n < kMaxLseParts ? n : kMaxLseParts);
}

cudaError_t launch_lse_parts(const float *logits, int batch, int64_t n_rows, float2 *parts, cudaStream_t stream) {
  const int n = lse_parts_for(n_rows);
  const int64_t chunk = (n_rows + n - 1) / n;           // n chunks cover every row
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n), batch);
  cfg.blockDim = dim3(kLseThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lse_parts_kernel, logits, n_rows, chunk, parts);
}

cudaError_t launch_logprob_apply(float *logits, int batch, int64_t n_rows, const float2 *parts, int n_parts,
                                 float *lse, cudaStream_t stream) {
  if (n_parts < 1 || n_parts > kMaxLseParts) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n_rows + kApplyChunk - 1) / kApplyChunk), batch);
  cfg.blockDim = dim3(kLseThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, logprob_apply_kernel, logits, n_rows, parts, n_parts, lse);
}

}  // namespace muse
