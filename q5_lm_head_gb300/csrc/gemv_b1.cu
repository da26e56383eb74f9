// Fused batch-1 output stage: final RMSNorm prologue, Q5_K weight-streaming
// GEMV on the CUDA cores, scale + soft cap epilogue and two-level argmax, in
// one persistent launch ("Chapter 20 — Final norm, LM head, and the soft cap",
// §20.1 what it computes, §20.3 the 924.6 MB weight stream, §20.4 the cap).
//
// Layout of the work
//   * A tile is kRows consecutive weight rows: kRows * (K/256) * 176 bytes,
//     contiguous in HBM.  CTAs take tiles round-robin (tile = blockIdx.x +
//     i * gridDim.x), so at any moment the whole GPU streams one contiguous
//     stretch of the matrix.
//   * One producer warp moves tiles into a ring of shared-memory stages with
//     1-D bulk copies (cp.async.bulk, mbarrier transaction counts, L2
//     evict-first); consumers release stages through "empty" mbarriers.  Every
//     wait is bounded.
//   * Consumer thread (kb, c) owns 64 columns: block kb, sub-blocks 2c and 2c+1.
//     Its 64 normalised activations live in registers for the whole launch
//     (column-stationary), so shared memory carries weights only.  The CTA has
//     four such teams ("streams"), each taking every fourth row of a tile.
//   * Per sub-block s the thread forms sum_j q_j x_j.  A 5-bit q is turned into
//     the float 1 + q/128 by placing (0x80 | q) under the exponent byte 0x3F
//     with one byte permute; the chain starts at -sum_j x_j, so it ends at
//     sum_j q_j x_j / 128 with no integer->float conversion per weight.  Then
//     raw += d*128*sc_s*that - dmin*m_s*sum_j x_j.
//   * Per-row partials (one per thread) meet in shared memory; one warp per row
//     sums them, applies scale and cap, stores the logit and keeps the running
//     argmax key.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace muse {
namespace {

constexpr int kRows = 8;            // weight rows per pipeline stage
constexpr int kStreams = 4;         // row teams per CTA
constexpr int kMaxSmem = 227 * 1024;

template <int NB>
struct B1Cfg {
  static constexpr int kUnits = 4 * NB;                    // (block, 64-column group) units per row
  static constexpr int kConsumers = kUnits * kStreams;
  static_assert(kConsumers % 32 == 0, "consumer threads must fill whole warps");
  static constexpr int kConsumerWarps = kConsumers / 32;
  static_assert(kConsumerWarps >= kRows, "one reducing warp per row of a stage");
  static constexpr int kThreads = kConsumers + 32;         // + one producer warp
  static constexpr int kRowBytes = NB * kBlockBytes;
  static constexpr int kStageBytes = kRows * kRowBytes;
  static constexpr int kPartialBytes = 2 * kRows * kUnits * 4;
  static constexpr int kFixedBytes = kPartialBytes + 1024;  // partials + barriers + scratch
  static constexpr int kStagesFit = (kMaxSmem - kFixedBytes) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static_assert(kStages >= 2, "need at least double buffering");
  static constexpr int kSmemBytes = kStages * kStageBytes + kFixedBytes;
};

// 1 + q/128 as a float, from byte `t` of Q (that byte holds 0x80 | q, q < 32).
template <int T>
__device__ __forceinline__ float q_as_float(uint32_t q4) {
  // result bytes (high..low): 0x3F, Q.byte[T], 0x00, 0x00
  return __uint_as_float(__byte_perm(q4, 0x3Fu, 0x4055u | (T << 8)));
}

template <int NB>
__global__ void __launch_bounds__(B1Cfg<NB>::kThreads, 1)
    gemv_b1_kernel(const float *__restrict__ hidden, const float *__restrict__ gamma, float eps,
                   const uint8_t *__restrict__ w, int64_t n_rows, float scale, float cap,
                   float *__restrict__ logits, unsigned long long *keys, unsigned int *ticket,
                   int32_t *argmax, uint32_t *status) {
  using C = B1Cfg<NB>;
  constexpr int K = NB * kBlockWeights;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *stages = smem;
  float *partial = reinterpret_cast<float *>(smem + C::kStages * C::kStageBytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStageBytes + C::kPartialBytes);
  uint64_t *empty = full + C::kStages;
  float *s_red = reinterpret_cast<float *>(empty + C::kStages);           // [32]
  unsigned long long *s_best = reinterpret_cast<unsigned long long *>(s_red + 32);
  uint32_t *s_abort = reinterpret_cast<uint32_t *>(s_best + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t n_tiles = (n_rows + kRows - 1) / kRows;

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], C::kConsumerWarps);
    }
    *s_best = 0ull;
    *s_abort = 0u;
    ptx::fence_barrier_init();
  }
  __syncthreads();

  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = ptx::policy_evict_first();
      int64_t issued = 0;
      for (int64_t it = 0;; ++it) {
        const int64_t tile = blockIdx.x + it * gridDim.x;
        if (tile >= n_tiles) break;
        const int st = static_cast<int>(it % C::kStages);
        if (it >= C::kStages) {
          const uint32_t par = static_cast<uint32_t>((it / C::kStages - 1) & 1);
          if (*reinterpret_cast<volatile uint32_t *>(s_abort) || !ptx::mbar_wait(&empty[st], par)) {
            atomicOr(status, kStatusWaitTimeout);
            *reinterpret_cast<volatile uint32_t *>(s_abort) = 1u;
            break;
          }
        }
        const int64_t r0 = tile * kRows;
        const int rows = static_cast<int>(n_rows - r0 < kRows ? n_rows - r0 : kRows);
        const uint32_t bytes = static_cast<uint32_t>(rows * C::kRowBytes);
        ptx::mbar_arrive_expect_tx(&full[st], bytes);
        ptx::bulk_g2s(stages + st * C::kStageBytes, w + r0 * C::kRowBytes, bytes, &full[st], policy);
        issued = it + 1;
      }
      // Never leave the CTA with copies in flight: wait (bounded) for the last
      // stage fills this warp armed.  In a normal run they completed long ago.
      for (int64_t it = issued > C::kStages ? issued - C::kStages : 0; it < issued; ++it)
        ptx::mbar_wait(&full[it % C::kStages], static_cast<uint32_t>((it / C::kStages) & 1));
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int stream = tid / C::kUnits;
    const int u = tid % C::kUnits;
    const int kb = u >> 2, c = u & 3;

    // Final RMSNorm prologue (every CTA recomputes r from the L2-resident hidden row).
    float r = 1.0f;
    if (gamma) {
      float ss = 0.0f;
      for (int j = tid * 4; j < K; j += C::kConsumers * 4) {
        const float4 v = *reinterpret_cast<const float4 *>(hidden + j);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_red[warp] = ss;
      ptx::named_bar_sync(1, C::kConsumers);
      float tot = 0.0f;
      for (int i = 0; i < C::kConsumerWarps; ++i) tot += s_red[i];
      r = 1.0f / sqrtf(tot / static_cast<float>(K) + eps);
    }
    // This thread's 64 activations: x_lo[l] for sub-block 2c, x_hi[l] for 2c+1.
    float x_lo[32], x_hi[32];
    const int col = kb * kBlockWeights + 64 * c;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 hl = *reinterpret_cast<const float4 *>(hidden + col + 4 * i);
      float4 hh = *reinterpret_cast<const float4 *>(hidden + col + 32 + 4 * i);
      if (gamma) {
        const float4 gl = *reinterpret_cast<const float4 *>(gamma + col + 4 * i);
        const float4 gh = *reinterpret_cast<const float4 *>(gamma + col + 32 + 4 * i);
        hl = make_float4(hl.x * r * gl.x, hl.y * r * gl.y, hl.z * r * gl.z, hl.w * r * gl.w);
        hh = make_float4(hh.x * r * gh.x, hh.y * r * gh.y, hh.z * r * gh.z, hh.w * r * gh.w);
      }
      x_lo[4 * i + 0] = hl.x; x_lo[4 * i + 1] = hl.y; x_lo[4 * i + 2] = hl.z; x_lo[4 * i + 3] = hl.w;
      x_hi[4 * i + 0] = hh.x; x_hi[4 * i + 1] = hh.y; x_hi[4 * i + 2] = hh.z; x_hi[4 * i + 3] = hh.w;
    }
    float sx_lo = 0.0f, sx_hi = 0.0f;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
      sx_lo += x_lo[l];
      sx_hi += x_hi[l];
    }
    const int sh_lo = 2 * c, sh_hi = 2 * c + 1;   // qh bit of each sub-block

    unsigned long long best = 0ull;
    for (int64_t it = 0;; ++it) {
      const int64_t tile = blockIdx.x + it * gridDim.x;
      if (tile >= n_tiles) break;
      const int st = static_cast<int>(it % C::kStages);
      const bool ok = ptx::mbar_wait(&full[st], static_cast<uint32_t>((it / C::kStages) & 1));
      const int64_t r0 = tile * kRows;
      const int rows = static_cast<int>(n_rows - r0 < kRows ? n_rows - r0 : kRows);
      float *part = partial + (it & 1) * (kRows * C::kUnits);
      const uint8_t *sbase = stages + st * C::kStageBytes;
#pragma unroll 1
      for (int rr = 0; rr < kRows / kStreams; ++rr) {
        const int rl = stream + rr * kStreams;
        if (ok && rl < rows) {
          const uint8_t *blk = sbase + rl * C::kRowBytes + kb * kBlockBytes;
          const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
          const uint4 qh0 = *reinterpret_cast<const uint4 *>(blk + kOffQh);
          const uint4 qh1 = *reinterpret_cast<const uint4 *>(blk + kOffQh + 16);
          const uint4 qs0 = *reinterpret_cast<const uint4 *>(blk + kOffQs + 32 * c);
          const uint4 qs1 = *reinterpret_cast<const uint4 *>(blk + kOffQs + 32 * c + 16);
          const uint32_t H[8] = {qh0.x, qh0.y, qh0.z, qh0.w, qh1.x, qh1.y, qh1.z, qh1.w};
          const uint32_t A[8] = {qs0.x, qs0.y, qs0.z, qs0.w, qs1.x, qs1.y, qs1.z, qs1.w};
          float acc_lo0 = -sx_lo, acc_lo1 = 0.0f, acc_hi0 = -sx_hi, acc_hi1 = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t qlo = (A[i] & 0x0F0F0F0Fu) | (((H[i] >> sh_lo) & 0x01010101u) << 4) | 0x80808080u;
            const uint32_t qhi = ((A[i] >> 4) & 0x0F0F0F0Fu) | (((H[i] >> sh_hi) & 0x01010101u) << 4) | 0x80808080u;
            acc_lo0 = fmaf(q_as_float<0>(qlo), x_lo[4 * i + 0], acc_lo0);
            acc_lo1 = fmaf(q_as_float<1>(qlo), x_lo[4 * i + 1], acc_lo1);
            acc_lo0 = fmaf(q_as_float<2>(qlo), x_lo[4 * i + 2], acc_lo0);
            acc_lo1 = fmaf(q_as_float<3>(qlo), x_lo[4 * i + 3], acc_lo1);
            acc_hi0 = fmaf(q_as_float<0>(qhi), x_hi[4 * i + 0], acc_hi0);
            acc_hi1 = fmaf(q_as_float<1>(qhi), x_hi[4 * i + 1], acc_hi1);
            acc_hi0 = fmaf(q_as_float<2>(qhi), x_hi[4 * i + 2], acc_hi0);
            acc_hi1 = fmaf(q_as_float<3>(qhi), x_hi[4 * i + 3], acc_hi1);
          }
          const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
          const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
          int sc0, m0, sc1, m1;
          q5k_scale_min(hdr.y, hdr.z, hdr.w, 2 * c, sc0, m0);
          q5k_scale_min(hdr.y, hdr.z, hdr.w, 2 * c + 1, sc1, m1);
          const float dot_lo = acc_lo0 + acc_lo1;   // sum q x / 128 over sub-block 2c
          const float dot_hi = acc_hi0 + acc_hi1;
          const float main = fmaf(static_cast<float>(sc0), dot_lo, static_cast<float>(sc1) * dot_hi);
          const float mins = fmaf(static_cast<float>(m0), sx_lo, static_cast<float>(m1) * sx_hi);
          part[rl * C::kUnits + u] = fmaf(d * 128.0f, main, -dmin * mins);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[st]);
      // All consumers learn together whether any of them timed out, so none is
      // left waiting at a barrier the others have abandoned.
      if (ptx::named_bar_red_or(1, C::kConsumers, !ok)) {
        if (tid == 0) {
          atomicOr(status, kStatusWaitTimeout);
          *reinterpret_cast<volatile uint32_t *>(s_abort) = 1u;
        }
        break;
      }
      if (warp < rows) {
        float s = 0.0f;
        for (int j = lane; j < C::kUnits; j += 32) s += part[warp * C::kUnits + j];
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) {
          const int64_t row = r0 + warp;
          const float out = scale_softcap(s, scale, cap);
          logits[row] = out;
          best = umax64(best, argmax_key(out, static_cast<uint32_t>(row)));
        }
      }
    }
    if (argmax && lane == 0 && best != 0ull) atomicMax(s_best, best);
  }

  if (argmax) {
    __syncthreads();
    if (tid == 0 && *s_best != 0ull) atomicMax(keys, *s_best);
    argmax_finish(keys, ticket, argmax, 1);
  }
}

template <int NB>
cudaError_t launch_b1_nb(const LaunchArgs &a) {
  using C = B1Cfg<NB>;
  static unsigned long long configured = 0;   // one bit per device: the attribute is per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    e = cudaFuncSetAttribute(gemv_b1_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured |= bit;
  }
  const int64_t n_tiles = (a.n_rows + kRows - 1) / kRows;
  const int64_t grid = n_tiles < a.num_sms ? n_tiles : a.num_sms;
  gemv_b1_kernel<NB><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, a.stream>>>(
      a.hidden, a.gamma, a.eps, a.w, a.n_rows, a.scale, a.cap, a.logits, a.ws.keys, a.ws.ticket,
      a.argmax, a.ws.status);
  return cudaGetLastError();
}

}  // namespace

bool b1_supported(int k) { return k == 26 * kBlockWeights || k == 16 * kBlockWeights; }

cudaError_t launch_b1(const LaunchArgs &a) {
  switch (a.k / kBlockWeights) {
    case 26: return launch_b1_nb<26>(a);
    case 16: return launch_b1_nb<16>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace muse
