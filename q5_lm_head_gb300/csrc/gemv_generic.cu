// Generic output-stage path: any batch (1..32), any K that is a multiple of 256.
//
//   launch 1 (only when gamma is given): final RMSNorm of each hidden row into
//            the handle's x buffer ("Chapter 20 — Final norm, LM head, and the
//            soft cap" §20.1: x = h / sqrt(mean(h^2) + eps) * gamma)
//   launch 2: one warp per weight row; every lane dequantises 8 weights of each
//            Q5_K (or Q4_K) block (w = d*sc*q - dmin*m, §20.3 block) straight from global
//            memory, multiplies them with x (read through L1), warp-shuffle
//            reduction, scale + soft cap epilogue (§20.4), and the two-level argmax
//            (per-CTA shared-memory max, then one global atomic per CTA and row).
//
// This path favours simplicity over speed; the batch-1 and tensor-core kernels
// are the fast paths.
#include "common.cuh"
#include "internal.h"

namespace muse {
namespace {

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_rows_kernel(const float *__restrict__ hidden, const float *__restrict__ gamma, float eps,
                        int k, float *__restrict__ x) {
  __shared__ float s_part[kNormThreads / 32];
  const int b = blockIdx.x;
  const float *h = hidden + static_cast<size_t>(b) * k;
  float ss = 0.0f;
  for (int j = threadIdx.x * 4; j < k; j += kNormThreads * 4) {
    const float4 v = *reinterpret_cast<const float4 *>(h + j);
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
  for (int i = 0; i < kNormThreads / 32; ++i) tot += s_part[i];
  const float r = 1.0f / sqrtf(tot / static_cast<float>(k) + eps);
  float *xo = x + static_cast<size_t>(b) * k;
  for (int j = threadIdx.x * 4; j < k; j += kNormThreads * 4) {
    const float4 v = *reinterpret_cast<const float4 *>(h + j);
    const float4 g = *reinterpret_cast<const float4 *>(gamma + j);
    float4 o;
    o.x = v.x * r * g.x;
    o.y = v.y * r * g.y;
    o.z = v.z * r * g.z;
    o.w = v.w * r * g.w;
    *reinterpret_cast<float4 *>(xo + j) = o;
  }
}

constexpr int kGemvThreads = 256;
constexpr int kBatchTile = 4;

template <bool kQ4>
__global__ void __launch_bounds__(kGemvThreads)
    gemv_generic_kernel(const uint8_t *__restrict__ w, const float *__restrict__ x, int batch,
                        int64_t n_rows, int k, float scale, float cap, float *__restrict__ logits,
                        unsigned long long *keys, unsigned int *ticket, int32_t *argmax, int argmax_precap) {
  __shared__ unsigned long long s_best[32];
  const int lane = threadIdx.x & 31;
  const int c = lane >> 3;   // 64-weight group inside a block: sub-blocks 2c and 2c+1
  const int j4 = lane & 7;   // positions l = 4*j4 .. 4*j4+3 of those sub-blocks
  const int nb = k / kBlockWeights;
  if (threadIdx.x < 32) s_best[threadIdx.x] = 0ull;
  __syncthreads();

  const int64_t warps_per_cta = kGemvThreads / 32;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * warps_per_cta;
  for (int64_t row = blockIdx.x * warps_per_cta + (threadIdx.x >> 5); row < n_rows; row += n_warps) {
    constexpr int kBB = kQ4 ? kBlockBytesQ4 : kBlockBytes;
    const uint8_t *wrow = w + row * nb * kBB;
    for (int b0 = 0; b0 < batch; b0 += kBatchTile) {
      float acc[kBatchTile];
#pragma unroll
      for (int t = 0; t < kBatchTile; ++t) acc[t] = 0.0f;
      for (int kb = 0; kb < nb; ++kb) {
        const uint8_t *blk = wrow + kb * kBB;
        const uint4 hdr = __ldg(reinterpret_cast<const uint4 *>(blk));
        const uint32_t qh = kQ4 ? 0u : __ldg(reinterpret_cast<const uint32_t *>(blk + kOffQh) + j4);
        const uint32_t qs = __ldg(reinterpret_cast<const uint32_t *>(blk + (kQ4 ? kOffQsQ4 : kOffQs) + 32 * c) + j4);
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
        const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
        int sc0, m0, sc1, m1;
        q5k_scale_min(hdr.y, hdr.z, hdr.w, 2 * c, sc0, m0);
        q5k_scale_min(hdr.y, hdr.z, hdr.w, 2 * c + 1, sc1, m1);
        const float a0 = d * static_cast<float>(sc0), n0 = dmin * static_cast<float>(m0);
        const float a1 = d * static_cast<float>(sc1), n1 = dmin * static_cast<float>(m1);
        float wl[4], wh[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ql = ((qs >> (8 * i)) & 15) | (((qh >> (8 * i + 2 * c)) & 1) << 4);
          const int qv = ((qs >> (8 * i + 4)) & 15) | (((qh >> (8 * i + 2 * c + 1)) & 1) << 4);
          wl[i] = fmaf(a0, static_cast<float>(ql), -n0);
          wh[i] = fmaf(a1, static_cast<float>(qv), -n1);
        }
        const int col = kb * kBlockWeights + 64 * c + 4 * j4;
#pragma unroll
        for (int t = 0; t < kBatchTile; ++t) {
          if (b0 + t < batch) {
            const float *xb = x + static_cast<size_t>(b0 + t) * k + col;
            const float4 xl = __ldg(reinterpret_cast<const float4 *>(xb));
            const float4 xh = __ldg(reinterpret_cast<const float4 *>(xb + 32));
            float s = acc[t];
            s = fmaf(wl[0], xl.x, s);
            s = fmaf(wl[1], xl.y, s);
            s = fmaf(wl[2], xl.z, s);
            s = fmaf(wl[3], xl.w, s);
            s = fmaf(wh[0], xh.x, s);
            s = fmaf(wh[1], xh.y, s);
            s = fmaf(wh[2], xh.z, s);
            s = fmaf(wh[3], xh.w, s);
            acc[t] = s;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kBatchTile; ++t) {
        float s = acc[t];
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == t && b0 + t < batch) {
          const float out = scale_softcap(s, scale, cap);
          logits[static_cast<size_t>(b0 + t) * n_rows + row] = out;
          if (argmax)
            atomicMax(&s_best[b0 + t], argmax_key(argmax_precap ? s * scale : out, static_cast<uint32_t>(row)));
        }
      }
    }
  }
  if (argmax) {
    __syncthreads();
    if (threadIdx.x < batch && s_best[threadIdx.x] != 0ull) atomicMax(keys + threadIdx.x, s_best[threadIdx.x]);
    argmax_finish(keys, ticket, argmax, batch);
  }
}

}  // namespace

int generic_launches(const LaunchArgs &a) { return a.gamma ? 2 : 1; }

cudaError_t launch_generic(const LaunchArgs &a) {
  const float *x = a.hidden;
  if (a.gamma) {
    rmsnorm_rows_kernel<<<a.batch, kNormThreads, 0, a.stream>>>(a.hidden, a.gamma, a.eps, a.k, a.ws.x);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    x = a.ws.x;
  }
  const int64_t warps_needed = a.n_rows;
  int64_t blocks = (warps_needed + (kGemvThreads / 32) - 1) / (kGemvThreads / 32);
  const int64_t cap_blocks = static_cast<int64_t>(a.num_sms) * 8;
  if (blocks > cap_blocks) blocks = cap_blocks;
  if (a.q4)
    gemv_generic_kernel<true><<<static_cast<unsigned>(blocks), kGemvThreads, 0, a.stream>>>(
        a.w, x, a.batch, a.n_rows, a.k, a.scale, a.cap, a.logits, a.ws.keys, a.ws.ticket, a.argmax,
        a.argmax_precap ? 1 : 0);
  else
    gemv_generic_kernel<false><<<static_cast<unsigned>(blocks), kGemvThreads, 0, a.stream>>>(
        a.w, x, a.batch, a.n_rows, a.k, a.scale, a.cap, a.logits, a.ws.keys, a.ws.ticket, a.argmax,
        a.argmax_precap ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace muse
