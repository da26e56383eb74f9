// Device helpers shared by the output-stage kernels (sm_103a).
//
// The arithmetic follows "Chapter 20 — Final norm, LM head, and the soft cap":
// final RMSNorm (§20.1), Q5_K dequantisation w = d*sc*q - dmin*m (§20.3 block
// of 256 weights in 176 bytes, ggml block_q5_K layout), scale then soft cap
// (§20.1/§20.4), and the greedy argmax that the strictly increasing cap leaves
// unchanged (§20.2).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace muse {

constexpr int kBlockWeights = 256;
constexpr int kBlockBytes = 176;
// byte offsets inside a Q5_K block
constexpr int kOffD = 0, kOffDmin = 2, kOffScales = 4, kOffQh = 16, kOffQs = 48;
// Q4_K block (144 bytes): the same d, dmin and scale bytes, then the nibbles
// (no high bits); ggml's block_q4_K, the FFN bulk's format.
constexpr int kBlockBytesQ4 = 144;
constexpr int kOffQsQ4 = 16;

// Scale then soft cap: v = raw * scale; cap > 0 ? cap * tanh(v / cap) : v.
__device__ __forceinline__ float scale_softcap(float raw, float scale, float cap) {
  float v = raw * scale;
  return cap > 0.0f ? cap * tanhf(v / cap) : v;
}

// 6-bit scale and min of sub-block s from the 12 packed scale bytes held as
// three little-endian words w0 = bytes 0..3, w1 = 4..7, w2 = 8..11.
__device__ __forceinline__ void q5k_scale_min(uint32_t w0, uint32_t w1, uint32_t w2, int s,
                                              int &sc, int &m) {
  if (s < 4) {
    sc = (w0 >> (8 * s)) & 63;
    m = (w1 >> (8 * s)) & 63;
  } else {
    const int j = s - 4;
    const uint32_t b8 = (w2 >> (8 * j)) & 0xFF;
    sc = (b8 & 15) | (((w0 >> (8 * j + 6)) & 3) << 4);
    m = (b8 >> 4) | (((w1 >> (8 * j + 6)) & 3) << 4);
  }
}

// Online (max, sum of exp) pair of a set of values: s = sum_j exp(v_j - m).
// The empty set is (-inf, 0).  log-softmax normaliser of the set: m + log(s).
struct MaxSum {
  float m, s;
};

__device__ __forceinline__ MaxSum ms_empty() { return {-INFINITY, 0.0f}; }

__device__ __forceinline__ MaxSum ms_add(MaxSum a, float v) {
  if (v <= a.m) {
    a.s += expf(v - a.m);
  } else {
    a.s = a.s * expf(a.m - v) + 1.0f;   // a.m = -inf: 0 * 0 + 1
    a.m = v;
  }
  return a;
}

__device__ __forceinline__ MaxSum ms_combine(MaxSum a, MaxSum b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return a;         // both empty
  return {m, a.s * expf(a.m - m) + b.s * expf(b.m - m)};
}

__device__ __forceinline__ MaxSum ms_warp_combine(MaxSum a) {
  for (int o = 16; o > 0; o >>= 1) {
    MaxSum b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
    a = ms_combine(a, b);
  }
  return a;
}

// Total order on finite floats as unsigned keys; -0 is folded onto +0 first.
__device__ __forceinline__ uint32_t float_order_key(float v) {
  v = v + 0.0f;
  uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Packed (value, index) key: larger value wins, then the lower index.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  return ((unsigned long long)float_order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

// The warp's largest argmax_key over its lanes' (v, idx), or 0 where no lane
// is valid: the highest value bits first, then the highest index bits among
// the lanes holding them (two warp reductions instead of a 64-bit butterfly).
__device__ __forceinline__ unsigned long long warp_argmax_key(float v, uint32_t idx, bool valid) {
  const uint32_t hi = valid ? float_order_key(v) : 0u;
  const uint32_t lo = valid ? 0xFFFFFFFFu - idx : 0u;
  const uint32_t m_hi = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t m_lo = __reduce_max_sync(0xffffffffu, hi == m_hi ? lo : 0u);
  return ((unsigned long long)m_hi << 32) | m_lo;
}

__device__ __forceinline__ uint32_t argmax_key_index(unsigned long long key) {
  return 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// Second level of the argmax: every CTA has folded its per-row best into
// keys[b] with atomicMax.  The CTA that finishes last (atomic ticket; no CTA
// waits on another) turns keys into indices and re-arms keys and ticket for the
// next forward.  Called by all threads of the CTA.
__device__ __forceinline__ void argmax_finish(unsigned long long *keys, unsigned int *ticket,
                                              int32_t *argmax, int batch) {
  __shared__ unsigned int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int t = atomicAdd(ticket, 1u);
    s_last = (t == gridDim.x - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
      unsigned long long key = atomicExch(keys + b, 0ull);
      argmax[b] = (int32_t)argmax_key_index(key);
    }
    if (threadIdx.x == 0) atomicExch(ticket, 0u);
  }
}

// Same result as argmax_finish, for a CTA whose per-batch-row keys sit in
// shared memory (cta_keys[b], 0 = none; final when the CTA calls this): one
// thread adds them with fire-and-forget max reductions and takes a ticket with
// acquire-release semantics (the release orders its reductions before the
// ticket), so the CTA pays a single global round trip; the last CTA reads the
// keys (acquire through the ticket) and re-arms keys and ticket.
__device__ __forceinline__ void argmax_publish_finish(unsigned long long *keys, unsigned int *ticket,
                                                      int32_t *argmax, const unsigned long long *cta_keys,
                                                      int batch) {
  __shared__ unsigned int s_last;
  if (threadIdx.x == 0) {
    for (int b = 0; b < batch; ++b)
      if (cta_keys[b] != 0ull)
        asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(keys + b), "l"(cta_keys[b]) : "memory");
    unsigned int t;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(t) : "l"(ticket) : "memory");
    s_last = (t == gridDim.x - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (s_last) {
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
      unsigned long long key;
      asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(key) : "l"(keys + b) : "memory");
      argmax[b] = (int32_t)argmax_key_index(key);
      asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(keys + b), "l"(0ull) : "memory");
    }
    if (threadIdx.x == 0) asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(ticket), "r"(0u) : "memory");
  }
}

}  // namespace muse
