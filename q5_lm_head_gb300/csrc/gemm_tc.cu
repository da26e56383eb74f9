// Batched output stage on the 5th-generation tensor cores (tcgen05), for
// batches of 2..32 rows: final RMSNorm, Q5_K LM-head contraction, scale + soft
// cap, argmax ("Chapter 20 — Final norm, LM head, and the soft cap", §20.1,
// §20.3, §20.4).  Two launches per forward:
//
// 1. prep_x_kernel: one CTA per Q5_K block column kb.  Normalises the hidden
//    rows and writes, per block, an "activation package" already in the
//    tensor-core operand layout (K-major, 8-row x 16-byte core matrices):
//      x     [2*NM rows][256]  rows 0..NM-1: f16(x); rows NM..2NM-1: f16(x - f16(x))
//                              (the two rows of a batch row sum to x to ~2^-22)
//      x_min [NM rows][16]     k < 8: f16 hi of S_s = sum of x over sub-block s,
//                              k >= 8: its f16 remainder
//    Rows >= batch are zero.
//
// 2. gemm_tc_kernel: a persistent CTA per SM works on pairs of 128-row tiles.
//    * producer warp: per block kb, one 2-D TMA box of 256 rows x 176 bytes
//      (both tiles of the pair) into a ring of weight stages, and the kb
//      activation package (1-D bulk copy) into a ring of package stages.
//    * two unpack warpgroups, one per tile: thread r owns row r.  It turns its
//      row's block into A[r][e] = sc_s * q_e as f16 (exact: at most 31*63) and
//      A_min[r][k] = m_(k mod 8), stores them into tensor memory
//      (tcgen05.st), and after the block's MMAs reads back D[r][b] and
//      Dmin[r][b] (tcgen05.ld) to accumulate
//          raw[r][b] += d * D[r][b] - dmin * Dmin[r][b]
//      which is sum_e (d*sc_s*q_e - dmin*m_s) * x[b][e] for the block.
//    * MMA warp (the whole warp runs the loop with warp-uniform operands, one
//      elected lane issues): per tile and block, 16 K-steps of f16 MMAs with f32
//      accumulation into D (M = 128, N = 2*NM: the x_hi and x_lo rows side by
//      side) and one MMA A_min x x_min into Dmin; tcgen05.commit hands the tile
//      back.
//    Each warpgroup has one A buffer and one D pair in tensor memory.  One
//    mbarrier pair per warpgroup paces everything: "A ready, D read" and
//    "A consumed, D written".
//    Epilogue per tile: scale, soft cap, store logits, per-batch-row argmax key.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace muse {
namespace {

constexpr int kTileRows = 128;               // M of one MMA and of one warpgroup's tile
constexpr int kPairRows = 2 * kTileRows;     // rows per weight box
constexpr int kWStageBytes = kPairRows * kBlockBytes;   // 45,056
constexpr int kXStages = 2;
constexpr int kThreads = 352;                // 2 warpgroups + weight producer + MMA + package producer
constexpr int kProducerWarp = 8;             // weight boxes
constexpr int kMmaWarp = 9;
constexpr int kPkgWarp = 10;                 // activation packages
constexpr uint32_t kTmemCols = 512;

template <int NM>
struct TcCfg {
  static_assert(NM == 16 || NM == 32, "MMA N");
  static constexpr int kXRows = 2 * NM;                           // x_hi rows, then x_lo rows
  static constexpr int kXBytes = kXRows * kBlockWeights * 2;      // f16 [2NM][256] operand tile
  static constexpr int kMinBytes = NM * 16 * 2;                   // [NM][16] f16
  static constexpr int kPkgBytes = kXBytes + kMinBytes;           // per block
  static constexpr int kWStages = NM == 16 ? 4 : 3;               // as many weight stages as fit
  static constexpr int kSmemBytes = kWStages * kWStageBytes + kXStages * kPkgBytes + 1024;
  static constexpr uint32_t kIdesc = tc::idesc_f16_f32(kTileRows, 2 * NM);
  static constexpr uint32_t kIdescMin = tc::idesc_f16_f32(kTileRows, NM);
  // tensor-memory columns of warpgroup w: A [128], A_min [8], D [2NM], Dmin [NM]
  __host__ __device__ static constexpr uint32_t col_a(int w) { return 256u * w; }
  __host__ __device__ static constexpr uint32_t col_amin(int w) { return 256u * w + 128u; }
  __host__ __device__ static constexpr uint32_t col_d(int w) { return 256u * w + 160u; }
  __host__ __device__ static constexpr uint32_t col_dmin(int w) { return 256u * w + 224u; }
};

// Byte offset of element (n, k) in a K-major operand tile of `rows` rows
// made of 8-row x 16-byte core matrices: core (n/8, k/8) at
// ((k/8) * (rows/8) + n/8) * 128, then 16 bytes per row, 2 bytes per element.
__host__ __device__ constexpr uint32_t kmajor_offset(int rows, int n, int k) {
  return static_cast<uint32_t>(((k >> 3) * (rows >> 3) + (n >> 3)) * 128 + (n & 7) * 16 + (k & 7) * 2);
}

// ------------------------------------------------------------------ prep kernel
template <int NM>
__global__ void __launch_bounds__(256)
    prep_x_kernel(const float *__restrict__ hidden, const float *__restrict__ gamma, float eps, int batch, int k,
                  uint8_t *__restrict__ pkgs) {
  using C = TcCfg<NM>;
  __shared__ float s_r[32];
  __shared__ float s_part[8];
  const int kb = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // per-row RMS factors (every CTA recomputes them from the L2-resident rows)
  for (int b = 0; b < batch; ++b) {
    float r = 1.0f;
    if (gamma) {
      float ss = 0.0f;
      const float *h = hidden + static_cast<size_t>(b) * k;
      for (int j = tid * 4; j < k; j += 256 * 4) {
        const float4 v = *reinterpret_cast<const float4 *>(h + j);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_part[warp] = ss;
      __syncthreads();
      float tot = 0.0f;
      for (int i = 0; i < 8; ++i) tot += s_part[i];
      r = 1.0f / sqrtf(tot / static_cast<float>(k) + eps);
      __syncthreads();
    }
    if (tid == 0) s_r[b] = r;
  }
  __syncthreads();
  uint8_t *pkg = pkgs + static_cast<size_t>(kb) * C::kPkgBytes;
  const int j = tid;                        // column inside the block; warp = sub-block
  const int col = kb * kBlockWeights + j;
  const float g = gamma ? gamma[col] : 1.0f;
  for (int b = 0; b < NM; ++b) {
    float x = 0.0f;
    if (b < batch) x = gamma ? hidden[static_cast<size_t>(b) * k + col] * s_r[b] * g
                             : hidden[static_cast<size_t>(b) * k + col];
    const __half hi = __float2half_rn(x);
    const __half lo = __float2half_rn(x - __half2float(hi));
    *reinterpret_cast<__half *>(pkg + kmajor_offset(C::kXRows, b, j)) = hi;
    *reinterpret_cast<__half *>(pkg + kmajor_offset(C::kXRows, NM + b, j)) = lo;
    float s = x;                            // sum over the 32 columns of sub-block `warp`
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      const __half shi = __float2half_rn(s);
      const __half slo = __float2half_rn(s - __half2float(shi));
      *reinterpret_cast<__half *>(pkg + C::kXBytes + kmajor_offset(NM, b, warp)) = shi;
      *reinterpret_cast<__half *>(pkg + C::kXBytes + kmajor_offset(NM, b, 8 + warp)) = slo;
    }
  }
}

// ------------------------------------------------------------------ main kernel
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(ptx::smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(ptx::smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint32_t rotl32(uint32_t v, uint32_t s) { return __funnelshift_l(v, v, s); }

// f16 pair (1024 + a, 1024 + b) from a = byte I and b = byte I+1 of q4 (both
// below 64): each byte goes under the f16 exponent byte 0x64.
template <int I>
__device__ __forceinline__ uint32_t magic_pair(uint32_t q4) {
  return __byte_perm(q4, 0x64u, 0x4040u | I | ((I + 1) << 8));
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b),
                      *reinterpret_cast<__half2 *>(&c));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t h2_bits(float v) {
  __half2 h = __float2half2_rn(v);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Header of one row's Q5_K block: d, dmin, the eight 6-bit scales and mins as
// bytes (sc[0..3], sc[4..7], m[0..3], m[4..7]) and the 32 high-bit bytes.
struct RowHdr {
  float d, dmin;
  uint32_t sc03, sc47, m03, m47;
  uint32_t H[8];
};

__device__ __forceinline__ void load_row_hdr(const uint8_t *blk, RowHdr &o) {
  const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
  const uint4 h0 = *reinterpret_cast<const uint4 *>(blk + kOffQh);
  const uint4 h1 = *reinterpret_cast<const uint4 *>(blk + kOffQh + 16);
  o.H[0] = h0.x; o.H[1] = h0.y; o.H[2] = h0.z; o.H[3] = h0.w;
  o.H[4] = h1.x; o.H[5] = h1.y; o.H[6] = h1.z; o.H[7] = h1.w;
  const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&hdr.x));
  o.d = dd.x;
  o.dmin = dd.y;
  const uint32_t w0 = hdr.y, w1 = hdr.z, w2 = hdr.w;
  o.sc03 = w0 & 0x3F3F3F3Fu;
  o.m03 = w1 & 0x3F3F3F3Fu;
  o.sc47 = (w2 & 0x0F0F0F0Fu) | ((w0 >> 2) & 0x30303030u);
  o.m47 = ((w2 >> 4) & 0x0F0F0F0Fu) | ((w1 >> 2) & 0x30303030u);
}

// A_min columns: k = 0..7 and 8..15 both hold m_0..m_7 (exact small integers).
__device__ __forceinline__ void amin_cols(const RowHdr &h, uint32_t (&o)[8]) {
  const uint32_t neg1024 = h2_bits(-1024.0f), one = h2_bits(1.0f);
  o[0] = o[4] = hfma2_u32(magic_pair<0>(h.m03), one, neg1024);
  o[1] = o[5] = hfma2_u32(magic_pair<2>(h.m03), one, neg1024);
  o[2] = o[6] = hfma2_u32(magic_pair<0>(h.m47), one, neg1024);
  o[3] = o[7] = hfma2_u32(magic_pair<2>(h.m47), one, neg1024);
}

// Columns 32c..32c+31 of A for one row: sub-blocks 2c (low nibbles, built as q)
// and 2c+1 (high nibbles, built as 2q), as f16 pairs sc_s*q in natural K order.
template <int C>
__device__ __forceinline__ void a_chunk(const uint8_t *blk, const RowHdr &h, uint32_t (&o)[32]) {
  const uint32_t scw = C < 2 ? h.sc03 : h.sc47;
  constexpr int sh = 16 * (C & 1);
  const float sc_lo = static_cast<float>((scw >> sh) & 0xFFu);
  const float sc_hi = static_cast<float>((scw >> (sh + 8)) & 0xFFu);
  const uint32_t mul_lo = h2_bits(sc_lo), add_lo = h2_bits(-1024.0f * sc_lo);
  const uint32_t mul_hi = h2_bits(0.5f * sc_hi), add_hi = h2_bits(-512.0f * sc_hi);
  const uint4 a0 = *reinterpret_cast<const uint4 *>(blk + kOffQs + 32 * C);
  const uint4 a1 = *reinterpret_cast<const uint4 *>(blk + kOffQs + 32 * C + 16);
  const uint32_t A[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  constexpr uint32_t rot = static_cast<uint32_t>(4 - 2 * C) & 31u;   // bit 2C -> 4, bit 2C+1 -> 5
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t t = rotl32(h.H[i], rot);
    const uint32_t qlo = (A[i] & 0x0F0F0F0Fu) | (t & 0x10101010u);        // q, positions 4i..4i+3
    const uint32_t qhi = ((A[i] >> 3) & 0x1E1E1E1Eu) | (t & 0x20202020u);  // 2q
    o[2 * i] = hfma2_u32(magic_pair<0>(qlo), mul_lo, add_lo);
    o[2 * i + 1] = hfma2_u32(magic_pair<2>(qlo), mul_lo, add_lo);
    o[16 + 2 * i] = hfma2_u32(magic_pair<0>(qhi), mul_hi, add_hi);
    o[16 + 2 * i + 1] = hfma2_u32(magic_pair<2>(qhi), mul_hi, add_hi);
  }
}

template <int NM>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const uint8_t *__restrict__ pkgs, int nb,
                   int64_t n_rows, int batch, float scale, float cap, float *__restrict__ logits,
                   unsigned long long *keys, unsigned int *ticket, int32_t *argmax, uint32_t *status) {
  using C = TcCfg<NM>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *wst = smem;                                            // [C::kWStages][256 rows][176 B]
  uint8_t *xst = smem + C::kWStages * kWStageBytes;                  // [kXStages][package]
  uint64_t *bars = reinterpret_cast<uint64_t *>(xst + kXStages * C::kPkgBytes);
  uint64_t *wfull = bars, *wempty = bars + C::kWStages;
  uint64_t *xfull = wempty + C::kWStages, *xempty = xfull + kXStages;
  uint64_t *aready = xempty + kXStages;                           // [2]: A written, D read
  uint64_t *adone = aready + 2;                                   // [2]: MMAs of the block complete
  uint64_t *mma_idle = adone + 2;                                 // all MMAs of this CTA complete
  unsigned long long *s_keys = reinterpret_cast<unsigned long long *>(mma_idle + 1);   // [32]
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(s_keys + 32);
  volatile uint32_t *s_abort = s_tmem + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n_tiles = (n_rows + kTileRows - 1) / kTileRows;
  const int64_t n_pairs = (n_tiles + 1) / 2;
  const int64_t my_pairs = blockIdx.x < n_pairs ? (n_pairs - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t total = my_pairs * nb;                            // (pair, block) steps of this CTA

  if (tid == 0) {
    for (int s = 0; s < C::kWStages; ++s) {
      ptx::mbar_init(&wfull[s], 1);
      ptx::mbar_init(&wempty[s], 8);                              // the eight unpack warps
    }
    for (int s = 0; s < kXStages; ++s) {
      ptx::mbar_init(&xfull[s], 1);
      ptx::mbar_init(&xempty[s], 1);                              // one commit after both tiles' MMAs
    }
    for (int w = 0; w < 2; ++w) {
      ptx::mbar_init(&aready[w], 4);
      ptx::mbar_init(&adone[w], 1);
    }
    ptx::mbar_init(mma_idle, 1);
    for (int b = 0; b < 32; ++b) s_keys[b] = 0ull;
    *s_abort = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::alloc(s_tmem, kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *s_tmem;

  auto fail = [&]() {
    atomicOr(status, kStatusWaitTimeout);
    *s_abort = 1u;
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      const uint64_t pol_w = ptx::policy_evict_first();
      int64_t issued = 0;
      for (int64_t g = 0; g < total && !*s_abort; ++g) {
        const int64_t pair = blockIdx.x + (g / nb) * gridDim.x;
        const int kb = static_cast<int>(g % nb);
        const int ws = static_cast<int>(g % C::kWStages);
        if (g >= C::kWStages &&
            !ptx::mbar_wait(&wempty[ws], static_cast<uint32_t>((g / C::kWStages - 1) & 1))) { fail(); break; }
        ptx::mbar_arrive_expect_tx(&wfull[ws], kWStageBytes);
        tma_load_2d(wst + ws * kWStageBytes, &wmap, kb * (kBlockBytes / 4), static_cast<int>(pair * kPairRows),
                    &wfull[ws], pol_w);
        issued = g + 1;
      }
      // never leave copies in flight
      for (int64_t g = issued > C::kWStages ? issued - C::kWStages : 0; g < issued; ++g)
        ptx::mbar_wait(&wfull[g % C::kWStages], static_cast<uint32_t>((g / C::kWStages) & 1));
    }
  } else if (warp == kPkgWarp) {
    // ------------------------------------------------------------ activation-package producer
    if (lane == 0) {
      int64_t issued = 0;
      for (int64_t g = 0; g < total && !*s_abort; ++g) {
        const int kb = static_cast<int>(g % nb);
        const int xs = static_cast<int>(g % kXStages);
        if (g >= kXStages &&
            !ptx::mbar_wait(&xempty[xs], static_cast<uint32_t>((g / kXStages - 1) & 1))) { fail(); break; }
        ptx::mbar_arrive_expect_tx(&xfull[xs], C::kPkgBytes);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         ptx::smem_u32(xst + xs * C::kPkgBytes)),
                     "l"(pkgs + static_cast<size_t>(kb) * C::kPkgBytes), "r"(C::kPkgBytes),
                     "r"(ptx::smem_u32(&xfull[xs]))
                     : "memory");
        issued = g + 1;
      }
      for (int64_t g = issued > kXStages ? issued - kXStages : 0; g < issued; ++g)
        ptx::mbar_wait(&xfull[g % kXStages], static_cast<uint32_t>((g / kXStages) & 1));
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and operands stay warp-uniform); one
    // elected lane issues the MMAs and commits.
    bool ok = true;
    for (int64_t g = 0; g < total && ok; ++g) {
      if (__any_sync(0xffffffffu, *s_abort != 0u)) break;
      const int xs = static_cast<int>(g % kXStages);
      const uint32_t par = static_cast<uint32_t>(g & 1);
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&xfull[xs], static_cast<uint32_t>((g / kXStages) & 1)))) {
        ok = false;
        break;
      }
      const uint32_t xbase = ptx::smem_u32(xst + xs * C::kPkgBytes);
      const uint64_t bdesc0 = tc::smem_desc_kmajor(xbase, C::kXRows * 16, 128);
      const uint64_t mdesc = tc::smem_desc_kmajor(xbase + C::kXBytes, NM * 16, 128);
      for (int w = 0; w < 2; ++w) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&aready[w], par))) {
          ok = false;
          break;
        }
        tc::fence_after();
        if (tc::elect_one()) {
          const uint32_t d = tbase + C::col_d(w);
          const uint32_t a = tbase + C::col_a(w);
#pragma unroll
          for (int ks = 0; ks < 16; ++ks)   // K-step ks: 16 columns of x = 2 core matrices along K
            tc::mma_f16_tmemA(d, a + 8 * ks, bdesc0 + ((ks * 2 * (C::kXRows / 8) * 128) >> 4), C::kIdesc, ks > 0);
          tc::mma_f16_tmemA(tbase + C::col_dmin(w), tbase + C::col_amin(w), mdesc, C::kIdescMin, false);
          tc::commit(&adone[w]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (tc::elect_one()) tc::commit(&xempty[xs]);
      __syncwarp();
    }
    if (!ok && lane == 0) fail();
    // tensor memory is freed below only after every MMA issued here completed
    if (tc::elect_one()) tc::commit(mma_idle);
    __syncwarp();
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(mma_idle, 0)) && lane == 0) fail();
  } else {
    // ------------------------------------------------------------ unpack + epilogue (warpgroup w)
    const int w = warp >> 2;                    // 0 or 1: which tile of the pair
    const int r = tid & 127;                    // row inside the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    float acc[32];
#pragma unroll
    for (int b = 0; b < 32; ++b) acc[b] = 0.0f;
    float d_prev = 0.0f, dmin_prev = 0.0f;
    int64_t row_prev = -1;
    auto finish_tile = [&](int64_t row) {      // scale, cap, store, argmax keys; reset accumulators
#pragma unroll
      for (int b = 0; b < 32; ++b) {
        if (b < batch) {
          const float v = scale_softcap(acc[b], scale, cap);
          unsigned long long key = 0ull;
          if (row < n_rows) {
            logits[static_cast<size_t>(b) * n_rows + row] = v;
            key = argmax_key(v, static_cast<uint32_t>(row));
          }
          for (int o = 16; o > 0; o >>= 1) key = umax64(key, __shfl_xor_sync(0xffffffffu, key, o));
          if (lane == 0 && key != 0ull) atomicMax(&s_keys[b], key);
        }
        acc[b] = 0.0f;
      }
    };
    // read back the previous block's D and Dmin (its MMAs are complete) and accumulate
    auto drain = [&]() {
      tc::fence_after();
#pragma unroll
      for (int c0 = 0; c0 < NM; c0 += 16) {
        uint32_t dh[16], dl[16], mv[16];
        tc::ld_32x32b_x16(tbase + lane_base + C::col_d(w) + c0, dh);        // x_hi columns
        tc::ld_32x32b_x16(tbase + lane_base + C::col_d(w) + NM + c0, dl);   // x_lo columns
        tc::ld_32x32b_x16(tbase + lane_base + C::col_dmin(w) + c0, mv);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float dot = __uint_as_float(dh[j]) + __uint_as_float(dl[j]);
          acc[c0 + j] = fmaf(d_prev, dot, fmaf(-dmin_prev, __uint_as_float(mv[j]), acc[c0 + j]));
        }
      }
    };
    bool ok_all = true;
    for (int64_t g = 0; g < total; ++g) {
      if (__any_sync(0xffffffffu, *s_abort != 0u)) { ok_all = false; break; }
      const int64_t pair = blockIdx.x + (g / nb) * gridDim.x;
      const int kb = static_cast<int>(g % nb);
      const int ws = static_cast<int>(g % C::kWStages);
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&wfull[ws], static_cast<uint32_t>((g / C::kWStages) & 1)))) {
        if (lane == 0) fail();
        ok_all = false;
        break;
      }
      const uint8_t *blk = wst + ws * kWStageBytes + (w * kTileRows + r) * kBlockBytes;
      RowHdr hd;
      load_row_hdr(blk, hd);
      uint32_t c0[32], c1[32];
      a_chunk<0>(blk, hd, c0);                  // overlaps the previous block's MMAs
      a_chunk<1>(blk, hd, c1);
      if (g >= 1) {                             // the previous block's MMAs: A consumed, D written
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&adone[w], static_cast<uint32_t>((g - 1) & 1)))) {
          if (lane == 0) fail();
          ok_all = false;
          break;
        }
        drain();
        if (kb == 0) finish_tile(row_prev);     // the previous block closed the previous tile
      }
      const uint32_t ta = tbase + lane_base + C::col_a(w);
      tc::st_32x32b_x32(ta, c0);
      tc::st_32x32b_x32(ta + 32, c1);
      a_chunk<2>(blk, hd, c0);
      tc::st_32x32b_x32(ta + 64, c0);
      a_chunk<3>(blk, hd, c1);
      tc::st_32x32b_x32(ta + 96, c1);
      uint32_t am[8];
      amin_cols(hd, am);
      tc::st_32x32b_x8(tbase + lane_base + C::col_amin(w), am);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&wempty[ws]);   // weight stage fully read
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&aready[w]);
      d_prev = hd.d;
      dmin_prev = hd.dmin;
      row_prev = (pair * 2 + w) * kTileRows + r;
    }
    if (ok_all && total > 0) {
      if (__all_sync(0xffffffffu, ptx::mbar_wait(&adone[w], static_cast<uint32_t>((total - 1) & 1)))) {
        drain();
        finish_tile(row_prev);
      } else if (lane == 0) {
        fail();
      }
    }
    tc::fence_before();
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after();
    tc::dealloc(tbase, kTmemCols);
  }
  if (argmax) {
    if (tid < batch && s_keys[tid] != 0ull) atomicMax(keys + tid, s_keys[tid]);
    argmax_finish(keys, ticket, argmax, batch);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

template <int NM>
cudaError_t launch_tc_nm(const LaunchArgs &a, const CUtensorMap &map) {
  using C = TcCfg<NM>;
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    e = cudaFuncSetAttribute(gemm_tc_kernel<NM>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured |= bit;
  }
  const int nb = a.k / kBlockWeights;
  prep_x_kernel<NM><<<nb, 256, 0, a.stream>>>(a.hidden, a.gamma, a.eps, a.batch, a.k, a.ws.xpkg);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n_tiles = (a.n_rows + kTileRows - 1) / kTileRows;
  const int64_t n_pairs = (n_tiles + 1) / 2;
  const int64_t grid = n_pairs < a.num_sms ? n_pairs : a.num_sms;
  gemm_tc_kernel<NM><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, a.stream>>>(
      map, a.ws.xpkg, nb, a.n_rows, a.batch, a.scale, a.cap, a.logits, a.ws.keys, a.ws.ticket, a.argmax,
      a.ws.status);
  return cudaGetLastError();
}

}  // namespace

size_t tc_workspace_bytes(int k) { return static_cast<size_t>(k / kBlockWeights) * TcCfg<32>::kPkgBytes; }

bool tc_supported(int batch) { return batch >= 2 && batch <= 32; }

cudaError_t tc_encode_weights(CUtensorMap *map, const void *weights, int64_t n_rows, int k) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(k / kBlockWeights) * (kBlockBytes / 4),
                              static_cast<cuuint64_t>(n_rows)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(k / kBlockWeights) * kBlockBytes};
  const cuuint32_t box[2] = {kBlockBytes / 4, kPairRows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(weights), gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_tc(const LaunchArgs &a, const CUtensorMap &map) {
  return a.batch <= 16 ? launch_tc_nm<16>(a, map) : launch_tc_nm<32>(a, map);
}

}  // namespace muse
