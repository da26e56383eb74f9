// Batched output stage on the 5th-generation tensor cores (tcgen05), for
// batches of 2..32 rows: final RMSNorm, Q5_K (or Q4_K) LM-head contraction,
// scale + soft cap, argmax ("Chapter 20 — Final norm, LM head, and the soft
// cap", §20.1, §20.3, §20.4, §20.7).  Two launches per forward:
//
// 1. prep_x_kernel: one CTA per (Q5_K block column kb, package row b).
//    Normalises hidden row b and writes its part of the block's "activation
//    package", already in the tensor-core operand layout (K-major, 8-row x
//    16-byte core matrices):
//      x     [2*NM rows][256]  rows 0..NM-1: f16(x); rows NM..2NM-1: f16(x - f16(x))
//                              (the two rows of a batch row sum to x to ~2^-22)
//      x_min [max(NM,16) rows][16]  k < 8: f16 hi of S_s = sum of x over
//                              sub-block s, k >= 8: its f16 remainder
//    Rows >= batch are zero.
//
// 2. gemm_tc_kernel: a persistent CTA per SM works on 128-row tiles.  It is a
//    programmatic dependent launch: everything but the package loads (set-up,
//    the weight stream, the first unpack steps) overlaps the prep kernel.
//    With up to 16 batch slots the (tile, block) steps are dealt out as equal
//    contiguous ranges (in pairs of steps), so every CTA streams the same
//    number of blocks; a tile cut by a range boundary is shared by two
//    neighbouring CTAs, which both leave their partial sums in global memory
//    and count in; the second to arrive adds the two (in a fixed order) and
//    finishes the rows.  With 32 slots the hand-off of the 32 partial columns
//    costs more than the balance gains (measured), and tiles go round-robin.
//    A narrow matrix (fewer 128-row tiles than SMs) runs a separate instance
//    (kNarrow) that deals the steps over up to one CTA per SM at any batch:
//    a tile is then shared by all the CTAs whose ranges meet it, each leaves
//    its sums in its slot and counts in on the tile's counter, and the last
//    to arrive adds the slots in CTA order and finishes the rows.
//    * weight producer warp: per block kb, one 2-D TMA box of 128 rows x 176
//      bytes (144 for Q4_K) into a ring of weight stages.  Package producer
//      warp: the kb activation package (1-D bulk copy) into a ring of package
//      stages.
//    * four unpack warpgroups in two pairs; pair p takes the blocks whose step
//      index has parity p, so the two pairs work on consecutive blocks at once
//      with their own tensor-memory buffers.  In a pair, thread r of either
//      warpgroup owns row r: one warpgroup sub-blocks 0..3 and batch columns
//      0..NM/2-1, the other sub-blocks 4..7 and the remaining columns.  A thread
//      turns its half of the row's block into A[r][e] = sc_s * q_e as f16 (exact:
//      at most 31*63) (the first warpgroup also A_min[r][k] = m_(k mod 8)),
//      stores it into tensor memory (tcgen05.st), and after that block's MMAs
//      reads back its columns of D[r][b] and Dmin[r][b] (tcgen05.ld) to
//      accumulate
//          raw[r][b] += d * D[r][b] - dmin * Dmin[r][b]
//      which is sum_e (d*sc_s*q_e - dmin*m_s) * x[b][e] for the block.  At the
//      end of a tile the two pairs add their sums through shared memory and the
//      first pair applies scale and soft cap, stores the logits and keeps the
//      per-batch-row argmax keys.
//    * MMA warp (the whole warp runs the loop with warp-uniform operands, one
//      elected lane issues): per block, 16 K-steps of f16 MMAs with f32
//      accumulation into D (M = 128, N = 2*NM: the x_hi and x_lo rows side by
//      side) and one MMA A_min x x_min into Dmin; tcgen05.commit hands the
//      buffer back.  With 16 and 32 slots (N = 32, 64) it issues the K-steps
//      of both warpgroups' first 64-column chunks as soon as those are in
//      tensor memory, and the rest once the whole A is: the longer MMAs then
//      overlap the second chunks' unpack instead of sitting in the pair's
//      chain.
//    * The weight tensor map promotes L2 fetches to 64 bytes: a 176-byte box
//      row shares its first and last 256-byte line with the neighbouring
//      boxes, whose bytes were often evicted (evict-first) before the
//      neighbour came for them.
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace muse {
namespace {

constexpr int kTileRows = 128;                          // M of one MMA
constexpr int kUnpackWarps = 16;                        // 2 pairs x 2 warpgroups
constexpr int kThreads = 32 * (kUnpackWarps + 3);       // + weight producer, MMA issuer, package producer
constexpr int kProducerWarp = kUnpackWarps;
constexpr int kMmaWarp = kUnpackWarps + 1;
constexpr int kPkgWarp = kUnpackWarps + 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemLimit = 227 * 1024 - 1024;           // opt-in limit minus static shared memory

// The min MMA needs N >= 16; for NM = 8 its operand tile has 16 rows, 8..15 zero.
template <int NM>
__host__ __device__ constexpr int min_rows() { return NM < 16 ? 16 : NM; }

// NM batch slots; kQ4: Q4_K weight blocks (144 bytes) instead of Q5_K (176).
// The activation package does not depend on the weight format.
template <int NM, bool kQ4 = false>
struct TcCfg {
  static_assert(NM == 8 || NM == 16 || NM == 32, "MMA N / 2");
  static constexpr int kBB = kQ4 ? kBlockBytesQ4 : kBlockBytes;   // bytes per block
  static constexpr int kWStageBytes = kTileRows * kBB;            // one block column of a tile
  static constexpr int kXRows = 2 * NM;                           // x_hi rows, then x_lo rows
  static constexpr int kXBytes = kXRows * kBlockWeights * 2;      // f16 [2NM][256] operand tile
  static constexpr int kMinBytes = min_rows<NM>() * 16 * 2;       // f16 [rows][16]
  static constexpr int kPkgBytes = kXBytes + kMinBytes;           // per block
  // Package ring: a stage is refilled only after the MMAs that read it are
  // complete, so the ring must cover the copy latency from L2 with a few steps.
  static constexpr int kXStages = NM == 32 ? 3 : 4;
  static constexpr int kXchgBytes = 2 * kTileRows * (NM / 2) * 4; // pair-1 sums handed to pair 0
  static constexpr int kFixed = kXStages * kPkgBytes + kXchgBytes + 1024;
  static constexpr int kWFit = (kSmemLimit - kFixed) / kWStageBytes;
  static constexpr int kWStages = (kWFit > 8 ? 8 : kWFit) & ~1;   // even: a stage always serves one pair
  static_assert(kWStages >= 4, "weight ring");
  static constexpr int kSmemBytes = kWStages * kWStageBytes + kFixed;
  static constexpr uint32_t kIdesc = tc::idesc_f16_f32(kTileRows, 2 * NM);
  static constexpr uint32_t kIdescMin = tc::idesc_f16_f32(kTileRows, min_rows<NM>());
  // tensor-memory columns of buffer j: A [128], A_min [8], D [2NM], Dmin [max(NM,16)]
  __host__ __device__ static constexpr uint32_t col_a(int j) { return 128u * j; }
  __host__ __device__ static constexpr uint32_t col_amin(int j) { return 256u + 8u * j; }
  __host__ __device__ static constexpr uint32_t col_d(int j) { return 288u + 96u * j; }
  __host__ __device__ static constexpr uint32_t col_dmin(int j) { return 288u + 96u * j + 64u; }
};

// Byte offset of element (n, k) in a K-major operand tile of `rows` rows
// made of 8-row x 16-byte core matrices: core (n/8, k/8) at
// ((k/8) * (rows/8) + n/8) * 128, then 16 bytes per row, 2 bytes per element.
__host__ __device__ constexpr uint32_t kmajor_offset(int rows, int n, int k) {
  return static_cast<uint32_t>(((k >> 3) * (rows >> 3) + (n >> 3)) * 128 + (n & 7) * 16 + (k & 7) * 2);
}

// ------------------------------------------------------------------ prep kernel
// Grid (nb, max(NM,16)), 128 threads; thread t covers columns t and t+128 of the
// block, so warp w holds sub-blocks w and 4+w.
constexpr int kPrepThreads = 128;

template <int NM>
__global__ void __launch_bounds__(kPrepThreads)
    prep_x_kernel(const float *__restrict__ hidden, const float *__restrict__ gamma, float eps, int batch, int k,
                  uint8_t *__restrict__ pkgs) {
  using C = TcCfg<NM>;
  __shared__ float s_part[kPrepThreads / 32];
  // A programmatic dependent of the previous forward's GEMM (which triggers
  // near its end): nothing is read or written before that grid has completed,
  // so this grid's launch overlaps its tail.  Then let the dependent GEMM
  // start its set-up and weight stream; it reads the packages only after this
  // grid has completed, and the writes it shares with the previous GEMM
  // (logits, argmax keys, shared-tile counters) follow from those packages.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int kb = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float x[2] = {0.0f, 0.0f};
  if (b < batch) {
    const float *h = hidden + static_cast<size_t>(b) * k;
    const int c0 = kb * kBlockWeights + tid;
    x[0] = h[c0];
    x[1] = h[c0 + 128];
    if (gamma) {
      float ss = 0.0f;
      for (int j = tid * 4; j < k; j += kPrepThreads * 4) {
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
      for (int w = 0; w < kPrepThreads / 32; ++w) tot += s_part[w];
      const float rr = 1.0f / sqrtf(tot / static_cast<float>(k) + eps);
      x[0] *= rr * gamma[c0];
      x[1] *= rr * gamma[c0 + 128];
    }
  }
  uint8_t *pkg = pkgs + static_cast<size_t>(kb) * C::kPkgBytes;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int j = tid + 128 * hh;           // column inside the block
    if (b < NM) {
      const __half hi = __float2half_rn(x[hh]);
      const __half lo = __float2half_rn(x[hh] - __half2float(hi));
      *reinterpret_cast<__half *>(pkg + kmajor_offset(C::kXRows, b, j)) = hi;
      *reinterpret_cast<__half *>(pkg + kmajor_offset(C::kXRows, NM + b, j)) = lo;
    }
    float sum = x[hh];                      // sum over the 32 columns of sub-block 4hh + warp
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      const int sb = 4 * hh + warp;
      const __half shi = __float2half_rn(sum);
      const __half slo = __float2half_rn(sum - __half2float(shi));
      *reinterpret_cast<__half *>(pkg + C::kXBytes + kmajor_offset(min_rows<NM>(), b, sb)) = shi;
      *reinterpret_cast<__half *>(pkg + C::kXBytes + kmajor_offset(min_rows<NM>(), b, 8 + sb)) = slo;
    }
  }
}

// ------------------------------------------------------------------ unpack helpers
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
};

__device__ __forceinline__ void load_row_hdr(const uint8_t *blk, RowHdr &o) {
  const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
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

// HFMA2 operands of one 32-column chunk: its low nibbles (sub-block 2c) are
// built as (1024 + q) * sc - 1024 sc, its high nibbles (sub-block 2c+1) as
// (1024 + 2q) * sc/2 - 512 sc; both exact.  scw holds the chunk's two 6-bit
// scales as bytes I and I+1.  A single HFMA2 turns the magic pair
// (1024 + sc_a, 1024 + sc_b) into (sc_a, sc_b / 2), so the constants need
// three byte permutes and two f16 multiplies, and no conversion.
struct ChunkK {
  uint32_t mul_lo, add_lo, mul_hi, add_hi;
};

constexpr uint32_t kH2OneHalf = 0x38003C00u;      // f16 pair (1, 0.5), low half first
constexpr uint32_t kH2Neg1024 = 0xE400E400u;      // (-1024, -1024)
constexpr uint32_t kH2Neg1024_512 = 0xE000E400u;  // (-1024, -512)

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

template <int I>
__device__ __forceinline__ ChunkK chunk_consts(uint32_t scw) {
  const uint32_t v = hfma2_u32(magic_pair<I>(scw), kH2OneHalf, kH2Neg1024_512);   // (sc_a, sc_b / 2)
  ChunkK k;
  k.mul_lo = __byte_perm(v, 0u, 0x1010u);
  k.mul_hi = __byte_perm(v, 0u, 0x3232u);
  k.add_lo = hmul2_u32(k.mul_lo, kH2Neg1024);
  k.add_hi = hmul2_u32(k.mul_hi, kH2Neg1024);
  return k;
}

// Columns 32C..32C+31 of A for one row: sub-blocks 2C (low nibbles, built as q)
// and 2C+1 (high nibbles, built as 2q), as f16 pairs sc_s*q in natural K order;
// stored to tensor memory at column `ta` in two 16-column halves.  Q5_K adds
// each quant's fifth bit from the 32 high-bit bytes H (bit 2C of byte l for the
// low nibble, 2C+1 for the high one); Q4_K has none.
template <bool kQ4, int C>
__device__ __forceinline__ void a_chunk_st(const uint8_t *blk, const ChunkK &k, uint32_t ta) {
  constexpr int kQs = kQ4 ? kOffQsQ4 : kOffQs;
  constexpr uint32_t kRot = static_cast<uint32_t>(4 - 2 * C) & 31u;   // bit 2C -> 4, bit 2C+1 -> 5
  const uint4 a0 = *reinterpret_cast<const uint4 *>(blk + kQs + 32 * C);
  const uint4 a1 = *reinterpret_cast<const uint4 *>(blk + kQs + 32 * C + 16);
  const uint32_t A[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  uint32_t Hr[8] = {};
  if constexpr (!kQ4) {
    const uint4 h0 = *reinterpret_cast<const uint4 *>(blk + kOffQh);
    const uint4 h1 = *reinterpret_cast<const uint4 *>(blk + kOffQh + 16);
    const uint32_t H[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) Hr[i] = kRot == 0 ? H[i] : rotl32(H[i], kRot);
  }
  uint32_t o[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t q = A[i] & 0x0F0F0F0Fu;                                          // q, positions 4i..4i+3
    if constexpr (!kQ4) q |= Hr[i] & 0x10101010u;
    o[2 * i] = hfma2_u32(magic_pair<0>(q), k.mul_lo, k.add_lo);
    o[2 * i + 1] = hfma2_u32(magic_pair<2>(q), k.mul_lo, k.add_lo);
  }
  tc::st_32x32b_x16(ta, o);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t q = (A[i] >> 3) & 0x1E1E1E1Eu;                                   // 2q
    if constexpr (!kQ4) q |= Hr[i] & 0x20202020u;
    o[2 * i] = hfma2_u32(magic_pair<0>(q), k.mul_hi, k.add_hi);
    o[2 * i + 1] = hfma2_u32(magic_pair<2>(q), k.mul_hi, k.add_hi);
  }
  tc::st_32x32b_x16(ta + 16, o);
}

__device__ __forceinline__ void ld_x4(uint32_t ta, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(ta)
               : "memory");
}

// ------------------------------------------------------------------ main kernel
template <int NM, bool kQ4, bool kNarrow>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const uint8_t *__restrict__ pkgs, int nb,
                   int64_t n_rows, int batch, float scale, float cap, float *__restrict__ logits,
                   unsigned long long *keys, unsigned int *ticket, int32_t *argmax, uint32_t *status,
                   float *split_part, unsigned int *split_cnt, int argmax_precap) {
  using C = TcCfg<NM, kQ4>;
  constexpr int HB = NM / 2;                                      // batch columns per warpgroup
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *wst = smem;                                            // [kWStages][128 rows][block bytes]
  uint8_t *xst = smem + C::kWStages * C::kWStageBytes;            // [C::kXStages][package]
  float *xchg = reinterpret_cast<float *>(xst + C::kXStages * C::kPkgBytes);   // [2 halves][128][HB]
  uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(xchg) + C::kXchgBytes);
  uint64_t *wfull = bars, *wempty = bars + C::kWStages;
  uint64_t *xfull = wempty + C::kWStages, *xempty = xfull + C::kXStages;
  uint64_t *aready = xempty + C::kXStages;                           // [2]: A written, D read
  uint64_t *adone = aready + 2;                                   // [2]: MMAs of the buffer complete
  uint64_t *mma_idle = adone + 2;                                 // all MMAs of this CTA complete
  uint64_t *xch_full = mma_idle + 1, *xch_empty = mma_idle + 2;   // tile-end hand-over, pair 1 -> pair 0
  unsigned long long *s_keys = reinterpret_cast<unsigned long long *>(mma_idle + 3);   // [32]
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(s_keys + 32);
  volatile uint32_t *s_abort = s_tmem + 1;
  // [2]: the first chunk of both warpgroups of pair j is in tensor memory (16
  // and 32 slots: the MMA warp starts on those K-steps while the second
  // chunks are built, which takes the longer MMAs of wide batches partly off
  // the pair's chain)
  uint64_t *ahalf = reinterpret_cast<uint64_t *>(s_tmem + 2);
  constexpr bool kEarlyHalf = NM >= 16;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n_tiles = (n_rows + kTileRows - 1) / kTileRows;
  // Balanced: this CTA's steps [s_begin, s_end) of the tile-major (tile,
  // block) sequence, equal shares in pairs of steps (nb is even, so both pairs
  // keep their parity across tiles).  With at most n_tiles CTAs a share is at
  // least nb steps, so a tile is cut at most once and shared by at most two
  // CTAs.  Round-robin: tiles blockIdx.x + j * gridDim.x, none shared.
  // Narrow instance: gridDim.x <= pairs, so no share is empty and the CTAs
  // meeting a tile are consecutive; a range may lie inside one tile.
  constexpr bool kBalanced = kNarrow || NM <= 16;
  const int64_t pairs = n_tiles * (nb / 2);
  int64_t total, tile_first, tile_last = -1, tile_step = 1;
  int kb_first = 0, kb_end = 0;                                   // kb_end 0: the range ends on a tile boundary
  if constexpr (kBalanced) {
    const int64_t s_begin = 2 * (pairs * blockIdx.x / gridDim.x);
    const int64_t s_end = 2 * (pairs * (blockIdx.x + 1) / gridDim.x);
    total = s_end - s_begin;
    tile_first = s_begin / nb;
    kb_first = static_cast<int>(s_begin - tile_first * nb);         // even
    tile_last = (s_end - 1) / nb;
    kb_end = static_cast<int>(s_end - (s_end / nb) * nb);
  } else {
    total = (blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0) * nb;
    tile_first = blockIdx.x;
    tile_step = gridDim.x;
  }

  if (tid == 0) {
    for (int s = 0; s < C::kWStages; ++s) {
      ptx::mbar_init(&wfull[s], 1);
      ptx::mbar_init(&wempty[s], 8);                              // the pair's eight warps
    }
    for (int s = 0; s < C::kXStages; ++s) {
      ptx::mbar_init(&xfull[s], 1);
      ptx::mbar_init(&xempty[s], 1);                              // one commit after the block's MMAs
    }
    for (int j = 0; j < 2; ++j) {
      ptx::mbar_init(&aready[j], 8);
      ptx::mbar_init(&adone[j], 1);
      ptx::mbar_init(&ahalf[j], 8);
    }
    ptx::mbar_init(mma_idle, 1);
    ptx::mbar_init(xch_full, 32 * kUnpackWarps / 2);
    ptx::mbar_init(xch_empty, 32 * kUnpackWarps / 2);
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
      // step g = (tile, block kb) in tile-major order; counters instead of divisions
      int64_t issued = 0;
      int kb = kb_first, ws = 0;
      uint32_t ph = 0;                          // parity of the current pass over the ring
      int64_t row0 = tile_first * kTileRows;
      for (int64_t g = 0; g < total && !*s_abort; ++g) {
        if (g >= C::kWStages && !ptx::mbar_wait(&wempty[ws], ph ^ 1u)) { fail(); break; }
        ptx::mbar_arrive_expect_tx(&wfull[ws], C::kWStageBytes);
        tma_load_2d(wst + ws * C::kWStageBytes, &wmap, kb * (C::kBB / 4), static_cast<int>(row0), &wfull[ws],
                    pol_w);
        issued = g + 1;
        if (++ws == C::kWStages) { ws = 0; ph ^= 1u; }
        if (++kb == nb) { kb = 0; row0 += tile_step * kTileRows; }
      }
      // never leave copies in flight
      for (int64_t g = issued > C::kWStages ? issued - C::kWStages : 0; g < issued; ++g)
        ptx::mbar_wait(&wfull[g % C::kWStages], static_cast<uint32_t>((g / C::kWStages) & 1));
    }
  } else if (warp == kPkgWarp) {
    // ------------------------------------------------------------ activation-package producer
    if (lane == 0) {
      asm volatile("griddepcontrol.wait;" ::: "memory");   // the prep grid has completed

      int64_t issued = 0;
      int kb = kb_first, xs = 0;
      uint32_t ph = 0;
      for (int64_t g = 0; g < total && !*s_abort; ++g) {
        if (g >= C::kXStages && !ptx::mbar_wait(&xempty[xs], ph ^ 1u)) { fail(); break; }
        ptx::mbar_arrive_expect_tx(&xfull[xs], C::kPkgBytes);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         ptx::smem_u32(xst + xs * C::kPkgBytes)),
                     "l"(pkgs + static_cast<size_t>(kb) * C::kPkgBytes), "r"(C::kPkgBytes),
                     "r"(ptx::smem_u32(&xfull[xs]))
                     : "memory");
        issued = g + 1;
        if (++xs == C::kXStages) { xs = 0; ph ^= 1u; }
        if (++kb == nb) kb = 0;
      }
      for (int64_t g = issued > C::kXStages ? issued - C::kXStages : 0; g < issued; ++g)
        ptx::mbar_wait(&xfull[g % C::kXStages], static_cast<uint32_t>((g / C::kXStages) & 1));
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and operands stay warp-uniform); one
    // elected lane issues the MMAs and commits.
    bool ok = true;
    int xs = 0;
    uint32_t xph = 0;
    // 16 and 32 slots: one lane, elected once, issues and commits every MMA
    bool issuer = false;
    if constexpr (kEarlyHalf) issuer = tc::elect_one();
    for (int64_t g = 0; g < total; ++g) {
      if (__any_sync(0xffffffffu, *s_abort != 0u)) break;
      const int j = static_cast<int>(g & 1);
      const uint32_t par = static_cast<uint32_t>((g >> 1) & 1);
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&xfull[xs], xph));
      if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(kEarlyHalf ? &ahalf[j] : &aready[j], par));
      if (!ok) break;
      tc::fence_after();
      const uint32_t xbase = ptx::smem_u32(xst + xs * C::kPkgBytes);
      const uint64_t bdesc0 = tc::smem_desc_kmajor(xbase, C::kXRows * 16, 128);
      const uint64_t mdesc = tc::smem_desc_kmajor(xbase + C::kXBytes, min_rows<NM>() * 16, 128);
      const uint32_t d = tbase + C::col_d(j);
      const uint32_t a = tbase + C::col_a(j);
      // K-step ks: 16 columns of x = 2 core matrices along K
      auto mma_ks = [&](int ks, bool acc) {
        tc::mma_f16_tmemA(d, a + 8 * ks, bdesc0 + ((ks * 2 * (C::kXRows / 8) * 128) >> 4), C::kIdesc, acc);
      };
      if constexpr (kEarlyHalf) {
        // the first chunks of both warpgroups (K-steps 0-3 and 8-11), then,
        // once the whole A is in, the second chunks and the mins
        if (issuer) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_ks(ks, ks > 0);
#pragma unroll
          for (int ks = 8; ks < 12; ++ks) mma_ks(ks, true);
        }
        __syncwarp();
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&aready[j], par))) {
          ok = false;
          break;
        }
        tc::fence_after();
        if (issuer) {
#pragma unroll
          for (int ks = 4; ks < 8; ++ks) mma_ks(ks, true);
#pragma unroll
          for (int ks = 12; ks < 16; ++ks) mma_ks(ks, true);
          tc::mma_f16_tmemA(tbase + C::col_dmin(j), tbase + C::col_amin(j), mdesc, C::kIdescMin, false);
          tc::commit(&adone[j]);
          tc::commit(&xempty[xs]);
        }
      } else if (tc::elect_one()) {
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) mma_ks(ks, ks > 0);
        tc::mma_f16_tmemA(tbase + C::col_dmin(j), tbase + C::col_amin(j), mdesc, C::kIdescMin, false);
        tc::commit(&adone[j]);
        tc::commit(&xempty[xs]);
      }
      __syncwarp();
      if (++xs == C::kXStages) { xs = 0; xph ^= 1u; }
    }
    if (!ok && lane == 0) fail();
    // tensor memory is freed below only after every MMA issued here completed
    if (kEarlyHalf ? issuer : tc::elect_one()) tc::commit(mma_idle);
    __syncwarp();
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(mma_idle, 0)) && lane == 0) fail();
  } else {
    // ------------------------------------------------------------ unpack + epilogue
    const int wg = warp >> 2;                   // warpgroup 0..3
    const int p = wg >> 1;                      // pair: steps of parity p, tensor-memory buffer p
    const int hf = wg & 1;                      // half of the block (sub-blocks 4hf..4hf+3)
    const int r = tid & 127;                    // row inside the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int b0 = hf * HB;
    float acc[HB];
#pragma unroll
    for (int b = 0; b < HB; ++b) acc[b] = 0.0f;
    float d_prev = 0.0f, dmin_prev = 0.0f;
    // read back this warpgroup's columns of buffer p's D and Dmin (the pair's
    // previous block: its MMAs are complete) and accumulate
    auto drain = [&]() {
      tc::fence_after();
      const uint32_t cd = tbase + lane_base + C::col_d(p) + b0;
      const uint32_t cm = tbase + lane_base + C::col_dmin(p) + b0;
#pragma unroll
      for (int c0 = 0; c0 < HB; c0 += 4) {
        uint32_t dh[4], dl[4], mv[4];
        ld_x4(cd + c0, dh);          // x_hi columns
        ld_x4(cd + NM + c0, dl);     // x_lo columns
        ld_x4(cm + c0, mv);
        tc::wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float dot = __uint_as_float(dh[q]) + __uint_as_float(dl[q]);
          acc[c0 + q] = fmaf(d_prev, dot, fmaf(-dmin_prev, __uint_as_float(mv[q]), acc[c0 + q]));
        }
      }
    };
    // End of a tile: pair 1 hands its sums to pair 0 through shared memory
    // (bounded mbarrier handshake), pair 0 finishes the rows.  A tile shared
    // with a neighbouring CTA (this CTA's first tile: side 1 of boundary
    // blockIdx.x - 1; its last: side 0 of boundary blockIdx.x) goes through
    // the boundary's slot, warp by warp (32 rows): both CTAs' warps store
    // their sums, then count in with one atomic per warp; the second adds
    // side 0 + side 1 (the same order in either CTA) and finishes the rows.
    // Narrow instance: each CTA stores to its own slot (side 0 its first
    // tile, 1 its last) and counts in on the tile's counter; the last of the
    // sharing CTAs adds their slots in CTA order.
    uint32_t n_fin = 0;
    auto finish_tile = [&](int64_t t) -> bool {
      const int64_t row = t * kTileRows + r;
      int side = -1;
      uint32_t slot = 0;
      if constexpr (kNarrow) {                  // slot (blockIdx.x, 0) for the first tile, 1 for the last
        if (t == tile_first && (kb_first != 0 || (tile_first == tile_last && kb_end != 0))) side = 0;
        else if (t == tile_last && kb_end != 0) side = 1;
      } else if (t == tile_first && kb_first != 0) {
        side = 1;
        slot = blockIdx.x - 1;
      } else if (t == tile_last && kb_end != 0) {
        side = 0;
        slot = blockIdx.x;
      }
      float *xw = xchg + (hf * kTileRows + r) * HB;
      bool ok = true;
      if (p == 1) {
        if (n_fin > 0) ok = __all_sync(0xffffffffu, ptx::mbar_wait(xch_empty, (n_fin - 1) & 1u));
        if (ok) {
#pragma unroll
          for (int b = 0; b < HB; ++b) xw[b] = acc[b];
          ptx::mbar_arrive(xch_full);
        }
      } else {
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(xch_full, n_fin & 1u));
        float v[HB];
        bool store = ok;
        if (ok) {
#pragma unroll
          for (int b = 0; b < HB; ++b) v[b] = acc[b] + xw[b];
          ptx::mbar_arrive(xch_empty);
        }
        if (kNarrow && ok && side >= 0) {
          // the CTAs c_lo..c_hi share t: owner of the tile's first and last step pair
          const int64_t c_lo = ((t * (nb / 2) + 1) * gridDim.x - 1) / pairs;
          const int64_t c_hi = (((t + 1) * (nb / 2)) * gridDim.x - 1) / pairs;
          const uint32_t last = static_cast<uint32_t>(c_hi - c_lo);
          float *mine = split_part + ((static_cast<size_t>(blockIdx.x) * 2 + side) * kTileRows + r) * NM + b0;
#pragma unroll
          for (int b = 0; b < HB; ++b) mine[b] = v[b];
          __threadfence();                       // this lane's sums before the warp's count
          __syncwarp();
          uint32_t who = 0u;
          unsigned int *cnt = split_cnt + t * (kUnpackWarps / 2) + (warp & 7);
          if (lane == 0) {
            who = atomicAdd(cnt, 1u);
            if (who == last) *cnt = 0u;          // every sharing CTA counted in: re-armed for the next launch
          }
          store = __shfl_sync(0xffffffffu, who, 0) == last;
          if (store) {
            __threadfence();                     // the other CTAs' sums after their counts
#pragma unroll
            for (int b = 0; b < HB; ++b) v[b] = 0.0f;
            for (int64_t c = c_lo; c <= c_hi; ++c) {
              const int64_t cs = (2 * (pairs * c / gridDim.x)) / nb == t ? 0 : 1;   // t is c's first tile?
              const float *src = split_part + ((static_cast<size_t>(c) * 2 + cs) * kTileRows + r) * NM + b0;
#pragma unroll
              for (int b = 0; b < HB; ++b) v[b] += __ldcg(src + b);
            }
          }
        } else if (ok && side >= 0) {
          float *base = split_part + (static_cast<size_t>(slot) * 2 * kTileRows + r) * NM + b0;
          float *mine = base + side * kTileRows * NM;
#pragma unroll
          for (int b = 0; b < HB; ++b) mine[b] = v[b];
          __threadfence();                       // this lane's sums before the warp's count
          __syncwarp();
          uint32_t who = 0u;
          unsigned int *cnt = split_cnt + slot * (kUnpackWarps / 2) + (warp & 7);
          if (lane == 0) {
            who = atomicAdd(cnt, 1u);
            if (who == 1u) *cnt = 0u;            // both warps counted in: re-armed for the next launch
          }
          store = __shfl_sync(0xffffffffu, who, 0) == 1u;
          if (store) {
            __threadfence();                     // the other CTA's sums after its count
            const float *other = base + (1 - side) * kTileRows * NM;
#pragma unroll
            for (int b = 0; b < HB; ++b) {
              const float o = __ldcg(other + b);
              v[b] = side == 0 ? v[b] + o : o + v[b];
            }
          }
        }
        if (store) {
#pragma unroll
          for (int b = 0; b < HB; ++b) {
            if (b0 + b < batch) {
              const float v_out = scale_softcap(v[b], scale, cap);
              const bool valid = row < n_rows;
              if (valid) logits[static_cast<size_t>(b0 + b) * n_rows + row] = v_out;
              const unsigned long long key =
                  warp_argmax_key(argmax_precap ? v[b] * scale : v_out, static_cast<uint32_t>(row), valid);
              if (lane == 0 && key != 0ull) atomicMax(&s_keys[b0 + b], key);
            }
          }
        }
      }
      ++n_fin;
#pragma unroll
      for (int b = 0; b < HB; ++b) acc[b] = 0.0f;
      return ok;
    };
    bool ok_all = true;
    // The pair's steps g = p, p+2, ...: weight stage, ring parity, block and
    // tile follow by counting (nb and the ring size are even).
    int ws = p, kb = kb_first + p;
    uint32_t wph = 0;
    int64_t tile = tile_first, tile_prev = -1;
    uint32_t i = 0;                             // the pair's step count
    for (int64_t g = p; g < total; g += 2, ++i) {
      if (__any_sync(0xffffffffu, *s_abort != 0u)) { ok_all = false; break; }
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&wfull[ws], wph))) {
        if (lane == 0) fail();
        ok_all = false;
        break;
      }
      const uint8_t *blk = wst + ws * C::kWStageBytes + r * C::kBB;
      RowHdr hd;
      load_row_hdr(blk, hd);
      const uint32_t ta = tbase + lane_base + C::col_a(p) + 64 * hf;
      if (i > 0) {                              // buffer p: previous block's A consumed, D written
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&adone[p], (i - 1) & 1u))) {
          if (lane == 0) fail();
          ok_all = false;
          break;
        }
        drain();
        if (tile != tile_prev && !finish_tile(tile_prev)) {   // that block closed a tile
          if (lane == 0) fail();
          ok_all = false;
          break;
        }
      }
      if constexpr (kEarlyHalf) {
        if (hf == 0) a_chunk_st<kQ4, 0>(blk, chunk_consts<0>(hd.sc03), ta);
        else a_chunk_st<kQ4, 2>(blk, chunk_consts<0>(hd.sc47), ta);
        tc::wait_st();                               // K-steps 0-3 and 8-11 are ready
        tc::fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ahalf[p]);
        if (hf == 0) a_chunk_st<kQ4, 1>(blk, chunk_consts<2>(hd.sc03), ta + 32);
        else a_chunk_st<kQ4, 3>(blk, chunk_consts<2>(hd.sc47), ta + 32);
      } else if (hf == 0) {
        a_chunk_st<kQ4, 0>(blk, chunk_consts<0>(hd.sc03), ta);
        a_chunk_st<kQ4, 1>(blk, chunk_consts<2>(hd.sc03), ta + 32);
      } else {
        a_chunk_st<kQ4, 2>(blk, chunk_consts<0>(hd.sc47), ta);
        a_chunk_st<kQ4, 3>(blk, chunk_consts<2>(hd.sc47), ta + 32);
      }
      if (hf == 0) {
        uint32_t am[8];
        amin_cols(hd, am);
        tc::st_32x32b_x8(tbase + lane_base + C::col_amin(p), am);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&wempty[ws]);   // weight stage fully read
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&aready[p]);
      d_prev = hd.d;
      dmin_prev = hd.dmin;
      tile_prev = tile;
      if ((ws += 2) >= C::kWStages) { ws -= C::kWStages; wph ^= 1u; }
      if ((kb += 2) >= nb) { kb -= nb; tile += tile_step; }
    }
    // The pair's last block and the last tile.  Both pairs get here having
    // taken part in the same tile hand-overs: nb is even, so each pair owns
    // blocks of every tile.
    if (ok_all && i > 0) {
      if (__all_sync(0xffffffffu, ptx::mbar_wait(&adone[p], (i - 1) & 1u))) {
        drain();
        if (!finish_tile(tile_prev) && lane == 0) fail();
      } else if (lane == 0) {
        fail();
      }
    }
    tc::fence_before();
  }

  __syncthreads();
  // the next forward's prep kernel may launch now (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised once even when host threads race to the first call).
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
  return fn;
}

template <int NM, bool kQ4, bool kNarrow>
cudaError_t launch_tc_nm(const LaunchArgs &a, const CUtensorMap &map) {
  using C = TcCfg<NM, kQ4>;
  static std::atomic<unsigned long long> configured{0};   // one bit per device; host threads may race here
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_tc_kernel<NM, kQ4, kNarrow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int nb = a.k / kBlockWeights;
  {
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(nb, min_rows<NM>());
    pc.blockDim = dim3(kPrepThreads);
    pc.stream = a.stream;
    cudaLaunchAttribute pa[1];
    pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // may start before the previous grid ends
    pa[0].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = pa;
    pc.numAttrs = 1;
    e = cudaLaunchKernelEx(&pc, prep_x_kernel<NM>, a.hidden, a.gamma, a.eps, a.batch, a.k, a.ws.xpkg);
    if (e != cudaSuccess) return e;
  }
  const int64_t n_tiles = (a.n_rows + kTileRows - 1) / kTileRows;
  const int64_t pairs = n_tiles * (nb / 2);   // a narrow matrix spreads its step pairs over the SMs
  const int64_t grid = kNarrow ? (pairs < a.num_sms ? pairs : a.num_sms) : (n_tiles < a.num_sms ? n_tiles : a.num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // may start before the prep grid ends
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<NM, kQ4, kNarrow>, map, static_cast<const uint8_t *>(a.ws.xpkg), nb,
                            a.n_rows, a.batch, a.scale, a.cap, a.logits, a.ws.keys, a.ws.ticket, a.argmax,
                            a.ws.status, a.ws.split_part, a.ws.split_cnt, a.argmax_precap ? 1 : 0);
}

}  // namespace

size_t tc_workspace_bytes(int k) { return static_cast<size_t>(k / kBlockWeights) * TcCfg<32>::kPkgBytes; }

int tc_batch_slots(int batch) { return batch <= 8 ? 8 : batch <= 16 ? 16 : 32; }

size_t tc_split_floats(int num_sms, int max_batch) {
  return static_cast<size_t>(num_sms) * 2 * kTileRows * tc_batch_slots(max_batch);
}

// per boundary between CTAs (one per SM) for a large matrix, per 128-row tile
// for a narrow one (fewer tiles than SMs): at most max(SMs, tiles) entries
size_t tc_split_counters(int num_sms) { return static_cast<size_t>(num_sms) * (kUnpackWarps / 2); }

// Batches 1..32 with an even number of blocks per row (both pairs of unpack
// warpgroups then own blocks of every tile), either weight format.  Batch 1
// takes this path only for a K the fused batch-1 kernel has no build for.
bool tc_supported(int batch, int k) {
  const int nb = k / kBlockWeights;
  return batch >= 1 && batch <= 32 && nb >= 2 && nb % 2 == 0;
}

cudaError_t tc_encode_weights(CUtensorMap *map, const void *weights, int64_t n_rows, int k, bool q4) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encoder();
  if (!enc) return cudaErrorNotSupported;
  // 32-bit elements: a block (176 or 144 bytes, both multiples of 16) is the
  // box's inner extent, so every box starts on a 16-byte boundary.  L2 fetches
  // are promoted to 64 bytes only: a box row is 176 bytes, and with 256-byte
  // promotion the evict-first lines around it were often gone before the
  // neighbouring box came for them (2.5 % more DRAM reads than the matrix)
  const int bb = q4 ? kBlockBytesQ4 : kBlockBytes;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(k / kBlockWeights) * (bb / 4),
                              static_cast<cuuint64_t>(n_rows)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(k / kBlockWeights) * bb};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(bb / 4), kTileRows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(weights), gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool kNarrow>
cudaError_t launch_tc_sched(const LaunchArgs &a, const CUtensorMap &map) {
  const int nm = tc_batch_slots(a.batch);
  if (a.q4) {
    if (nm == 8) return launch_tc_nm<8, true, kNarrow>(a, map);
    if (nm == 16) return launch_tc_nm<16, true, kNarrow>(a, map);
    return launch_tc_nm<32, true, kNarrow>(a, map);
  }
  if (nm == 8) return launch_tc_nm<8, false, kNarrow>(a, map);
  if (nm == 16) return launch_tc_nm<16, false, kNarrow>(a, map);
  return launch_tc_nm<32, false, kNarrow>(a, map);
}

cudaError_t launch_tc(const LaunchArgs &a, const CUtensorMap &map) {
  const int64_t n_tiles = (a.n_rows + kTileRows - 1) / kTileRows;
  return n_tiles < a.num_sms ? launch_tc_sched<true>(a, map) : launch_tc_sched<false>(a, map);
}

}  // namespace muse
