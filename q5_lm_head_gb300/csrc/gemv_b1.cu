// Fused batch-1 output stage: final RMSNorm prologue, Q5_K weight-streaming
// GEMV on the CUDA cores, scale + soft cap epilogue and two-level argmax, in
// one persistent launch ("Chapter 20 — Final norm, LM head, and the soft cap",
// §20.1 what it computes, §20.3 the 924.6 MB weight stream, §20.4 the cap).
//
// The same kernel also runs a group of up to four matrices against one normed
// input in one launch (the Q/K/V/gate projections, "Chapter 9 — The Muse
// Glimmer architecture", Figure 9.1 and §9.8): the weight tiles of all
// matrices form one sequence, each tile belongs to one matrix and writes that
// matrix's output with its own scale and cap.
//
// A K that is S times a built width (S x 6,656 or S x 4,096 columns) runs the
// same kernel split along K: CTAs [c*G/S, (c+1)*G/S) of a G-CTA grid stream
// column chunk c of every row, with chunk c of the input row; a tile of a
// chunk is kRows row-strided copies, one per producer lane.  A row tile's S
// chunk partials meet in global memory: each chunk CTA stores its rows' sums
// as it goes; after its last tile the CTA counts in on each of its tiles'
// counters (a thread per tile: release fence, atomic add, acquire fence when
// last), and the whole CTA finishes the tiles it arrived last on: the S
// partials added in chunk order (the same bits whichever CTA that is), then
// scale, cap and argmax.  No CTA waits on another.
//
// A Q4_K matrix of at most three chunks with few rows (an even share over the
// SMs is at most eight tiles per CTA, the FFN down projection's shape) has no
// hand-off at all: the K loop.  Each CTA takes an even share of rows and
// streams all chunks of them, chunk after chunk (its tiles, rounded up to an
// even count with an empty tile, for chunk 0, then for chunk 1, ...).  The
// whole input row is staged once (in the last stage and the later chunks'
// plane slots, so that only one stage waits for the prologue); the consumers
// quantise all chunks in one pass (one RMS factor for the row), keep chunk 0's
// planes in registers and the later chunks' plane words, step and column sums
// in shared memory, and load a chunk's as its first tile comes up.  A producer keeps the
// chunk sums of its rows in registers (tile t of every chunk is its tile),
// adds them in chunk order and finishes a row with the last chunk.
//
// The argmax ranks the returned logit, or (argmax_precap) scale * raw before
// the cap; the two orders agree except where the f32 cap rounds distinct
// values to the same float.
//
// Warp roles (one CTA per SM)
//   * consumer warps: thread (kb, c) owns 64 columns, block kb, sub-blocks 2c
//     and 2c+1, for the whole launch (column-stationary).  Four teams of such
//     threads ("streams") split the rows of a tile.  The four threads of one
//     block add their row contributions with two shuffles and one of them
//     writes the block's partial into a ring of partial slots.  Consumers wait
//     for nothing but "stage full".
//   * two producer warps: move tiles of kRows consecutive weight rows
//     (contiguous in HBM) into a ring of shared-memory stages with 1-D bulk
//     copies (cp.async.bulk + mbarrier transaction counts, L2 evict-first);
//     producer p owns the stages of parity p, so two copies are always being
//     armed independently.  CTAs take tiles round-robin, so the whole GPU
//     streams one contiguous stretch; a small single matrix, where the CTA with
//     the most rows sets the time, is instead cut into even shares of rows
//     (12-row tiles and one shorter one per CTA).  The arming thread writes each
//     stage's row count for the consumers.  Each time consumers release one of its
//     stages, a producer first re-arms it with its next tile and then finishes
//     the released stage's rows: fixed-order sum of the block partials, scale +
//     soft cap, store, argmax key.  The partial ring has two slots more than
//     the stage ring, so a slot is never rewritten before its producer has read
//     it (the rewrite needs a stage that the same producer arms only
//     afterwards).
//   * prologue: thread 0 bulk-copies the hidden row (and gamma) into the last
//     stage (gamma into the one before when both do not fit) before anything
//     else, then initialises the other barriers and arms the first weight
//     tiles of the other stages itself, before the CTA-wide barrier; the
//     producers arm the rest.
//     The consumers build the RMS factor and their activation planes from
//     shared memory (the four threads of a unit each quantise a quarter of its
//     64 columns and share the plane words through the same stage), then
//     release the stage, and only then is it armed with its first weight tile.
//
// Arithmetic of a consumer thread (exact up to f32 rounding of the last steps)
//   Its 64 normalised activations x_j = r * h_j * gamma_j are written as
//   x_j = r * sigma * xi_j with integers |xi_j| < 2^22 and a per-unit power of
//   two sigma (the largest |h * gamma| of the unit's 64 columns lies in
//   [2^21, 2^22) sigma, so the scaling is exact and needs no division), stored
//   as three byte planes xi = 65536*x2 + 256*x1 + x0 (x2 signed, x1 and x0
//   unsigned).  The RMS factor r only scales sigma and the column sums.
//   For each sub-block s, sum_j q_j xi_j is built with dp4a on four 5-bit quants
//   per word (low nibble | high bit << 4; high nibbles are taken as 2q so no
//   extra shift is needed) against each plane, in exact integer arithmetic.
//   Then raw += d * r * sigma * sum_s sc_s * (that) - dmin * sum_s m_s * sum_j x_j,
//   which is sum_j (d*sc_s*q_j - dmin*m_s) x_j up to rounding (§20.1 matvec
//   with the Q5_K weight w = d*sc*q - dmin*m).
#include <atomic>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace muse {
namespace {

constexpr int kRows = 12;           // weight rows per pipeline stage (one 1-D bulk copy)
constexpr int kStreams = 4;         // row teams of consumer threads
constexpr int kMaxSmem = 227 * 1024 - 1024;   // opt-in limit minus static shared memory
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

// K loop inside the CTA (kKLoop): a K of up to kMaxKLoopChunks chunks of NB
// blocks, every CTA streaming all chunks of its own rows, chunk after chunk.
constexpr int kMaxKLoopChunks = 3;
constexpr int kMaxKLoopTiles = 8;      // tiles of a CTA's rows (even), so its row sums fit in registers

// NB blocks per row; kQ4: Q4_K blocks (144 bytes, nibbles only) instead of Q5_K.
template <int NB, bool kQ4, bool kKLoop = false>
struct B1Cfg {
  static constexpr int kUnits = 4 * NB;                    // (block, 64-column group) units per row
  static constexpr int kConsumers = kUnits * kStreams;
  static_assert(kConsumers % 32 == 0, "consumer threads must fill whole warps");
  static_assert(kUnits % 4 == 0, "the four units of a block stay inside one stream");
  static_assert(kRows % kStreams == 0, "each stream takes the same number of rows");
  static constexpr int kConsumerWarps = kConsumers / 32;
  static constexpr int kProducerWarps = 2;
  static constexpr int kThreads = kConsumers + 32 * kProducerWarps;
  static constexpr int kBB = kQ4 ? kBlockBytesQ4 : kBlockBytes;   // bytes per block
  static constexpr int kRowBytes = NB * kBB;
  static constexpr int kStageBytes = kRows * kRowBytes;
  static constexpr int kSlotBytes = kRows * NB * 4;         // one partial per (row, block)
  static constexpr int kFixedBytes = 640;                   // barriers, scratch, tile table, stage row counts
  // (max, sum) of every quarter in the prologue; with the K loop (one table
  // per chunk) chunk 0's is at the end of the staging stage and the later
  // chunks' in the partial slots (unused until the first tile)
  static constexpr int kExBytes = kKLoop ? 0 : kUnits * 4 * 8;
  // K loop: the plane words, RMS-scaled step and column sums of chunks 1 and 2
  // of every unit (chunk 0 stays in registers until its tiles are done)
  static constexpr int kKPlaneStride = 52;                  // 48 plane words, sigma/2, two sums, pad
  static constexpr int kPlanesBytes = kKLoop ? (kMaxKLoopChunks - 1) * kUnits * kKPlaneStride * 4 : 0;
  static constexpr int kStagesFit =
      (kMaxSmem - kFixedBytes - kExBytes - kPlanesBytes - 2 * kSlotBytes) / (kStageBytes + kSlotBytes);
  static constexpr int kStages = (kStagesFit > 8 ? 8 : kStagesFit) & ~1;   // even: one parity per producer
  static_assert(kStages >= 4, "need at least double buffering per producer");
  static constexpr int kSlots = kStages + 2;
  static constexpr int kSmemBytes =
      kStages * kStageBytes + kSlots * kSlotBytes + kFixedBytes + kExBytes + kPlanesBytes;
  static_assert(kSmemBytes <= kMaxSmem, "shared memory budget");
  // the prologue stages hidden (and gamma) in the last stage, or gamma in the one
  // before when both do not fit one stage.  The K loop stages the whole hidden
  // row (every chunk; gamma is read from global memory) in the last stage up
  // to chunk 0's quarter table (kKStageRowBytes) and the rest in the plane
  // slots, which are written only after the row has been read.
  static_assert(NB * kBlockWeights * 4 <= kStageBytes, "hidden fits one stage");
  static constexpr int kKStageRowBytes = kStageBytes - kUnits * 4 * 8;
  static_assert(!kKLoop || (kKStageRowBytes >= NB * kBlockWeights * 4 && kKStageRowBytes % 64 == 0 &&
                            kMaxKLoopChunks * NB * kBlockWeights * 4 <= kKStageRowBytes + kPlanesBytes),
                "K loop: chunk 0 in the staging stage, the hidden row in the stage and the plane slots");
  static_assert(kUnits * kKPlaneStride <= NB * kBlockWeights, "K loop: chunk 0's planes over its columns");
  static constexpr int kHoldStages = !kKLoop && 2 * NB * kBlockWeights * 4 > kStageBytes ? 2 : 1;
  static constexpr int kEarlyTiles = kStages - kHoldStages;   // armed before the CTA-wide barrier
  // after the activations are loaded the staging stage holds, per unit, its
  // plane words (p2, p1, p0: 16 words each, padded to 52 so the units' rows
  // fall on distinct banks)
  static constexpr int kPlaneStride = 52;
  static_assert(kUnits * kPlaneStride * 4 <= kStageBytes, "plane area");
  static_assert(!kKLoop || (kMaxKLoopChunks - 1) * kUnits * 4 * 8 <= kSlots * kSlotBytes,
                "K loop: the later chunks' quarter tables fit the partial slots");
};

__device__ __forceinline__ uint32_t rotl32(uint32_t v, uint32_t s) { return __funnelshift_l(v, v, s); }

// Four bytes, one per 4 consecutive activations, of the 24-bit integer planes.
struct XPlanes {
  uint32_t p2[8], p1[8], p0[8];   // word i holds positions 4i..4i+3
};

// The three plane words (byte t = activation t) of four consecutive activations.
// fmaf(x, inv, 1.5*2^23) rounds x*inv to the nearest integer (ties to even) in
// the mantissa: for |xi| < 2^22 its bits are 0x4B400000 + xi, so bytes 0 and 1
// are those of xi and byte 2 is xi's signed high byte plus 0x40.
__device__ __forceinline__ void quantize_chunk(const float (&x)[4], float inv, uint32_t &w2, uint32_t &w1,
                                               uint32_t &w0) {
  uint32_t b[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) b[t] = __float_as_uint(fmaf(x[t], inv, kRoundMagic));
  const uint32_t t01 = __byte_perm(b[0], b[1], 0x5140);   // b0.0 b1.0 b0.1 b1.1
  const uint32_t t23 = __byte_perm(b[2], b[3], 0x5140);
  w0 = __byte_perm(t01, t23, 0x5410);
  w1 = __byte_perm(t01, t23, 0x7632);
  const uint32_t u01 = __byte_perm(b[0], b[1], 0x0062);   // b0.2 b1.2 - -
  const uint32_t u23 = __byte_perm(b[2], b[3], 0x0062);
  // high byte h + 0x40 in 0..127 -> h: flip bit 6, then copy bit 6 into bit 7
  const uint32_t h = __byte_perm(u01, u23, 0x5410) ^ 0x40404040u;
  w2 = h | ((h & 0x40404040u) << 1);
}

// Biased exponent of the power-of-two quantisation factor inv of a unit whose
// largest |value| is m > 0 (finite): for m in [2^(E-127), 2^(E-126)), E its
// biased exponent, inv = 2^(148-E), so m * inv lies in [2^21, 2^22) and every
// |xi| < 2^22; x * inv is exact.  Capped at 252 (m below 2^-104 gets a coarser
// step) so that 1 / (2 inv) = 2^(126-eb) stays a normal float.
__device__ __forceinline__ int pow2_step_exponent(float m) {
  const int e = static_cast<int>(__float_as_uint(m) >> 23);
  return 275 - e < 252 ? 275 - e : 252;
}

// Per-thread constants that select this thread's sub-blocks 2c and 2c+1.
struct UnitSel {
  uint32_t rot;        // rotate that brings bit 2c of each qh byte to bit 4
  uint32_t sh_sc, sh_m, msk_lo, sh_hi2, msk_hi;
  bool upper;          // sub-blocks 4..7: scales split over two bytes
  int qs_off;          // byte offset of this thread's 32 low-nibble bytes
};

template <bool kQ4>
__device__ __forceinline__ UnitSel make_unit_sel(int c) {
  UnitSel u;
  u.upper = c >= 2;
  u.sh_sc = u.upper ? 16u * (c - 2) : 16u * c;
  u.sh_m = u.upper ? 16u * (c - 2) + 4u : 16u * c;
  u.msk_lo = u.upper ? 0x0F0Fu : 0x3F3Fu;
  u.sh_hi2 = u.upper ? 16u * (c - 2) + 2u : 0u;
  u.msk_hi = u.upper ? 0x3030u : 0u;
  u.rot = static_cast<uint32_t>(4 - 2 * c) & 31u;
  u.qs_off = (kQ4 ? kOffQsQ4 : kOffQs) + 32 * c;
  return u;
}

// This thread's contribution to one row: sum over its 64 columns of
// (d*sc_s*q - dmin*m_s) * x, from the row's Q5_K (or Q4_K) block `blk` in
// shared memory.
template <bool kQ4>
__device__ __forceinline__ float unit_partial(const uint8_t *blk, const UnitSel &us, const XPlanes &xl,
                                              const XPlanes &xh, float sx_lo, float sx_hi, float sigma_half) {
  const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
  const uint4 qs0 = *reinterpret_cast<const uint4 *>(blk + us.qs_off);
  const uint4 qs1 = *reinterpret_cast<const uint4 *>(blk + us.qs_off + 16);
  const uint32_t A[8] = {qs0.x, qs0.y, qs0.z, qs0.w, qs1.x, qs1.y, qs1.z, qs1.w};
  uint32_t H[8] = {};
  if constexpr (!kQ4) {
    const uint4 qh0 = *reinterpret_cast<const uint4 *>(blk + kOffQh);
    const uint4 qh1 = *reinterpret_cast<const uint4 *>(blk + kOffQh + 16);
    H[0] = qh0.x; H[1] = qh0.y; H[2] = qh0.z; H[3] = qh0.w;
    H[4] = qh1.x; H[5] = qh1.y; H[6] = qh1.z; H[7] = qh1.w;
  }
  int l2 = 0, h2 = 0;
  unsigned l1 = 0, l0 = 0, h1 = 0, h0 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t qlo, qhi;
    if constexpr (kQ4) {
      qlo = A[i] & 0x0F0F0F0Fu;                                          // q
      qhi = (A[i] >> 3) & 0x1E1E1E1Eu;                                   // 2q
    } else {
      const uint32_t t = rotl32(H[i], us.rot);                           // high bits at 4 (lo) and 5 (hi)
      qlo = (A[i] & 0x0F0F0F0Fu) | (t & 0x10101010u);                    // q
      qhi = ((A[i] >> 3) & 0x1E1E1E1Eu) | (t & 0x20202020u);             // 2q
    }
    l2 = __dp4a(static_cast<int>(qlo), static_cast<int>(xl.p2[i]), l2);
    l1 = __dp4a(qlo, xl.p1[i], l1);
    l0 = __dp4a(qlo, xl.p0[i], l0);
    h2 = __dp4a(static_cast<int>(qhi), static_cast<int>(xh.p2[i]), h2);
    h1 = __dp4a(qhi, xh.p1[i], h1);
    h0 = __dp4a(qhi, xh.p0[i], h0);
  }
  // scales and mins of sub-blocks 2c (low byte) and 2c+1 (high byte)
  const uint32_t wsc = us.upper ? hdr.w : hdr.y;
  const uint32_t wm = us.upper ? hdr.w : hdr.z;
  const uint32_t scp = ((wsc >> us.sh_sc) & us.msk_lo) | ((hdr.y >> us.sh_hi2) & us.msk_hi);
  const uint32_t mp = ((wm >> us.sh_m) & us.msk_lo) | ((hdr.z >> us.sh_hi2) & us.msk_hi);
  const int sc_lo2 = static_cast<int>((scp & 0xFFu) << 1);   // x2: low nibbles carry q, high 2q
  const int sc_hi = static_cast<int>(scp >> 8);
  const int a2 = l2 * sc_lo2 + h2 * sc_hi;
  const int a1 = static_cast<int>(l1) * sc_lo2 + static_cast<int>(h1) * sc_hi;
  const int a0 = static_cast<int>(l0) * sc_lo2 + static_cast<int>(h0) * sc_hi;
  const float dotv = fmaf(static_cast<float>(a2), 65536.0f, fmaf(static_cast<float>(a1), 256.0f, static_cast<float>(a0)));
  const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&hdr.x));   // (d, dmin)
  const float mins = fmaf(static_cast<float>(mp & 0xFFu), sx_lo, static_cast<float>(mp >> 8) * sx_hi);
  return fmaf(dd.x * sigma_half, dotv, -dd.y * mins);
}

// The matrices of one launch: tiles [tile_end[s-1], tile_end[s]) belong to
// matrix s (tile_end[-1] = 0).
struct SegTable {
  GemvSegment seg[kMaxSegments];
  int64_t tile_end[kMaxSegments];
  int n;
  int argmax_precap;   // argmax key: raw * scale (before the cap) instead of the returned logit
  // Balanced tiles (one small matrix): CTA c takes rows_per (+1 for c < extra)
  // consecutive rows, cut into tiles of kRows rows and one shorter last tile.
  // Otherwise CTA c takes the kRows-row tiles c, c + grid, ...
  int balanced;
  int rows_per, extra;
  int grid;            // CTAs of the launch
};

// Where global tile `tile` lives: its matrix, its first row there and its rows.
struct TileLoc {
  int s;
  int64_t r0;
  int rows;
};

template <bool kGroup>
__device__ __forceinline__ TileLoc locate(const SegTable &T, int64_t tile) {
  TileLoc L;
  L.s = 0;
  int64_t t0 = 0;
  if constexpr (kGroup) {
#pragma unroll
    for (int i = 1; i < kMaxSegments; ++i)
      if (i < T.n && tile >= T.tile_end[i - 1]) {
        L.s = i;
        t0 = T.tile_end[i - 1];
      }
  }
  L.r0 = (tile - t0) * kRows;
  const int64_t n_rows = T.seg[L.s].n_rows;
  L.rows = n_rows - L.r0 < kRows ? static_cast<int>(n_rows - L.r0) : kRows;
  return L;
}

template <int NB, bool kGroup, bool kQ4, bool kSplit, bool kKLoop>
__global__ void __launch_bounds__(B1Cfg<NB, kQ4, kKLoop>::kThreads, 1)
    gemv_b1_kernel(const float *__restrict__ hidden, const float *__restrict__ gamma, float eps,
                   const __grid_constant__ SegTable segs, unsigned long long *keys, unsigned int *ticket,
                   int32_t *argmax, uint32_t *status, float2 *lse_parts, int n_chunks, float *split_part,
                   unsigned int *split_cnt) {
  static_assert(!(kSplit && kGroup), "a grouped launch is not split along K");
  static_assert(!kKLoop || (kSplit && kQ4), "the K loop runs Q4_K launches split along K");
  using C = B1Cfg<NB, kQ4, kKLoop>;
  constexpr int K = NB * kBlockWeights;                                    // columns of one chunk
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *stages = smem;
  float *slots = reinterpret_cast<float *>(smem + C::kStages * C::kStageBytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStageBytes + C::kSlots * C::kSlotBytes);
  uint64_t *empty = full + C::kStages;
  uint64_t *pro_full = empty + C::kStages;                                 // hidden (+ gamma) staged
  uint64_t *pro_done = pro_full + 1;                                       // consumers done with them
  float *s_red = reinterpret_cast<float *>(pro_done + 1);                  // [32]
  // the prologue's staging area: the last stage (and the one before, for gamma,
  // when both rows do not fit one stage), until their first weight tiles
  const float *s_hidden = reinterpret_cast<const float *>(stages + (C::kStages - 1) * C::kStageBytes);
  const float *s_gamma = C::kHoldStages == 1
                             ? s_hidden + K
                             : reinterpret_cast<const float *>(stages + (C::kStages - 2) * C::kStageBytes);
  unsigned long long *s_best = reinterpret_cast<unsigned long long *>(s_red + 32);
  volatile uint32_t *s_abort = reinterpret_cast<volatile uint32_t *>(s_best + 1);
  float2 *s_ms = reinterpret_cast<float2 *>(s_best + 2);                   // [2] producers' (max, sum exp)
  // [kUnits][4]; with the K loop chunk 0's at the end of the staging stage
  float2 *s_ex = kKLoop ? reinterpret_cast<float2 *>(const_cast<float *>(s_hidden) + C::kKStageRowBytes / 4)
                        : reinterpret_cast<float2 *>(reinterpret_cast<uint8_t *>(full) + C::kFixedBytes);
  // K loop: [chunk 1, 2][kUnits][kKPlaneStride] words
  uint32_t *s_planes = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(full) + C::kFixedBytes + C::kExBytes);
  static_assert(16 * C::kStages + 176 <= 512, "fixed area: barriers and scratch");
  // rows of the tile in each stage, written by whoever arms the stage before its
  // expect-tx arrive (release) and read by the consumers after the stage's
  // completion (acquire): the consumers never look the tile up themselves
  int *s_rows = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(full) + 512);   // [kStages]
  static_assert(512 + 4 * C::kStages <= C::kFixedBytes, "stage row counts");

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // Programmatic dependent launch: nothing of the previous launch's memory is
  // touched before it has completed, and the next launch in the stream may
  // start its CTAs as this launch's CTAs leave their SMs (one CTA fills an SM,
  // so they cannot share one).  Not with the (max, sum exp) pairs: the small
  // normaliser kernel that follows would then sit on the SMs beside this one.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (lse_parts == nullptr) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // This CTA's tiles: tile_first, tile_first + tile_step, ... of its chunk
  // (one chunk, all CTAs, unless split along K).  32-bit arithmetic: the grid
  // is at most the SM count and a tile count fits easily.
  int chunk = 0, tile_first = static_cast<int>(blockIdx.x), tile_step = static_cast<int>(gridDim.x);
  if constexpr (kSplit && !kKLoop) {
    const int g = static_cast<int>(gridDim.x), bx = static_cast<int>(blockIdx.x);
    chunk = ((bx + 1) * n_chunks - 1) / g;
    const int lo = chunk * g / n_chunks;
    tile_first = bx - lo;
    tile_step = (chunk + 1) * g / n_chunks - lo;
  }
  const float *x_src = hidden + static_cast<size_t>(chunk) * K;           // the chunk's input columns
  const float *g_src = gamma ? gamma + static_cast<size_t>(chunk) * K : nullptr;
  if (tid == 0) {
    // The hidden row and gamma go out first, ahead of everything else: the
    // prologue waits on them, and a launch this small is a chain of latencies.
    ptx::mbar_init(pro_full, 1);
    ptx::fence_barrier_init();
    const uint32_t row_bytes = static_cast<uint32_t>(K) * 4u;
    if constexpr (kKLoop) {                // every chunk of the row; gamma stays in global memory
      const uint32_t total = static_cast<uint32_t>(n_chunks) * row_bytes;
      const uint32_t first = total < C::kKStageRowBytes ? total : C::kKStageRowBytes;
      ptx::mbar_arrive_expect_tx(pro_full, total);
      ptx::bulk_g2s_nohint(const_cast<float *>(s_hidden), hidden, first, pro_full);
      if (total > first) ptx::bulk_g2s_nohint(s_planes, hidden + first / 4, total - first, pro_full);
    } else {
      ptx::mbar_arrive_expect_tx(pro_full, gamma ? 2u * row_bytes : row_bytes);
      ptx::bulk_g2s_nohint(const_cast<float *>(s_hidden), x_src, row_bytes, pro_full);
      if (gamma) ptx::bulk_g2s_nohint(const_cast<float *>(s_gamma), g_src, row_bytes, pro_full);
    }
  }
  const int n_tiles = static_cast<int>(segs.tile_end[segs.n - 1]);
  int my_tiles = tile_first < n_tiles ? (n_tiles - 1 - tile_first) / tile_step + 1 : 0;
  // balanced share: rows [b_first, b_first + b_rows) of matrix 0
  const int bx = static_cast<int>(blockIdx.x);
  const int b_first = bx * segs.rows_per + (bx < segs.extra ? bx : segs.extra);
  const int b_rows = segs.rows_per + (bx < segs.extra ? 1 : 0);
  if (segs.balanced) my_tiles = (b_rows + kRows - 1) / kRows;
  // K loop: the CTA's tiles (rounded up to an even count, an empty tile
  // padding an odd one, so that every chunk's tile t goes to producer t mod 2)
  // for chunk 0, then for chunk 1, ...: local tile j is tile j mod kl_tiles of
  // chunk j / kl_tiles
  const int kl_tiles = my_tiles + (my_tiles & 1);
  if constexpr (kKLoop) my_tiles = kl_tiles * n_chunks;
  // local tile j of this CTA: its matrix, first row and rows
  auto tile_at = [&](int j) -> TileLoc {
    if (segs.balanced) {
      if constexpr (kKLoop) j %= kl_tiles;
      const int left = b_rows - j * kRows;
      return TileLoc{0, b_first + j * kRows, left <= 0 ? 0 : (left < kRows ? left : kRows)};
    }
    return locate<kGroup>(segs, tile_first + static_cast<int64_t>(j) * tile_step);
  };
  // weight tiles armed by the barrier thread before the CTA-wide barrier; a
  // split chunk's tiles are row-strided (one copy per row), so its producers
  // arm them, a row per lane, but the K loop's first tile (which its consumers
  // wait for first) goes out ahead of the others from the barrier thread
  constexpr int kEarly = kKLoop ? 1 : kSplit ? 0 : C::kEarlyTiles;
  // the rows of local tile j: one bulk copy, or one per row of a split chunk
  // (rows n_chunks * kRowBytes apart); lanes l0, l0 + ls, ... issue them
  auto issue_tile = [&](const TileLoc &L, int st, uint64_t policy, int l0, int ls, int q) {
    uint8_t *dst = stages + st * C::kStageBytes;
    if constexpr (kSplit) {
      const int64_t stride = static_cast<int64_t>(n_chunks) * C::kRowBytes;
      const uint8_t *src = segs.seg[0].w + L.r0 * stride + static_cast<int64_t>(q) * C::kRowBytes;
      for (int i = l0; i < L.rows; i += ls)
        ptx::bulk_g2s(dst + i * C::kRowBytes, src + i * stride, C::kRowBytes, &full[st], policy);
    } else if (l0 == 0) {
      ptx::bulk_g2s(dst, segs.seg[L.s].w + L.r0 * C::kRowBytes, static_cast<uint32_t>(L.rows * C::kRowBytes),
                    &full[st], policy);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], C::kConsumerWarps);
    }
    ptx::mbar_init(pro_done, C::kConsumerWarps);
    *s_best = 0ull;
    *s_abort = 0u;
    ptx::fence_barrier_init();
    // Then the first weight tiles (the stages that hold no prologue data),
    // from code this thread is already running; the producers arm the later
    // tiles.
    const uint64_t policy = ptx::policy_evict_first();
    for (int j = 0; j < kEarly && j < my_tiles; ++j) {
      const TileLoc L = tile_at(j);
      s_rows[j] = L.rows;
      ptx::mbar_arrive_expect_tx(&full[j], static_cast<uint32_t>(L.rows * C::kRowBytes));
      issue_tile(L, j, policy, 0, 1, kKLoop ? j / kl_tiles : chunk);
    }
  }
  __syncthreads();

  auto fail = [&]() {
    atomicOr(status, kStatusWaitTimeout);
    *s_abort = 1u;
  };

  if (warp >= C::kConsumerWarps) {
    // ------------------------------------------------------------ producers + row epilogue
    // Producer pw handles the CTA's tiles of local index j = pw, pw+2, ...: stage
    // j % kStages and partial slot j % kSlots (both rings have even length).
    const int pw = warp - C::kConsumerWarps;
    const uint64_t policy = ptx::policy_evict_first();
    constexpr int kHoldTile = C::kStages - 1;  // local tile whose stage holds the prologue data
    // epilogue: lane pair (2er, 2er+1) sums row er's block partials, alternating
    static_assert(kRows <= 16, "two lanes per row");
    const int er = lane >> 1, eq = lane & 1;
    unsigned long long best = 0ull;
    MaxSum ms = ms_empty();                     // log-softmax normaliser of this lane's rows
    // K loop: the chunk sums so far of row er of this producer's tiles t = pw,
    // pw + 2, ... (register k holds tile 2k + pw)
    float racc[kMaxKLoopTiles / 2];
#pragma unroll
    for (int i = 0; i < kMaxKLoopTiles / 2; ++i) racc[i] = 0.0f;
    // finish the rows of local tile j (its consumers have released its stage)
    auto finish = [&](int j) {
      const TileLoc L = tile_at(j);
      const GemvSegment &G = segs.seg[L.s];
      const float *pr = slots + (j % C::kSlots) * (C::kSlotBytes / 4) + er * NB;
      float sacc = 0.0f;
      if (er < kRows) {
#pragma unroll
        for (int g = 0; g < NB; g += 2)
          if (g + eq < NB) sacc += pr[g + eq];
      }
      sacc += __shfl_xor_sync(0xffffffffu, sacc, 1);
      if constexpr (kKLoop) {
        // the chunk partials of a row added in chunk order, from zero; the
        // rows are finished with the last chunk
        const int q = j / kl_tiles, k2 = (j % kl_tiles) >> 1;
        float prev = 0.0f;
#pragma unroll
        for (int i = 0; i < kMaxKLoopTiles / 2; ++i)
          if (i == k2) prev = racc[i];
        sacc = (q == 0 ? 0.0f : prev) + sacc;
        if (q < n_chunks - 1) {
#pragma unroll
          for (int i = 0; i < kMaxKLoopTiles / 2; ++i)
            if (i == k2) racc[i] = sacc;
          return;
        }
      } else if constexpr (kSplit) {
        // this chunk's row sums out (plain stores); the CTA counts the tile in
        // and finishes it after its last tile, off the copy-issue path
        if (eq == 0 && er < L.rows) split_part[static_cast<int64_t>(chunk) * G.n_rows + L.r0 + er] = sacc;
        __syncwarp();
        return;
      }
      if (eq == 0 && er < L.rows) {
        const int64_t row = L.r0 + er;
        const float out = scale_softcap(sacc, G.scale, G.cap);
        G.out[row] = out;
        if constexpr (!kGroup) {
          best = umax64(best, argmax_key(segs.argmax_precap ? sacc * G.scale : out, static_cast<uint32_t>(row)));
          if (lse_parts) ms = ms_add(ms, out);
        }
      }
      __syncwarp();
    };
    auto wait_released = [&](int j) -> bool {   // all lanes; lane 0 polls
      bool ok = true;
      if (lane == 0) ok = ptx::mbar_wait(&empty[j % C::kStages], static_cast<uint32_t>((j / C::kStages) & 1));
      return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    };
    int issued = pw;                           // next local tile of this producer
    bool aborted = false;
    for (; issued < my_tiles; issued += 2) {
      if (__any_sync(0xffffffffu, *s_abort != 0u)) { aborted = true; break; }
      const int j = issued;
      if (j >= C::kStages && !wait_released(j - C::kStages)) {
        if (lane == 0) fail();
        aborted = true;
        break;
      }
      if (j == kHoldTile || (C::kHoldStages == 2 && j == kHoldTile - 1)) {   // prologue data still there
        bool ok = true;
        if (lane == 0) ok = ptx::mbar_wait(pro_done, 0);
        if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) {
          if (lane == 0) fail();
          aborted = true;
          break;
        }
      }
      if constexpr (kSplit) {                  // every tile, one row per lane
        if (j >= kEarly) {
          const TileLoc L = tile_at(j);
          const int st = j % C::kStages;
          if (lane == 0) {
            s_rows[st] = L.rows;
            ptx::mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(L.rows * C::kRowBytes));
          }
          __syncwarp();
          issue_tile(L, st, policy, lane, 32, kKLoop ? j / kl_tiles : chunk);
        }
      } else if (lane == 0 && j >= C::kEarlyTiles) {   // the first ones went out with the barrier set-up
        const TileLoc L = tile_at(j);
        const uint32_t bytes = static_cast<uint32_t>(L.rows * C::kRowBytes);
        const int st = j % C::kStages;
        s_rows[st] = L.rows;
        ptx::mbar_arrive_expect_tx(&full[st], bytes);
        ptx::bulk_g2s(stages + st * C::kStageBytes, segs.seg[L.s].w + L.r0 * C::kRowBytes, bytes, &full[st],
                      policy);
      }
      if (j >= C::kStages) finish(j - C::kStages);
    }
    // the last tiles this producer armed: wait for their release, finish them
    int first = issued - C::kStages;
    if (first < pw) first = pw;
    for (int j = first; j < issued && !aborted; j += 2) {
      if (__any_sync(0xffffffffu, *s_abort != 0u) || !wait_released(j)) {
        if (lane == 0) fail();
        aborted = true;
        break;
      }
      finish(j);
    }
    if (aborted && lane == 0) {
      // Never leave the CTA with copies in flight: wait (bounded) for the fills
      // of this producer's parity armed last, by it or, before the CTA-wide
      // barrier, by the barrier thread (tiles below min(kEarly, my_tiles)).
      int armed_end = issued;
      const int early = kEarly < my_tiles ? kEarly : my_tiles;
      while (armed_end < early) armed_end += 2;
      for (int j = armed_end - C::kStages > pw ? armed_end - C::kStages : pw; j < armed_end; j += 2)
        ptx::mbar_wait(&full[j % C::kStages], static_cast<uint32_t>((j / C::kStages) & 1));
    }
    for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (lane == 0 && best != 0ull) atomicMax(s_best, best);
    if (lse_parts) {
      ms = ms_warp_combine(ms);
      if (lane == 0) s_ms[pw] = make_float2(ms.m, ms.s);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int stream = tid / C::kUnits;
    const int u = tid % C::kUnits;
    const int kb = u >> 2, c = u & 3;

    // Prologue: the hidden row (and gamma) arrive in the last stage.  Unit u's
    // 64 columns are quantised by its four threads (one per stream), a quarter
    // (16 columns) each: quarter q = (stream + qoff(u mod 4)) mod 4 with qoff =
    // 0, 1, 1, 2, its four 4-column pieces taken in an order rotated by
    // ((u mod 8) / 2 + the lane's quarter-warp) mod 4.  That puts the eight
    // lanes of every quarter-warp on distinct banks for the row's 16-byte
    // loads, and the 32 lanes of a warp on distinct banks for each plane-word
    // store (two ways where a warp spans two streams).  The quantisation step
    // is a power of two fixed by the largest |h * gamma| of the unit, so it
    // needs neither the RMS factor r nor a division: r only scales sigma and
    // the column sums.  Two
    // barriers: after the first every consumer has read the staged row and
    // posted its sum of squares and its quarter's (max, sum); after the second
    // the unit's plane words are in shared memory.
    XPlanes xl, xh;
    float sx_lo, sx_hi, sigma_half;
    bool pro_ok;
    if constexpr (kKLoop) {
      // All chunks at once, each the same way as the one chunk below (a
      // thread's quarters of all units tile the row once, so they also give
      // the row's sum of squares: one RMS factor for all chunks).  Chunk 0's
      // plane words are shared over its own (by then consumed) hidden columns
      // and loaded into registers; the later chunks' plane words, sigma/2 and
      // column sums go to their slots (over the rest of the consumed row) for
      // the main loop.  The gamma quarters are loaded from global memory while
      // the row is copied.
      const int q = (stream + (((u & 3) + 1) >> 1)) & 3;
      const int rot = (((u & 7) >> 1) + ((tid >> 3) & 3)) & 3;
      const int base = kb * kBlockWeights + 64 * c + 16 * q;
      float4 gv[kMaxKLoopChunks][4];
#pragma unroll
      for (int cc = 0; cc < kMaxKLoopChunks; ++cc)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          gv[cc][i] = gamma && cc < n_chunks
                          ? __ldg(reinterpret_cast<const float4 *>(gamma + cc * K + base + 4 * ((i + rot) & 3)))
                          : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
      pro_ok = __all_sync(0xffffffffu, ptx::mbar_wait(pro_full, 0));
      if (!pro_ok && lane == 0) fail();
      float xv[kMaxKLoopChunks][4][4];
      float ss = 0.0f;
#pragma unroll
      for (int cc = 0; cc < kMaxKLoopChunks; ++cc) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int off = cc * K + base + 4 * ((i + rot) & 3);
          float4 h = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (cc < n_chunks) {             // a quarter (64 bytes) never straddles the two parts
            constexpr int kIn = C::kKStageRowBytes / 4;   // columns in the staging stage
            h = *reinterpret_cast<const float4 *>(off < kIn ? s_hidden + off
                                                            : reinterpret_cast<const float *>(s_planes) + (off - kIn));
            if (gamma) {
              const float4 g = gv[cc][i];
              ss = fmaf(h.x, h.x, ss);
              ss = fmaf(h.y, h.y, ss);
              ss = fmaf(h.z, h.z, ss);
              ss = fmaf(h.w, h.w, ss);
              h = make_float4(h.x * g.x, h.y * g.y, h.z * g.z, h.w * g.w);
            }
          }
          xv[cc][i][0] = h.x; xv[cc][i][1] = h.y; xv[cc][i][2] = h.z; xv[cc][i][3] = h.w;
        }
        if (cc < n_chunks) {
          float amax = 0.0f, psum = 0.0f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            psum += (xv[cc][i][0] + xv[cc][i][1]) + (xv[cc][i][2] + xv[cc][i][3]);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(xv[cc][i][0]), fabsf(xv[cc][i][1])),
                                     fmaxf(fabsf(xv[cc][i][2]), fabsf(xv[cc][i][3]))));
          }
          float2 *ex = cc == 0 ? s_ex : reinterpret_cast<float2 *>(slots) + (cc - 1) * C::kUnits * 4;
          ex[u * 4 + q] = make_float2(amax, psum);
        }
      }
      if (gamma) {
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s_red[warp] = ss;
      }
      ptx::named_bar_sync(1, C::kConsumers);
      float r = 1.0f;
      if (gamma) {                              // the warps' sums in warp order
        float tot = 0.0f;
        for (int i = 0; i < C::kConsumerWarps; ++i) tot += s_red[i];
        r = rsqrtf(fmaf(tot, 1.0f / static_cast<float>(K * n_chunks), eps));
      }
#pragma unroll
      for (int cc = 0; cc < kMaxKLoopChunks; ++cc) {
        if (cc >= n_chunks) break;
        const float2 *ex = cc == 0 ? s_ex : reinterpret_cast<const float2 *>(slots) + (cc - 1) * C::kUnits * 4;
        const float4 e01 = *reinterpret_cast<const float4 *>(ex + u * 4);
        const float4 e23 = *reinterpret_cast<const float4 *>(ex + u * 4 + 2);
        const float umax = fmaxf(fmaxf(e01.x, e01.z), fmaxf(e23.x, e23.z));
        const float slo = r * (e01.y + e01.w), shi = r * (e23.y + e23.w);
        float inv = 0.0f, sh = 0.0f;
        if (umax > 0.0f) {
          const int eb = pow2_step_exponent(umax);
          inv = __uint_as_float(static_cast<uint32_t>(eb) << 23);
          sh = r * __uint_as_float(static_cast<uint32_t>(253 - eb) << 23);
        }
        uint32_t *s_pl = cc == 0 ? reinterpret_cast<uint32_t *>(const_cast<float *>(s_hidden)) + u * C::kKPlaneStride
                                 : s_planes + ((cc - 1) * C::kUnits + u) * C::kKPlaneStride;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t w2, w1, w0;
          quantize_chunk(xv[cc][i], inv, w2, w1, w0);
          const int ch = 4 * q + ((i + rot) & 3);
          s_pl[ch] = w2;
          s_pl[16 + ch] = w1;
          s_pl[32 + ch] = w0;
        }
        if (cc == 0) {
          sx_lo = slo;
          sx_hi = shi;
          sigma_half = sh;
        } else if (stream == 0) {
          s_pl[48] = __float_as_uint(sh);
          s_pl[49] = __float_as_uint(slo);
          s_pl[50] = __float_as_uint(shi);
        }
      }
      ptx::named_bar_sync(1, C::kConsumers);
      const uint32_t *s_pl = reinterpret_cast<const uint32_t *>(s_hidden) + u * C::kKPlaneStride;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint4 a2 = *reinterpret_cast<const uint4 *>(s_pl + 4 * m);
        const uint4 a1 = *reinterpret_cast<const uint4 *>(s_pl + 16 + 4 * m);
        const uint4 a0 = *reinterpret_cast<const uint4 *>(s_pl + 32 + 4 * m);
        const uint4 b2 = *reinterpret_cast<const uint4 *>(s_pl + 8 + 4 * m);
        const uint4 b1 = *reinterpret_cast<const uint4 *>(s_pl + 24 + 4 * m);
        const uint4 b0 = *reinterpret_cast<const uint4 *>(s_pl + 40 + 4 * m);
        xl.p2[4 * m] = a2.x; xl.p2[4 * m + 1] = a2.y; xl.p2[4 * m + 2] = a2.z; xl.p2[4 * m + 3] = a2.w;
        xl.p1[4 * m] = a1.x; xl.p1[4 * m + 1] = a1.y; xl.p1[4 * m + 2] = a1.z; xl.p1[4 * m + 3] = a1.w;
        xl.p0[4 * m] = a0.x; xl.p0[4 * m + 1] = a0.y; xl.p0[4 * m + 2] = a0.z; xl.p0[4 * m + 3] = a0.w;
        xh.p2[4 * m] = b2.x; xh.p2[4 * m + 1] = b2.y; xh.p2[4 * m + 2] = b2.z; xh.p2[4 * m + 3] = b2.w;
        xh.p1[4 * m] = b1.x; xh.p1[4 * m + 1] = b1.y; xh.p1[4 * m + 2] = b1.z; xh.p1[4 * m + 3] = b1.w;
        xh.p0[4 * m] = b0.x; xh.p0[4 * m + 1] = b0.y; xh.p0[4 * m + 2] = b0.z; xh.p0[4 * m + 3] = b0.w;
      }
      uint32_t dep = (xl.p2[0] ^ xl.p2[4]) ^ (xl.p1[0] ^ xl.p1[4]) ^ (xl.p0[0] ^ xl.p0[4]) ^
                     (xh.p2[0] ^ xh.p2[4]) ^ (xh.p1[0] ^ xh.p1[4]) ^ (xh.p0[0] ^ xh.p0[4]);
      asm volatile("mov.b32 %0, %0;" : "+r"(dep));
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(pro_done);
    } else {
    pro_ok = __all_sync(0xffffffffu, ptx::mbar_wait(pro_full, 0));
    if (!pro_ok && lane == 0) fail();
    {
      const int q = (stream + (((u & 3) + 1) >> 1)) & 3;
      const int rot = (((u & 7) >> 1) + ((tid >> 3) & 3)) & 3;
      const int base = kb * kBlockWeights + 64 * c + 16 * q;
      float xv[4][4];
      float amax = 0.0f, psum = 0.0f, ss = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int off = base + 4 * ((i + rot) & 3);
        float4 h = *reinterpret_cast<const float4 *>(s_hidden + off);
        if (gamma) {
          if constexpr (!kSplit) {              // the quarters of all threads tile the row once
            ss = fmaf(h.x, h.x, ss);
            ss = fmaf(h.y, h.y, ss);
            ss = fmaf(h.z, h.z, ss);
            ss = fmaf(h.w, h.w, ss);
          }
          const float4 g = *reinterpret_cast<const float4 *>(s_gamma + off);
          h = make_float4(h.x * g.x, h.y * g.y, h.z * g.z, h.w * g.w);
        }
        xv[i][0] = h.x; xv[i][1] = h.y; xv[i][2] = h.z; xv[i][3] = h.w;
        psum += (h.x + h.y) + (h.z + h.w);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w))));
      }
      if constexpr (kSplit) {                   // the whole row's mean square (all chunks), from global memory
        if (gamma) {
          const int kt = K * n_chunks;
          for (int j = tid * 4; j < kt; j += C::kConsumers * 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(hidden + j));
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
          }
        }
      }
      if (gamma) {
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s_red[warp] = ss;
      }
      s_ex[u * 4 + q] = make_float2(amax, psum);
      ptx::named_bar_sync(1, C::kConsumers);
      // Final RMSNorm factor r = 1 / sqrt(mean(h^2) + eps), the warps' sums
      // added in warp order (every CTA the same bits).
      float r = 1.0f;
      if (gamma) {
        float tot = 0.0f;
        for (int i = 0; i < C::kConsumerWarps; ++i) tot += s_red[i];
        r = rsqrtf(fmaf(tot, 1.0f / static_cast<float>(kSplit ? K * n_chunks : K), eps));
      }
      const float4 e01 = *reinterpret_cast<const float4 *>(s_ex + u * 4);
      const float4 e23 = *reinterpret_cast<const float4 *>(s_ex + u * 4 + 2);
      const float umax = fmaxf(fmaxf(e01.x, e01.z), fmaxf(e23.x, e23.z));
      sx_lo = r * (e01.y + e01.w);             // quarters 0 and 1
      sx_hi = r * (e23.y + e23.w);             // quarters 2 and 3
      float inv = 0.0f;
      sigma_half = 0.0f;
      if (umax > 0.0f) {
        const int eb = pow2_step_exponent(umax);
        inv = __uint_as_float(static_cast<uint32_t>(eb) << 23);
        sigma_half = r * __uint_as_float(static_cast<uint32_t>(253 - eb) << 23);   // the 1/2 undoes the 2q form
      }
      uint32_t *s_pl = reinterpret_cast<uint32_t *>(stages + (C::kStages - 1) * C::kStageBytes) + u * C::kPlaneStride;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t w2, w1, w0;
        quantize_chunk(xv[i], inv, w2, w1, w0);
        const int ch = 4 * q + ((i + rot) & 3);           // natural chunk
        s_pl[ch] = w2;
        s_pl[16 + ch] = w1;
        s_pl[32 + ch] = w0;
      }
      ptx::named_bar_sync(1, C::kConsumers);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint4 a2 = *reinterpret_cast<const uint4 *>(s_pl + 4 * m);
        const uint4 a1 = *reinterpret_cast<const uint4 *>(s_pl + 16 + 4 * m);
        const uint4 a0 = *reinterpret_cast<const uint4 *>(s_pl + 32 + 4 * m);
        const uint4 b2 = *reinterpret_cast<const uint4 *>(s_pl + 8 + 4 * m);
        const uint4 b1 = *reinterpret_cast<const uint4 *>(s_pl + 24 + 4 * m);
        const uint4 b0 = *reinterpret_cast<const uint4 *>(s_pl + 40 + 4 * m);
        xl.p2[4 * m] = a2.x; xl.p2[4 * m + 1] = a2.y; xl.p2[4 * m + 2] = a2.z; xl.p2[4 * m + 3] = a2.w;
        xl.p1[4 * m] = a1.x; xl.p1[4 * m + 1] = a1.y; xl.p1[4 * m + 2] = a1.z; xl.p1[4 * m + 3] = a1.w;
        xl.p0[4 * m] = a0.x; xl.p0[4 * m + 1] = a0.y; xl.p0[4 * m + 2] = a0.z; xl.p0[4 * m + 3] = a0.w;
        xh.p2[4 * m] = b2.x; xh.p2[4 * m + 1] = b2.y; xh.p2[4 * m + 2] = b2.z; xh.p2[4 * m + 3] = b2.w;
        xh.p1[4 * m] = b1.x; xh.p1[4 * m + 1] = b1.y; xh.p1[4 * m + 2] = b1.z; xh.p1[4 * m + 3] = b1.w;
        xh.p0[4 * m] = b0.x; xh.p0[4 * m + 1] = b0.y; xh.p0[4 * m + 2] = b0.z; xh.p0[4 * m + 3] = b0.w;
      }
      // release the staging stage once every word loaded from it is in a
      // register: the move below consumes one word of each load, so it (and
      // the arrive after it) waits for all of them
      uint32_t dep = (xl.p2[0] ^ xl.p2[4]) ^ (xl.p1[0] ^ xl.p1[4]) ^ (xl.p0[0] ^ xl.p0[4]) ^
                     (xh.p2[0] ^ xh.p2[4]) ^ (xh.p1[0] ^ xh.p1[4]) ^ (xh.p0[0] ^ xh.p0[4]);
      asm volatile("mov.b32 %0, %0;" : "+r"(dep));
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(pro_done);
    }
    }
    const UnitSel us = make_unit_sel<kQ4>(c);

    int st = 0, ps = 0;
    uint32_t ph = 0;                           // round parity of the stage ring
    int in_chunk = 0, kchunk = 0;              // K loop: tiles done of the current chunk
    for (int j = 0; j < my_tiles && pro_ok; ++j) {
      // every exit decision is taken by the whole warp (the loop body shuffles)
      if (__any_sync(0xffffffffu, *s_abort != 0u)) break;
      if constexpr (kKLoop) {
        if (in_chunk == kl_tiles) {            // the next chunk's activations
          in_chunk = 0;
          ++kchunk;
          const uint32_t *s_pl = s_planes + ((kchunk - 1) * C::kUnits + u) * C::kKPlaneStride;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const uint4 a2 = *reinterpret_cast<const uint4 *>(s_pl + 4 * m);
            const uint4 a1 = *reinterpret_cast<const uint4 *>(s_pl + 16 + 4 * m);
            const uint4 a0 = *reinterpret_cast<const uint4 *>(s_pl + 32 + 4 * m);
            const uint4 b2 = *reinterpret_cast<const uint4 *>(s_pl + 8 + 4 * m);
            const uint4 b1 = *reinterpret_cast<const uint4 *>(s_pl + 24 + 4 * m);
            const uint4 b0 = *reinterpret_cast<const uint4 *>(s_pl + 40 + 4 * m);
            xl.p2[4 * m] = a2.x; xl.p2[4 * m + 1] = a2.y; xl.p2[4 * m + 2] = a2.z; xl.p2[4 * m + 3] = a2.w;
            xl.p1[4 * m] = a1.x; xl.p1[4 * m + 1] = a1.y; xl.p1[4 * m + 2] = a1.z; xl.p1[4 * m + 3] = a1.w;
            xl.p0[4 * m] = a0.x; xl.p0[4 * m + 1] = a0.y; xl.p0[4 * m + 2] = a0.z; xl.p0[4 * m + 3] = a0.w;
            xh.p2[4 * m] = b2.x; xh.p2[4 * m + 1] = b2.y; xh.p2[4 * m + 2] = b2.z; xh.p2[4 * m + 3] = b2.w;
            xh.p1[4 * m] = b1.x; xh.p1[4 * m + 1] = b1.y; xh.p1[4 * m + 2] = b1.z; xh.p1[4 * m + 3] = b1.w;
            xh.p0[4 * m] = b0.x; xh.p0[4 * m + 1] = b0.y; xh.p0[4 * m + 2] = b0.z; xh.p0[4 * m + 3] = b0.w;
          }
          const uint4 ex = *reinterpret_cast<const uint4 *>(s_pl + 48);
          sigma_half = __uint_as_float(ex.x);
          sx_lo = __uint_as_float(ex.y);
          sx_hi = __uint_as_float(ex.z);
        }
        ++in_chunk;
      }
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&full[st], ph))) {
        if (lane == 0) fail();
        break;
      }
      const int rows = s_rows[st];
      float *slot = slots + ps * (C::kSlotBytes / 4) + kb;
      const uint8_t *sbase = stages + st * C::kStageBytes + kb * C::kBB;
      float pv[kRows / kStreams];
      if (rows == kRows) {
#pragma unroll
        for (int rr = 0; rr < kRows / kStreams; ++rr)
          pv[rr] = unit_partial<kQ4>(sbase + (stream + rr * kStreams) * C::kRowBytes, us, xl, xh, sx_lo, sx_hi,
                                sigma_half);
      } else {
#pragma unroll
        for (int rr = 0; rr < kRows / kStreams; ++rr) {
          const int rl = stream + rr * kStreams;
          pv[rr] = rl < rows ? unit_partial<kQ4>(sbase + rl * C::kRowBytes, us, xl, xh, sx_lo, sx_hi, sigma_half)
                             : 0.0f;
        }
      }
#pragma unroll
      for (int rr = 0; rr < kRows / kStreams; ++rr) {
        float v = pv[rr];
        v += __shfl_xor_sync(0xffffffffu, v, 1);   // the four units of block kb
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (c == 0) slot[(stream + rr * kStreams) * NB] = v;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[st]);
      if (++st == C::kStages) { st = 0; ph ^= 1u; }
      if (++ps == C::kSlots) ps = 0;
    }
  }

  __syncthreads();
  if constexpr (kSplit && !kKLoop) {
    // Count this CTA's tiles in, a thread per tile; the tiles it arrived last on
    // are finished by the whole CTA, a (tile, row) job per thread: the chunk
    // partials added in chunk order, then scale, cap, store and argmax key.
    if (*s_abort == 0u) {
      int *s_list = reinterpret_cast<int *>(stages);                 // every stage is free again
      unsigned int *s_nlast = reinterpret_cast<unsigned int *>(s_red);
      const GemvSegment &G = segs.seg[0];
      unsigned long long best = 0ull;
      for (int base = 0; base < my_tiles; base += C::kThreads) {
        if (tid == 0) *s_nlast = 0u;
        __syncthreads();
        const int j = base + tid;
        if (j < my_tiles) {
          const int64_t tile = tile_first + static_cast<int64_t>(j) * tile_step;
          ptx::fence_acq_rel_gpu();            // release: the CTA's partial stores (seen through the barrier)
          if (atomicAdd(split_cnt + tile, 1u) == static_cast<uint32_t>(n_chunks - 1)) {
            split_cnt[tile] = 0u;              // every chunk counted in: re-armed for the next launch
            ptx::fence_acq_rel_gpu();          // acquire: the other chunks' partials, for the CTA after the barrier
            s_list[atomicAdd(s_nlast, 1u)] = j;
          }
        }
        __syncthreads();
        const int n_jobs = static_cast<int>(*s_nlast) * kRows;
        for (int job0 = tid; job0 < n_jobs; job0 += 4 * C::kThreads) {
          float acc[4];
          int64_t row[4];
          bool ok[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int job = job0 + i * C::kThreads;
            ok[i] = job < n_jobs;
            const TileLoc L = locate<kGroup>(segs, tile_first + static_cast<int64_t>(ok[i] ? s_list[job / kRows] : 0) * tile_step);
            ok[i] = ok[i] && job % kRows < L.rows;
            row[i] = L.r0 + job % kRows;
            acc[i] = 0.0f;
          }
          for (int q = 0; q < n_chunks; ++q) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (ok[i]) acc[i] += __ldcg(split_part + static_cast<int64_t>(q) * G.n_rows + row[i]);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (ok[i]) {
              const float out = scale_softcap(acc[i], G.scale, G.cap);
              G.out[row[i]] = out;
              best = umax64(best, argmax_key(segs.argmax_precap ? acc[i] * G.scale : out,
                                             static_cast<uint32_t>(row[i])));
            }
          }
        }
        __syncthreads();                        // s_list and s_nlast are rewritten next round
      }
      for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
      if (lane == 0 && best != 0ull) atomicMax(s_best, best);
    }
    __syncthreads();
  }
  if (lse_parts && tid == 0) {                  // this CTA's pair, in a fixed order
    const MaxSum c = ms_combine({s_ms[0].x, s_ms[0].y}, {s_ms[1].x, s_ms[1].y});
    lse_parts[blockIdx.x] = make_float2(c.m, c.s);
  }
  if (argmax) argmax_publish_finish(keys, ticket, argmax, s_best, 1);
}

template <int NB, bool kGroup, bool kQ4, bool kSplit = false, bool kKLoop = false>
cudaError_t launch_b1_nb(const float *hidden, const float *gamma, float eps, const SegTable &T,
                         unsigned long long *keys, unsigned int *ticket, int32_t *argmax, uint32_t *status,
                         float2 *lse_parts, int num_sms, cudaStream_t stream, int n_chunks = 1,
                         float *split_part = nullptr, unsigned int *split_cnt = nullptr) {
  using C = B1Cfg<NB, kQ4, kKLoop>;
  static std::atomic<unsigned long long> configured{0};   // one bit per device: the attribute is per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemv_b1_kernel<NB, kGroup, kQ4, kSplit, kKLoop>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int64_t n_tiles = T.tile_end[T.n - 1];
  // split along K: n_chunks row tiles per tile of rows, at least one CTA per chunk
  const int64_t units = n_tiles * n_chunks;
  const int64_t grid = kSplit && !kKLoop ? (units < num_sms ? units : num_sms) : T.grid;
  if (kKLoop) {   // balanced shares of at most kMaxKLoopTiles tiles, every chunk in every CTA
    const int share = T.rows_per + (T.extra ? 1 : 0);
    if (n_chunks < 2 || n_chunks > kMaxKLoopChunks || !T.balanced || share > kMaxKLoopTiles * kRows)
      return cudaErrorInvalidValue;
  } else if (kSplit && (n_chunks < 2 || grid < n_chunks || !split_part || !split_cnt)) {
    return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_b1_kernel<NB, kGroup, kQ4, kSplit, kKLoop>, hidden, gamma, eps, T, keys,
                            ticket, argmax, status, lse_parts, n_chunks, split_part, split_cnt);
}

// The matrices' tile table and how the CTAs share the tiles.  Round-robin
// kRows-row tiles stream the whole GPU through one contiguous stretch of the
// weights, the right order for large matrices.  A small launch is a chain of
// latencies in which the CTA with the most work sets the time: for a single
// matrix an even share of rows per CTA (balanced mode) is taken when it lowers
// the most row rounds any CTA runs (a round = one row per consumer stream; a
// share of m rows takes ceil(m / 4) rounds) and a share is at most
// kMaxBalancedRows rows.
constexpr int64_t kMaxBalancedRows = 12 * kRows;

SegTable make_table(const GemvSegment *segs, int n, int num_sms, bool allow_balanced) {
  SegTable T = {};
  int64_t end = 0, rows = 0;
  for (int i = 0; i < n; ++i) {
    T.seg[i] = segs[i];
    end += (segs[i].n_rows + kRows - 1) / kRows;
    T.tile_end[i] = end;
    rows += segs[i].n_rows;
  }
  T.n = n;
  T.grid = static_cast<int>(end < num_sms ? end : num_sms);
  if (allow_balanced && n == 1 && rows > 0 && num_sms > 0) {
    const int64_t rr_rounds = (end + num_sms - 1) / num_sms * (kRows / kStreams);
    const int64_t grid = rows < num_sms ? rows : num_sms;
    const int64_t share = (rows + grid - 1) / grid;
    const int64_t rounds = (share + kStreams - 1) / kStreams;
    if (share <= kMaxBalancedRows && rounds < rr_rounds) {
      T.balanced = 1;
      T.grid = static_cast<int>(grid);
      T.rows_per = static_cast<int>(rows / grid);
      T.extra = static_cast<int>(rows % grid);
    }
  }
  return T;
}

}  // namespace

bool b1_supported(int k) { return k == 26 * kBlockWeights || k == 16 * kBlockWeights; }

// Chunk width (26 or 16 blocks) and count of a split-K batch-1 launch.
static void split_shape(int k, int &chunk_nb, int &chunks) {
  const int nb = k / kBlockWeights;
  chunk_nb = nb % 26 == 0 ? 26 : nb % 16 == 0 ? 16 : 0;
  chunks = chunk_nb ? nb / chunk_nb : 0;
}

int b1_split_chunks(int k) {
  int cnb, s;
  split_shape(k, cnb, s);
  return k % kBlockWeights == 0 && s >= 2 && s <= kMaxSplitChunks ? s : 0;
}

size_t b1_split_floats(int64_t n_rows, int k) { return static_cast<size_t>(n_rows) * b1_split_chunks(k); }

size_t b1_split_counters(int64_t n_rows) { return static_cast<size_t>((n_rows + kRows - 1) / kRows); }

cudaError_t launch_b1_split(const LaunchArgs &a) {
  int cnb, s;
  split_shape(a.k, cnb, s);
  if (b1_split_chunks(a.k) == 0 || a.num_sms < s) return cudaErrorInvalidValue;
  const GemvSegment one = {a.w, a.logits, a.n_rows, a.scale, a.cap};
  // no (max, sum exp) pairs: which CTA finishes a row varies from run to run,
  // so the logprobs take the separate pass over the logits (fixed order)
  float2 *parts = nullptr;
  // A Q4_K matrix of up to kMaxKLoopChunks chunks whose rows, shared evenly
  // over the SMs, give every CTA at most kMaxKLoopTiles tiles: each CTA runs
  // all chunks of its own rows (no partials through global memory).
  const int64_t kl_grid = a.n_rows < a.num_sms ? a.n_rows : a.num_sms;
  if (a.q4 && s <= kMaxKLoopChunks && a.n_rows > 0 &&
      (a.n_rows + kl_grid - 1) / kl_grid <= static_cast<int64_t>(kMaxKLoopTiles) * kRows) {
    SegTable T = make_table(&one, 1, a.num_sms, false);
    T.balanced = 1;
    T.grid = static_cast<int>(kl_grid);
    T.rows_per = static_cast<int>(a.n_rows / kl_grid);
    T.extra = static_cast<int>(a.n_rows % kl_grid);
    T.argmax_precap = a.argmax_precap ? 1 : 0;
    if (cnb == 26)
      return launch_b1_nb<26, false, true, true, true>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket, a.argmax,
                                                       a.ws.status, parts, a.num_sms, a.stream, s);
    return launch_b1_nb<16, false, true, true, true>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket, a.argmax,
                                                     a.ws.status, parts, a.num_sms, a.stream, s);
  }
  SegTable T = make_table(&one, 1, a.num_sms, false);
  T.argmax_precap = a.argmax_precap ? 1 : 0;
  float *part = a.ws.b1_part;
  unsigned int *cnt = a.ws.b1_cnt;
  if (cnb == 26)
    return a.q4 ? launch_b1_nb<26, false, true, true>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket, a.argmax,
                                                      a.ws.status, parts, a.num_sms, a.stream, s, part, cnt)
                : launch_b1_nb<26, false, false, true>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket,
                                                       a.argmax, a.ws.status, parts, a.num_sms, a.stream, s, part,
                                                       cnt);
  return a.q4 ? launch_b1_nb<16, false, true, true>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket, a.argmax,
                                                    a.ws.status, parts, a.num_sms, a.stream, s, part, cnt)
              : launch_b1_nb<16, false, false, true>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket, a.argmax,
                                                     a.ws.status, parts, a.num_sms, a.stream, s, part, cnt);
}

int b1_grid(int64_t n_rows, int num_sms) {
  const GemvSegment one = {nullptr, nullptr, n_rows, 1.0f, 0.0f};
  return make_table(&one, 1, num_sms, true).grid;
}

cudaError_t launch_b1(const LaunchArgs &a) {
  const GemvSegment one = {a.w, a.logits, a.n_rows, a.scale, a.cap};
  SegTable T = make_table(&one, 1, a.num_sms, true);
  T.argmax_precap = a.argmax_precap ? 1 : 0;
  float2 *parts = a.lse_parts ? a.ws.lse_parts : nullptr;   // batch row 0: one pair per CTA
  const int nb = a.k / kBlockWeights;
  if (a.q4) {
    if (nb == 26) return launch_b1_nb<26, false, true>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket,
                                                       a.argmax, a.ws.status, parts, a.num_sms, a.stream);
    if (nb == 16) return launch_b1_nb<16, false, true>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket,
                                                       a.argmax, a.ws.status, parts, a.num_sms, a.stream);
    return cudaErrorInvalidValue;
  }
  switch (nb) {
    case 26: return launch_b1_nb<26, false, false>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket, a.argmax,
                                                   a.ws.status, parts, a.num_sms, a.stream);
    case 16: return launch_b1_nb<16, false, false>(a.hidden, a.gamma, a.eps, T, a.ws.keys, a.ws.ticket, a.argmax,
                                                   a.ws.status, parts, a.num_sms, a.stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_b1_group(const float *hidden, const float *gamma, float eps, int k, const GemvSegment *segs,
                            int n, uint32_t *status, int num_sms, cudaStream_t stream, bool q4) {
  if (n < 1 || n > kMaxSegments) return cudaErrorInvalidValue;
  const SegTable T = make_table(segs, n, num_sms, true);
  if (q4) {
    switch (k / kBlockWeights) {
      case 26: return launch_b1_nb<26, true, true>(hidden, gamma, eps, T, nullptr, nullptr, nullptr, status,
                                                   nullptr, num_sms, stream);
      case 16: return launch_b1_nb<16, true, true>(hidden, gamma, eps, T, nullptr, nullptr, nullptr, status,
                                                   nullptr, num_sms, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (k / kBlockWeights) {
    case 26: return launch_b1_nb<26, true, false>(hidden, gamma, eps, T, nullptr, nullptr, nullptr, status,
                                                  nullptr, num_sms, stream);
    case 16: return launch_b1_nb<16, true, false>(hidden, gamma, eps, T, nullptr, nullptr, nullptr, status,
                                                  nullptr, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace muse
