// Internal interface between the C-ABI layer (muse_lmhead.cu) and the kernel
// translation units.  Not installed, not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace muse {

// Device status word bits (the handle's workspace; read back by
// muse_lmhead_device_status).
constexpr uint32_t kStatusWaitTimeout = 1u << 0;   // a bounded mbarrier wait gave up

struct Workspace {
  unsigned long long *keys;  // [max_batch] packed argmax keys, zero between forwards
  unsigned int *ticket;      // CTA completion counter for the argmax, zero between forwards
  uint32_t *status;          // sticky device status bits
  float *x;                  // [max_batch][k] normalised input (generic path)
  uint8_t *xpkg;             // per-block activation packages (tensor-core path)
  float2 *lse_parts;         // [MUSE_MAX_BATCH][kMaxLseParts] (max, sum exp) partials of the logprobs
  float *split_part;         // tensor-core path: [num_sms][2][128][slots] partial sums of shared tiles
  unsigned int *split_cnt;   // [num_sms][8] arrivals per shared tile and warp (per CTA boundary, or per tile when tiles < SMs), zero between forwards
  float *b1_part;            // split-K batch-1 path: [chunks][n_rows] chunk partial sums
  unsigned int *b1_cnt;      // split-K batch-1 path: [12-row tiles] chunk arrivals, zero between forwards
};

constexpr int kMaxLseParts = 256;

struct LaunchArgs {
  const float *hidden;   // [batch][k]
  const float *gamma;    // [k] or nullptr
  float eps;
  const uint8_t *w;      // [n_rows][k/256][176]
  float scale, cap;
  float *logits;         // [batch][n_rows]
  int32_t *argmax;       // [batch] or nullptr
  int batch;
  int64_t n_rows;
  int k;
  int num_sms;
  Workspace ws;
  cudaStream_t stream;
  bool lse_parts = false;    // batch-1 kernel: also write each CTA's (max, sum exp) pair
  bool q4 = false;           // weights are Q4_K (144-byte blocks) instead of Q5_K
  bool argmax_precap = false;  // argmax key: raw * scale (before the cap) instead of the returned logit
};

// One matrix of a grouped batch-1 launch: Q5_K rows `w` ([n_rows][k/256][176]),
// output `out` ([n_rows] f32), out = cap > 0 ? cap*tanh(raw*scale/cap) : raw*scale.
struct GemvSegment {
  const uint8_t *w;
  float *out;
  int64_t n_rows;
  float scale, cap;
};
constexpr int kMaxSegments = 4;

// Each returns cudaSuccess or the launch error.
cudaError_t launch_generic(const LaunchArgs &a);     // RMSNorm pre-pass (if gamma) + generic GEMV
bool b1_supported(int k);                            // fast batch-1 kernel compiled for this K
cudaError_t launch_b1(const LaunchArgs &a);          // fused batch-1 kernel
// Up to kMaxSegments matrices against one normed input row, one launch (K as for b1_supported).
cudaError_t launch_b1_group(const float *hidden, const float *gamma, float eps, int k, const GemvSegment *segs,
                            int n, uint32_t *status, int num_sms, cudaStream_t stream, bool q4 = false);

int generic_launches(const LaunchArgs &a);

// Logprobs over finished logits [batch][n_rows] (in place): partial (max, sum
// exp) pairs per chunk of each row, then logits -= lse (a programmatic
// dependent launch of whatever wrote the logits and pairs).
int lse_parts_for(int64_t n_rows);         // chunks per row used by launch_lse_parts
cudaError_t launch_lse_parts(const float *logits, int batch, int64_t n_rows, float2 *parts, cudaStream_t stream);
cudaError_t launch_logprob_apply(float *logits, int batch, int64_t n_rows, const float2 *parts, int n_parts,
                                 float *lse, cudaStream_t stream);
int b1_grid(int64_t n_rows, int num_sms);   // CTAs of the batch-1 kernel = its (max, sum exp) pairs

// Batch 1 at a K of S (2..kMaxSplitChunks) chunks of a built width (6,656 or
// 4,096 columns): the batch-1 kernel split along K (one chunk per CTA, chunk
// partial sums combined by the last CTA of each row tile).
constexpr int kMaxSplitChunks = 16;
int b1_split_chunks(int k);                          // S, or 0 when K does not split so
size_t b1_split_floats(int64_t n_rows, int k);       // b1_part size
size_t b1_split_counters(int64_t n_rows);            // b1_cnt size
cudaError_t launch_b1_split(const LaunchArgs &a);

// One-thread kernel whose bounded wait on a never-completed mbarrier gives up
// and sets kStatusWaitTimeout in *status.
cudaError_t launch_wait_timeout_selftest(uint32_t *status, cudaStream_t stream);

// Tensor-core path (batches 2..32): activation-package prep + tcgen05 kernel.
bool tc_supported(int batch, int k);
size_t tc_workspace_bytes(int k);
int tc_batch_slots(int batch);                       // the kernel's batch slots (8, 16 or 32)
size_t tc_split_floats(int num_sms, int max_batch);  // split_part size
size_t tc_split_counters(int num_sms);                // split_cnt size
cudaError_t tc_encode_weights(CUtensorMap *map, const void *weights, int64_t n_rows, int k, bool q4);
cudaError_t launch_tc(const LaunchArgs &a, const CUtensorMap &map);

}  // namespace muse
