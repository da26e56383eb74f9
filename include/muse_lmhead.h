/*
 * muse_lmhead — decode-time output stage of the 52-layer Muse Glimmer model on
 * one GB300 (sm_103a): final RMSNorm -> Q5_K LM-head matvec -> logit scale ->
 * soft cap -> optional greedy argmax, as one asynchronous call.
 *
 * What the operation is ("Chapter 20 — Final norm, LM head, and the soft cap",
 * §20.1; the order scale-then-cap is also fixed by "Chapter 9 — The Muse
 * Glimmer architecture", §9.10), for every batch row b and weight row i:
 *
 *     r_b      = 1 / sqrt( sum_j hidden[b][j]^2 / k + eps )        (final norm)
 *     x[b][j]  = hidden[b][j] * r_b * gamma[j]
 *     raw[b][i]= sum_j W[i][j] * x[b][j]                            (LM head)
 *     v        = raw[b][i] * scale                                   (logit_scale)
 *     logits[b][i] = cap > 0 ? cap * tanh(v / cap) : v               (soft cap)
 *     argmax[b]    = lowest i with the largest logits[b][i]          (greedy pick)
 *
 * W is [n_rows x k] in Q5_K super-blocks (§20.3: 256 weights per 176 bytes,
 * k/256 blocks per row, rows contiguous): fp16 d, fp16 dmin, 12 bytes of 6-bit
 * sub-block scales/mins, 32 bytes of high bits, 128 bytes of low nibbles, with
 * w = d*sc*q - dmin*m (the ggml block_q5_K layout).
 *
 * Conventions for every call:
 *   - Device pointers are global-memory addresses on the handle's device.  The
 *     caller owns every input and output buffer; the library never frees them.
 *   - Layouts are dense row-major: hidden [batch][k] f32, gamma [k] f32,
 *     weights [n_rows][k/256][176] bytes, logits [batch][n_rows] f32,
 *     argmax [batch] int32.
 *   - hidden, gamma, weights and logits must be 16-byte aligned; argmax 4-byte.
 *   - Every call validates its arguments first and fails closed: on any error it
 *     returns a negative status and launches nothing.  Nothing aborts, traps or
 *     prints.  Asynchronous device faults surface on the caller's next
 *     synchronisation, as usual in CUDA.
 *   - A handle keeps a small device workspace (argmax partial keys, a
 *     completion counter, a status word, and the batched paths' normalised
 *     inputs).  Two forwards that may run at the same time on the GPU must use
 *     two handles.
 */
#ifndef MUSE_LMHEAD_H
#define MUSE_LMHEAD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define MUSE_OK 0
#define MUSE_ERR_NULL (-1)      /* a required pointer is NULL */
#define MUSE_ERR_SHAPE (-2)     /* n_rows < 1, k < 256, k % 256 != 0, or too large */
#define MUSE_ERR_BATCH (-3)     /* batch outside 1..max_batch, or max_batch outside 1..32 */
#define MUSE_ERR_ALIGN (-4)     /* a pointer is not aligned as stated above */
#define MUSE_ERR_VALUE (-5)     /* eps < 0 or not finite, scale or cap not finite */
#define MUSE_ERR_DEVICE (-6)    /* bad device index, or not an sm_103 GPU */
#define MUSE_ERR_CUDA (-7)      /* a CUDA runtime call failed (message via status_string) */
#define MUSE_ERR_NOMEM (-8)     /* workspace or host allocation failed */

/* Largest batch a handle can be created for. */
#define MUSE_MAX_BATCH 32

/* Weight formats (muse_lmhead_init_format). */
#define MUSE_FORMAT_Q5_K 0   /* 176-byte blocks: the LM head's format (Chapter 20 §20.3) */
#define MUSE_FORMAT_Q4_K 1   /* 144-byte blocks: the FFN bulk's format, and the 756.5 MB head alternative of §20.7 */

typedef struct muse_lmhead muse_lmhead;

/*
 * Create a handle for an [n_rows x k] Q5_K weight matrix and batches of up to
 * max_batch rows on CUDA device `device`.  Allocates the handle's device
 * workspace (zeroed) on that device.  *out receives the handle, or NULL on
 * error.  Returns MUSE_OK or a negative status.
 * The shapes of the pages: n_rows = 202,048 (vocabulary), k = 6,656 (hidden
 * width), Chapter 20 §20.3.
 */
int muse_lmhead_init(muse_lmhead **out, int device, int64_t n_rows, int64_t k,
                     int max_batch);

/*
 * The same for a matrix in another weight format: MUSE_FORMAT_Q5_K (what
 * muse_lmhead_init uses) or MUSE_FORMAT_Q4_K, else MUSE_ERR_VALUE.  Q4_K is
 * ggml's block_q4_K: fp16 d, fp16 dmin, the same 12 bytes of packed 6-bit
 * scales and mins, then 128 bytes of nibbles placed as in Q5_K, no high bits
 * (q in 0..15, w = d*sc*q - dmin*m); 144 bytes per 256 weights.  Every forward
 * of the handle reads its weights in this format (weights = n_rows * (k/256) *
 * 144 bytes for Q4_K).  Batch 1 with k = 4,096 or 6,656 runs the fused kernel;
 * batch 1 with k = S x 6,656 or S x 4,096 (S = 2..16, n_rows * S at most 2^26)
 * runs the same kernel split along k into S column chunks (the workspace then
 * holds n_rows * S floats of chunk partial sums and one counter per 12 rows);
 * other batches (and batch 1 at another k) with an even number of blocks per
 * row the tensor-core kernel, other shapes the generic kernel, in either
 * format.  muse_lmhead_forward_group
 * reads the handle's format; muse_lmhead_forward_b1_noalloc reads Q5_K only.
 */
int muse_lmhead_init_format(muse_lmhead **out, int device, int64_t n_rows, int64_t k,
                            int max_batch, int format);

/*
 * One forward on `stream` (a cudaStream_t; NULL = the legacy default stream),
 * asynchronous with respect to the host.
 *   hidden  [batch][k] f32, device.  The residual stream after the last layer.
 *   gamma   [k] f32, device, or NULL to skip the final norm (then x = hidden).
 *   eps     RMSNorm epsilon (1e-5 on the pages); ignored when gamma is NULL.
 *   weights Q5_K blocks, device, n_rows * (k/256) * 176 bytes.
 *   scale   logit scale (0.196116 on the pages).
 *   cap     soft cap (20 on the pages); cap <= 0 turns the cap off.
 *   logits  [batch][n_rows] f32, device, written.
 *   argmax  [batch] int32, device, written; or NULL to skip the argmax.
 * hidden/gamma/weights are only read; logits must not overlap them.
 */
int muse_lmhead_forward(muse_lmhead *h, const float *hidden, int batch,
                        const float *gamma, float eps, const void *weights,
                        float scale, float cap, float *logits, int32_t *argmax,
                        void *stream);

/*
 * The same forward, returning logprobs instead of logits: per batch row b,
 *     lse[b]         = log sum_i exp(logits[b][i])       (log-softmax normaliser)
 *     logprobs[b][i] = logits[b][i] - lse[b]
 * over the logits after scale and cap — the pages take softmax and logprobs
 * over the capped logits ("Chapter 20 — Final norm, LM head, and the soft cap",
 * §20.7).  The logits themselves are logprobs[b][i] + lse[b].
 *   logprobs [batch][n_rows] f32, device, 16-byte aligned, written.
 *   lse      [batch] f32, device, 4-byte aligned, written; or NULL to skip it.
 *   argmax   as for muse_lmhead_forward (the largest logprob's index).
 * Other arguments and validation as for muse_lmhead_forward.  At batch 1 with
 * the fused kernel (k = 4,096 or 6,656) the normaliser is accumulated in the kernel's epilogue and
 * one more small launch subtracts it; other paths add a pass over the logits.
 */
int muse_lmhead_forward_logprobs(muse_lmhead *h, const float *hidden, int batch,
                                 const float *gamma, float eps, const void *weights,
                                 float scale, float cap, float *logprobs, float *lse,
                                 int32_t *argmax, void *stream);

/*
 * The same forward for callers whose activations live in host memory: copies
 * hidden_host to the device, runs the forward, brings the logits (and argmax)
 * back, and waits for `stream` before returning.  gamma and weights are device
 * pointers (they stay resident).  logits_host may be NULL to fetch only the
 * argmax; argmax_host may be NULL to skip it.  An output buffer that is
 * page-locked for this device (cudaHostAlloc, cudaHostRegister) is written by
 * the kernels directly through the device's mapping of host memory, with no
 * copy after the kernels; a pageable one is filled from a device staging
 * buffer by a copy.  The input should be page-locked for full copy bandwidth;
 * pageable memory also works.  The first call allocates the handle's device
 * staging buffers (max_batch rows).
 */
int muse_lmhead_forward_host(muse_lmhead *h, const float *hidden_host, int batch,
                             const float *gamma, float eps, const void *weights,
                             float scale, float cap, float *logits_host,
                             int32_t *argmax_host, void *stream);

/*
 * Number of kernel launches one forward issues for this batch size, with
 * (with_norm != 0) or without the final norm, or a negative status.  Host-only
 * query.
 */
int muse_lmhead_launches_per_forward(const muse_lmhead *h, int batch, int with_norm);

/*
 * Name of the kernel path a forward with this batch size takes ("gemv_b1",
 * "gemv_b1_split", "gemm_tc" or "gemv_generic"), or NULL for an invalid
 * handle/batch.  Host-only query;
 * the string is static.
 */
const char *muse_lmhead_path_name(const muse_lmhead *h, int batch);

/*
 * Read the handle's sticky device status word (synchronous device-to-host copy
 * on the legacy default stream, after all prior work on the device).  Bit 0:
 * a kernel's bounded wait for a pipeline stage gave up (the forward's outputs
 * are then invalid).  0 means no fault has been recorded since init.
 */
int muse_lmhead_device_status(muse_lmhead *h, uint32_t *status_out);

/*
 * Clear the handle's status word (asynchronous memsets on `stream`), for
 * example after a recorded timeout, once the caller has dealt with it.  Also
 * re-arms the tensor-core path's per-boundary arrival counters and the
 * split-K batch-1 path's per-tile chunk counters, which a forward that gave up
 * may have left counted in.
 */
int muse_lmhead_clear_device_status(muse_lmhead *h, void *stream);

/*
 * Self-test of the failure path the pipelined kernels rely on: launches a
 * one-thread kernel on `stream` that waits on an mbarrier nothing ever arrives
 * on.  The wait is bounded like every wait in the library (at most 2^16 polls,
 * each suspended for at most 20 us); it gives up, sets bit 0 of the handle's
 * status word and the kernel returns normally — no trap, no fault, the context
 * stays usable.  Read the result with muse_lmhead_device_status and clear it
 * with muse_lmhead_clear_device_status.  The pages have no counterpart.
 */
int muse_lmhead_selftest_wait_timeout(muse_lmhead *h, void *stream);

/*
 * Batch-1 forward for callers that cannot allocate device memory at call time:
 * runtimes that reserve all device memory up front through their own
 * allocator and refuse any later cudaMalloc, and serving loops that must not
 * risk the implicit device synchronisation of cudaMalloc/cudaFree.  No handle:
 * the few bytes of scratch the fused batch-1 kernel needs (argmax key,
 * completion ticket, status word) live in a fixed 256-byte array inside the
 * library's device memory, which every GPU that loads the library holds until
 * the process exits.  The pages have no counterpart of this call; it is a
 * deployment convenience.
 *   device   CUDA device the pointers live on (made current for the call).
 *   hidden   [k] f32, one row; gamma/eps/weights/scale/cap/logits/argmax as for
 *            muse_lmhead_forward with batch 1 (logits [n_rows], argmax [1]).
 *            Weights are Q5_K.  The argmax always ranks the returned (capped)
 *            logits, MUSE_ARGMAX_CAPPED: there is no handle to select the
 *            pre-cap key on.
 *   n_rows   1 .. 2^31-1;  k: 4,096 or 6,656 only (the fused kernel's widths),
 *            anything else is rejected with MUSE_ERR_SHAPE before any launch.
 * Calls no cudaMalloc/cudaFree and no allocating library routine.  It clears
 * the argmax key and ticket with an asynchronous 12-byte memset on `stream`,
 * then launches the kernel.  The first call on a device performs one-time
 * set-up (looks up the scratch array's device address, sets the kernel's
 * shared-memory limit); make that first call before any stream capture.  All
 * calls on a device share the scratch: calls that may overlap on the GPU race
 * on it and must be ordered by the caller (same stream, or events).
 * A bounded wait that gave up inside the kernel (its outputs are then
 * invalid) sets bit 0 of the scratch's status word, which later calls do not
 * clear: read it with muse_lmhead_noalloc_device_status.
 */
int muse_lmhead_forward_b1_noalloc(int device, const float *hidden,
                                   const float *gamma, float eps,
                                   const void *weights, int64_t n_rows,
                                   int64_t k, float scale, float cap,
                                   float *logits, int32_t *argmax,
                                   void *stream);

/*
 * Status word of the no-alloc forward on `device` (bit 0: a bounded wait in
 * one of the kernels gave up since the last read; 0: every such forward ran to
 * completion).  Waits for the work already queued on `stream` (the stream the
 * forwards ran on), copies the word into *status and clears it; allocates
 * nothing.  Forwards still running on other streams race with the read.
 * The pages have no counterpart.
 */
int muse_lmhead_noalloc_device_status(int device, void *stream, uint32_t *status);

/*
 * One matrix of a grouped forward (muse_lmhead_forward_group).
 *   weights  Q5_K blocks, device, n_rows * (k/256) * 176 bytes, 16-byte aligned.
 *   n_rows   1 .. 2^31-1.
 *   out      [n_rows] f32, device, 4-byte aligned, written:
 *            out[i] = cap > 0 ? cap * tanh(raw[i] * scale / cap) : raw[i] * scale.
 */
typedef struct muse_gemv_segment {
  const void *weights;
  int64_t n_rows;
  float *out;
  float scale;
  float cap;
} muse_gemv_segment;

/* Largest number of matrices in one grouped forward. */
#define MUSE_MAX_SEGMENTS 4

/*
 * Batch-1 forward of up to MUSE_MAX_SEGMENTS weight matrices that share one
 * input row, in one launch: the input is normalised once (the same RMSNorm as
 * muse_lmhead_forward: x = hidden * r * gamma, or x = hidden when gamma is
 * NULL) and every matrix s writes segments[s].out = its matvec with x, scaled
 * and capped with its own scale and cap.  No argmax.  This is the pages'
 * concurrent group of the Q, K, V and attention-gate projections that share
 * the attention block's normed input ("Chapter 9 — The Muse Glimmer
 * architecture", Figure 9.1 and §9.8: Q and gate [6656 -> 4096], K and V
 * [6656 -> 256]).
 *   h         a handle; only its k (4,096 or 6,656, else MUSE_ERR_SHAPE), its
 *             weight format (every segment's weights are in it), its device
 *             and its status word are used.
 *   hidden    [k] f32, device, 16-byte aligned.
 *   gamma     [k] f32, device, 16-byte aligned, or NULL; eps as for forward.
 *   segments  host array of n_segments (1..MUSE_MAX_SEGMENTS) descriptions.
 * Validation fails closed as for muse_lmhead_forward; outputs must not overlap
 * each other or the inputs.  Bit 0 of the handle's status word reports a
 * bounded wait that gave up, as for forward.
 */
int muse_lmhead_forward_group(muse_lmhead *h, const float *hidden, const float *gamma,
                              float eps, const muse_gemv_segment *segments,
                              int n_segments, void *stream);

/*
 * The grouped forward for callers whose input row and outputs live in host
 * memory: copies hidden_host ([k] f32, host, any alignment) to the device,
 * runs muse_lmhead_forward_group, brings every segment's output back, and
 * waits for `stream` before returning.  gamma and each segment's weights are
 * device pointers; each segments[s].out is a HOST buffer of n_rows floats
 * (4-byte aligned).  An output that is page-locked for this device is written
 * by the kernel directly through the device's mapping of host memory; a
 * pageable one goes through a device staging buffer that the handle keeps
 * (grown on demand; growing it waits for `stream` first).  Validation as for
 * muse_lmhead_forward_group.
 */
int muse_lmhead_forward_group_host(muse_lmhead *h, const float *hidden_host, const float *gamma,
                                   float eps, const muse_gemv_segment *segments,
                                   int n_segments, void *stream);

/* Argmax keys (muse_lmhead_set_argmax_key). */
#define MUSE_ARGMAX_CAPPED 0   /* the returned logit, after scale and cap (the default) */
#define MUSE_ARGMAX_PRECAP 1   /* scale * raw, before the cap */

/*
 * Choose what the handle's argmax ranks, for every later forward (logits and
 * logprobs alike; the logits themselves do not change).  The cap is strictly
 * increasing, so in exact arithmetic both keys pick the same index ("Chapter
 * 20 — Final norm, LM head, and the soft cap", §20.2: greedy selection is
 * invariant to the cap).  In f32 the cap merges distinct large values into
 * ties: pre-cap values from about 170 up land on a few floats just below 20
 * (170 and 190 both give 19.999998f; from about 200 on every value gives
 * 20.0f), and the capped key then returns the lowest index among them, where
 * the pre-cap key keeps their order.  Ties of the key itself go to the lowest
 * index either way.  Host-only
 * setting, takes effect for forwards enqueued after it; MUSE_ERR_VALUE for an
 * unknown key.
 */
int muse_lmhead_set_argmax_key(muse_lmhead *h, int key);

/* Free the handle and its workspace.  NULL is allowed.  Must not be called
 * while a forward using the handle may still be running on the GPU. */
void muse_lmhead_destroy(muse_lmhead *h);

/* Static English text for a status code; for MUSE_ERR_CUDA it names the last
 * CUDA error seen by this thread's failing call. */
const char *muse_lmhead_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MUSE_LMHEAD_H */
