// C-ABI of the output-stage library: argument validation (fail closed, launch
// nothing on error), handle and workspace management, kernel-path dispatch and
// the host-buffer convenience forward.  The public contract is in
// include/muse_lmhead.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "internal.h"
#include "muse_lmhead.h"

struct muse_lmhead {
  int device;
  int format;              // MUSE_FORMAT_Q5_K or MUSE_FORMAT_Q4_K
  int argmax_key;          // MUSE_ARGMAX_CAPPED (default) or MUSE_ARGMAX_PRECAP
  int64_t n_rows;
  int64_t k;
  int max_batch;
  int num_sms;
  muse::Workspace ws;
  void *ws_base;           // single device allocation backing ws
  size_t ws_split_cnt_bytes;  // size of ws.split_cnt (0 without the tensor-core path)
  size_t ws_b1_cnt_bytes;     // size of ws.b1_cnt (0 without the split-K batch-1 path)
  CUtensorMap wmap;        // weight tensor map of the tensor-core path, for wmap_ptr
  const void *wmap_ptr;
  float *stage_hidden;     // forward_host staging (lazy)
  float *stage_logits;
  int32_t *stage_argmax;
  float *stage_group;      // forward_group_host staging of pageable outputs (lazy, grows)
  int64_t stage_group_n;   // its size in floats
};

namespace {

thread_local char g_cuda_msg[256] = "CUDA error";

int cuda_fail(cudaError_t e) {
  std::snprintf(g_cuda_msg, sizeof(g_cuda_msg), "CUDA runtime call failed: %s (%s)", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return MUSE_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

enum class Path { B1, B1Split, TensorCore, Generic };

// Partial sums of the split-K batch-1 path are [chunks][n_rows] floats: taken
// only while that stays within this bound (larger handles use the tensor cores).
constexpr size_t kMaxSplitFloats = size_t{1} << 26;

bool b1_split_ok(int64_t n_rows, int64_t k) {
  return muse::b1_split_chunks(static_cast<int>(k)) > 0 &&
         muse::b1_split_floats(n_rows, static_cast<int>(k)) <= kMaxSplitFloats;
}

Path choose_path(const muse_lmhead *h, int batch) {
  if (batch == 1 && muse::b1_supported(static_cast<int>(h->k))) return Path::B1;
  if (batch == 1 && b1_split_ok(h->n_rows, h->k)) return Path::B1Split;
  if (muse::tc_supported(batch, static_cast<int>(h->k))) return Path::TensorCore;
  return Path::Generic;
}

int validate_forward(const muse_lmhead *h, const void *hidden, int batch, const float *gamma, float eps,
                     const void *weights, float scale, float cap, const void *logits,
                     const int32_t *argmax) {
  if (!h || !hidden || !weights || !logits) return MUSE_ERR_NULL;
  if (batch < 1 || batch > h->max_batch) return MUSE_ERR_BATCH;
  if (!std::isfinite(scale) || !std::isfinite(cap)) return MUSE_ERR_VALUE;
  if (gamma && (!std::isfinite(eps) || eps < 0.0f)) return MUSE_ERR_VALUE;
  if (!aligned(weights, 16) || (gamma && !aligned(gamma, 16))) return MUSE_ERR_ALIGN;
  if (argmax && !aligned(argmax, 4)) return MUSE_ERR_ALIGN;
  return MUSE_OK;
}

int run_forward(muse_lmhead *h, const float *hidden, int batch, const float *gamma, float eps,
                const void *weights, float scale, float cap, float *logits, int32_t *argmax,
                cudaStream_t stream, bool lse_parts = false) {
  muse::LaunchArgs a;
  a.hidden = hidden;
  a.gamma = gamma;
  a.eps = eps;
  a.w = static_cast<const uint8_t *>(weights);
  a.scale = scale;
  a.cap = cap;
  a.logits = logits;
  a.argmax = argmax;
  a.batch = batch;
  a.n_rows = h->n_rows;
  a.k = static_cast<int>(h->k);
  a.num_sms = h->num_sms;
  a.ws = h->ws;
  a.stream = stream;
  a.lse_parts = lse_parts;
  a.q4 = h->format == MUSE_FORMAT_Q4_K;
  a.argmax_precap = h->argmax_key == MUSE_ARGMAX_PRECAP;
  cudaError_t e;
  switch (choose_path(h, batch)) {
    case Path::B1: e = muse::launch_b1(a); break;
    case Path::B1Split:
      e = h->ws.b1_part && h->ws.b1_cnt ? muse::launch_b1_split(a) : cudaErrorInvalidValue;
      break;
    case Path::TensorCore:
      if (!h->ws.xpkg || !h->ws.split_cnt || !h->ws.split_part) {   // never launch without its workspace
        e = cudaErrorInvalidValue;
        break;
      }
      if (h->wmap_ptr != weights) {
        e = muse::tc_encode_weights(&h->wmap, weights, h->n_rows, static_cast<int>(h->k), a.q4);
        if (e != cudaSuccess) break;
        h->wmap_ptr = weights;
      }
      e = muse::launch_tc(a, h->wmap);
      break;
    default: e = muse::launch_generic(a); break;
  }
  return e == cudaSuccess ? MUSE_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int muse_lmhead_init(muse_lmhead **out, int device, int64_t n_rows, int64_t k, int max_batch) {
  return muse_lmhead_init_format(out, device, n_rows, k, max_batch, MUSE_FORMAT_Q5_K);
}

int muse_lmhead_init_format(muse_lmhead **out, int device, int64_t n_rows, int64_t k, int max_batch,
                            int format) {
  if (!out) return MUSE_ERR_NULL;
  *out = nullptr;
  if (format != MUSE_FORMAT_Q5_K && format != MUSE_FORMAT_Q4_K) return MUSE_ERR_VALUE;
  if (n_rows < 1 || n_rows > (int64_t{1} << 31) - 1 || k < 256 || k % 256 != 0 || k > (1 << 20))
    return MUSE_ERR_SHAPE;
  if (max_batch < 1 || max_batch > MUSE_MAX_BATCH) return MUSE_ERR_BATCH;
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (device < 0 || device >= ndev) return MUSE_ERR_DEVICE;
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return cuda_fail(e);
  if (prop.major != 10 || prop.minor != 3) return MUSE_ERR_DEVICE;  // built for sm_103a only
  DeviceGuard g(device);
  if (!g.ok) return MUSE_ERR_DEVICE;

  muse_lmhead *h = new (std::nothrow) muse_lmhead();
  if (!h) return MUSE_ERR_NOMEM;
  h->device = device;
  h->format = format;
  h->n_rows = n_rows;
  h->k = k;
  h->max_batch = max_batch;
  h->num_sms = prop.multiProcessorCount;

  // One zeroed allocation: keys | ticket | status | logprob pairs | x | activation packages |
  // shared-tile counters | shared-tile partial sums (those three for the tensor-core path) |
  // chunk counters | chunk partial sums (the split-K batch-1 path)
  const size_t keys_b = sizeof(unsigned long long) * MUSE_MAX_BATCH;
  const size_t misc_b = 256;
  const size_t lse_b = sizeof(float2) * static_cast<size_t>(max_batch) * muse::kMaxLseParts;
  const size_t x_b = sizeof(float) * static_cast<size_t>(max_batch) * static_cast<size_t>(k);
  // the tensor-core path's workspace, wherever some batch size of this handle
  // takes that path (batch 1 does for a K without a fused batch-1 build)
  const bool split = b1_split_ok(n_rows, k);
  const bool tc = muse::tc_supported(max_batch, static_cast<int>(k)) &&
                  (max_batch >= 2 || (!muse::b1_supported(static_cast<int>(k)) && !split));
  const size_t pkg_b = tc ? muse::tc_workspace_bytes(static_cast<int>(k)) : 0;
  const size_t cnt_b = tc ? (sizeof(unsigned int) * muse::tc_split_counters(h->num_sms) + 255) / 256 * 256 : 0;
  const size_t part_b = tc ? sizeof(float) * muse::tc_split_floats(h->num_sms, max_batch) : 0;
  const size_t bcnt_b = split ? (sizeof(unsigned int) * muse::b1_split_counters(n_rows) + 255) / 256 * 256 : 0;
  const size_t bpart_b = split ? sizeof(float) * muse::b1_split_floats(n_rows, static_cast<int>(k)) : 0;
  const size_t total = keys_b + misc_b + lse_b + x_b + pkg_b + cnt_b + part_b + bcnt_b + bpart_b;
  void *base = nullptr;
  e = cudaMalloc(&base, total);
  if (e != cudaSuccess) {
    delete h;
    return e == cudaErrorMemoryAllocation ? MUSE_ERR_NOMEM : cuda_fail(e);
  }
  e = cudaMemset(base, 0, total);
  if (e != cudaSuccess) {
    cudaFree(base);
    delete h;
    return cuda_fail(e);
  }
  auto *p = static_cast<uint8_t *>(base);
  h->ws_base = base;
  h->ws.keys = reinterpret_cast<unsigned long long *>(p);
  h->ws.ticket = reinterpret_cast<unsigned int *>(p + keys_b);
  h->ws.status = reinterpret_cast<uint32_t *>(p + keys_b + 16);
  h->ws.lse_parts = reinterpret_cast<float2 *>(p + keys_b + misc_b);
  h->ws.x = reinterpret_cast<float *>(p + keys_b + misc_b + lse_b);
  h->ws.xpkg = pkg_b ? p + keys_b + misc_b + lse_b + x_b : nullptr;
  h->ws.split_cnt = cnt_b ? reinterpret_cast<unsigned int *>(p + keys_b + misc_b + lse_b + x_b + pkg_b) : nullptr;
  h->ws.split_part = part_b ? reinterpret_cast<float *>(p + keys_b + misc_b + lse_b + x_b + pkg_b + cnt_b) : nullptr;
  h->ws_split_cnt_bytes = cnt_b;
  // part_b is a multiple of 256 bytes (num_sms * 2 * 128 * slots floats)
  uint8_t *pb = p + keys_b + misc_b + lse_b + x_b + pkg_b + cnt_b + part_b;
  h->ws.b1_cnt = bcnt_b ? reinterpret_cast<unsigned int *>(pb) : nullptr;
  h->ws.b1_part = bpart_b ? reinterpret_cast<float *>(pb + bcnt_b) : nullptr;
  h->ws_b1_cnt_bytes = bcnt_b;
  *out = h;
  return MUSE_OK;
}

namespace {

// Checks shared by the grouped calls (hidden may be a host or device pointer:
// the caller checks what it needs of it); fills segs.
int validate_group(const muse_lmhead *h, const float *hidden, const float *gamma, float eps,
                   const muse_gemv_segment *segments, int n_segments, muse::GemvSegment *segs) {
  if (!h || !hidden || !segments) return MUSE_ERR_NULL;
  if (n_segments < 1 || n_segments > MUSE_MAX_SEGMENTS) return MUSE_ERR_SHAPE;
  if (!muse::b1_supported(static_cast<int>(h->k))) return MUSE_ERR_SHAPE;
  if (gamma && (!std::isfinite(eps) || eps < 0.0f)) return MUSE_ERR_VALUE;
  if (gamma && !aligned(gamma, 16)) return MUSE_ERR_ALIGN;
  for (int i = 0; i < n_segments; ++i) {
    const muse_gemv_segment &g = segments[i];
    if (!g.weights || !g.out) return MUSE_ERR_NULL;
    if (g.n_rows < 1 || g.n_rows > (int64_t{1} << 31) - 1) return MUSE_ERR_SHAPE;
    if (!std::isfinite(g.scale) || !std::isfinite(g.cap)) return MUSE_ERR_VALUE;
    if (!aligned(g.weights, 16) || !aligned(g.out, 4)) return MUSE_ERR_ALIGN;
    segs[i] = {static_cast<const uint8_t *>(g.weights), g.out, g.n_rows, g.scale, g.cap};
  }
  return MUSE_OK;
}

int run_group(muse_lmhead *h, const float *hidden, const float *gamma, float eps, const muse::GemvSegment *segs,
              int n_segments, cudaStream_t stream) {
  const cudaError_t e = muse::launch_b1_group(hidden, gamma, eps, static_cast<int>(h->k), segs, n_segments,
                                              h->ws.status, h->num_sms, stream, h->format == MUSE_FORMAT_Q4_K);
  return e == cudaSuccess ? MUSE_OK : cuda_fail(e);
}

// The forward_host staging buffers (max_batch rows of input and logits, the argmax), allocated once.
int ensure_host_staging(muse_lmhead *h) {
  if (h->stage_hidden) return MUSE_OK;
  const size_t hb = sizeof(float) * h->max_batch * h->k;
  const size_t lb = sizeof(float) * h->max_batch * h->n_rows;
  const size_t ab = sizeof(int32_t) * MUSE_MAX_BATCH;
  void *p1 = nullptr, *p2 = nullptr, *p3 = nullptr;
  cudaError_t e;
  if ((e = cudaMalloc(&p1, hb)) != cudaSuccess || (e = cudaMalloc(&p2, lb)) != cudaSuccess ||
      (e = cudaMalloc(&p3, ab)) != cudaSuccess) {
    if (p1) cudaFree(p1);
    if (p2) cudaFree(p2);
    return e == cudaErrorMemoryAllocation ? MUSE_ERR_NOMEM : cuda_fail(e);
  }
  h->stage_hidden = static_cast<float *>(p1);
  h->stage_logits = static_cast<float *>(p2);
  h->stage_argmax = static_cast<int32_t *>(p3);
  return MUSE_OK;
}

}  // namespace

int muse_lmhead_forward_group(muse_lmhead *h, const float *hidden, const float *gamma, float eps,
                              const muse_gemv_segment *segments, int n_segments, void *stream) {
  muse::GemvSegment segs[muse::kMaxSegments];
  const int st = validate_group(h, hidden, gamma, eps, segments, n_segments, segs);
  if (st != MUSE_OK) return st;
  if (!aligned(hidden, 16)) return MUSE_ERR_ALIGN;
  DeviceGuard dg(h->device);
  if (!dg.ok) return MUSE_ERR_DEVICE;
  return run_group(h, hidden, gamma, eps, segs, n_segments, static_cast<cudaStream_t>(stream));
}

int muse_lmhead_forward_logprobs(muse_lmhead *h, const float *hidden, int batch, const float *gamma, float eps,
                                 const void *weights, float scale, float cap, float *logprobs, float *lse,
                                 int32_t *argmax, void *stream) {
  int st = validate_forward(h, hidden, batch, gamma, eps, weights, scale, cap, logprobs, argmax);
  if (st != MUSE_OK) return st;
  if (!aligned(hidden, 16) || !aligned(logprobs, 16) || (lse && !aligned(lse, 4))) return MUSE_ERR_ALIGN;
  DeviceGuard g(h->device);
  if (!g.ok) return MUSE_ERR_DEVICE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the batch-1 kernel leaves one (max, sum exp) pair per CTA; other paths get a pass over the logits
  // (the split-K kernel too: which CTA finishes a row varies, the pass keeps the sum's order fixed).
  // The pairs' buffer holds kMaxLseParts per batch row: a grid wider than that (a device with more
  // SMs than the buffer has slots) takes the separate pass as well.
  const bool fused = choose_path(h, batch) == Path::B1 && muse::b1_grid(h->n_rows, h->num_sms) <= muse::kMaxLseParts;
  st = run_forward(h, hidden, batch, gamma, eps, weights, scale, cap, logprobs, argmax, s, fused);
  if (st != MUSE_OK) return st;
  int n_parts;
  cudaError_t e = cudaSuccess;
  if (fused) {
    n_parts = muse::b1_grid(h->n_rows, h->num_sms);
  } else {
    n_parts = muse::lse_parts_for(h->n_rows);
    e = muse::launch_lse_parts(logprobs, batch, h->n_rows, h->ws.lse_parts, s);
  }
  if (e == cudaSuccess) e = muse::launch_logprob_apply(logprobs, batch, h->n_rows, h->ws.lse_parts, n_parts, lse, s);
  return e == cudaSuccess ? MUSE_OK : cuda_fail(e);
}

int muse_lmhead_forward(muse_lmhead *h, const float *hidden, int batch, const float *gamma, float eps,
                        const void *weights, float scale, float cap, float *logits, int32_t *argmax,
                        void *stream) {
  int st = validate_forward(h, hidden, batch, gamma, eps, weights, scale, cap, logits, argmax);
  if (st != MUSE_OK) return st;
  if (!aligned(hidden, 16) || !aligned(logits, 16)) return MUSE_ERR_ALIGN;
  DeviceGuard g(h->device);
  if (!g.ok) return MUSE_ERR_DEVICE;
  return run_forward(h, hidden, batch, gamma, eps, weights, scale, cap, logits, argmax,
                     static_cast<cudaStream_t>(stream));
}

namespace {

// The device's address of a page-locked host buffer (cudaHostAlloc or
// cudaHostRegister memory mapped for this handle's device), or nullptr for
// pageable memory and memory pinned for another device's context.
void *mapped_alias(const void *p, int device) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();                   // clear the sticky-free error of an unknown pointer
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer || at.device != device) return nullptr;
  return at.devicePointer;
}

}  // namespace

int muse_lmhead_forward_host(muse_lmhead *h, const float *hidden_host, int batch, const float *gamma,
                             float eps, const void *weights, float scale, float cap, float *logits_host,
                             int32_t *argmax_host, void *stream) {
  if (!h) return MUSE_ERR_NULL;
  if (!logits_host && !argmax_host) return MUSE_ERR_NULL;
  // logits_host stands in for the logits pointer in the shared checks
  const void *out_probe = logits_host ? static_cast<const void *>(logits_host) : argmax_host;
  int st = validate_forward(h, hidden_host, batch, gamma, eps, weights, scale, cap, out_probe, nullptr);
  if (st != MUSE_OK) return st;
  DeviceGuard g(h->device);
  if (!g.ok) return MUSE_ERR_DEVICE;
  cudaError_t e;
  if ((st = ensure_host_staging(h)) != MUSE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t in_b = sizeof(float) * static_cast<size_t>(batch) * h->k;
  if ((e = cudaMemcpyAsync(h->stage_hidden, hidden_host, in_b, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e);
  // Page-locked output buffers are written by the kernels themselves, through
  // the device's mapping of host memory (the link carries the same bytes, with
  // no copy after the kernel); pageable ones go through the staging buffers.
  float *logits_out = h->stage_logits;              // the kernels' logits when none reach the host
  int32_t *argmax_out = argmax_host ? h->stage_argmax : nullptr;
  if (void *a = logits_host ? mapped_alias(logits_host, h->device) : nullptr) {
    logits_out = static_cast<float *>(a);
    logits_host = nullptr;                           // nothing left to copy
  }
  if (void *a = argmax_host ? mapped_alias(argmax_host, h->device) : nullptr) {
    argmax_out = static_cast<int32_t *>(a);
    argmax_host = nullptr;
  }
  st = run_forward(h, h->stage_hidden, batch, gamma, eps, weights, scale, cap, logits_out, argmax_out, s);
  if (st != MUSE_OK) return st;
  if (logits_host) {
    const size_t out_b = sizeof(float) * static_cast<size_t>(batch) * h->n_rows;
    if ((e = cudaMemcpyAsync(logits_host, h->stage_logits, out_b, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
      return cuda_fail(e);
  }
  if (argmax_host) {
    if ((e = cudaMemcpyAsync(argmax_host, h->stage_argmax, sizeof(int32_t) * batch, cudaMemcpyDeviceToHost,
                             s)) != cudaSuccess)
      return cuda_fail(e);
  }
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
  return MUSE_OK;
}

int muse_lmhead_forward_group_host(muse_lmhead *h, const float *hidden_host, const float *gamma, float eps,
                                   const muse_gemv_segment *segments, int n_segments, void *stream) {
  muse::GemvSegment segs[muse::kMaxSegments];
  int st = validate_group(h, hidden_host, gamma, eps, segments, n_segments, segs);
  if (st != MUSE_OK) return st;
  DeviceGuard g(h->device);
  if (!g.ok) return MUSE_ERR_DEVICE;
  if ((st = ensure_host_staging(h)) != MUSE_OK) return st;
  // page-locked outputs are written through the device's mapping of host
  // memory; pageable ones go through the group staging buffer
  float *host_out[muse::kMaxSegments] = {};
  int64_t staged = 0;
  for (int i = 0; i < n_segments; ++i) {
    if (void *a = mapped_alias(segs[i].out, h->device)) {
      segs[i].out = static_cast<float *>(a);
    } else {
      host_out[i] = segs[i].out;
      staged += segs[i].n_rows;
    }
  }
  cudaError_t e;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (staged > h->stage_group_n) {
    if (h->stage_group) {
      if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);   // earlier calls' copies done
      cudaFree(h->stage_group);
      h->stage_group = nullptr;
      h->stage_group_n = 0;
    }
    void *p = nullptr;
    if ((e = cudaMalloc(&p, sizeof(float) * static_cast<size_t>(staged))) != cudaSuccess)
      return e == cudaErrorMemoryAllocation ? MUSE_ERR_NOMEM : cuda_fail(e);
    h->stage_group = static_cast<float *>(p);
    h->stage_group_n = staged;
  }
  int64_t off = 0;
  for (int i = 0; i < n_segments; ++i) {
    if (host_out[i]) {
      segs[i].out = h->stage_group + off;
      off += segs[i].n_rows;
    }
  }
  if ((e = cudaMemcpyAsync(h->stage_hidden, hidden_host, sizeof(float) * h->k, cudaMemcpyHostToDevice, s)) !=
      cudaSuccess)
    return cuda_fail(e);
  if ((st = run_group(h, h->stage_hidden, gamma, eps, segs, n_segments, s)) != MUSE_OK) return st;
  for (int i = 0; i < n_segments; ++i) {
    if (host_out[i] &&
        (e = cudaMemcpyAsync(host_out[i], segs[i].out, sizeof(float) * segs[i].n_rows, cudaMemcpyDeviceToHost,
                             s)) != cudaSuccess)
      return cuda_fail(e);
  }
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
  return MUSE_OK;
}

int muse_lmhead_set_argmax_key(muse_lmhead *h, int key) {
  if (!h) return MUSE_ERR_NULL;
  if (key != MUSE_ARGMAX_CAPPED && key != MUSE_ARGMAX_PRECAP) return MUSE_ERR_VALUE;
  h->argmax_key = key;
  return MUSE_OK;
}

int muse_lmhead_launches_per_forward(const muse_lmhead *h, int batch, int with_norm) {
  if (!h) return MUSE_ERR_NULL;
  if (batch < 1 || batch > h->max_batch) return MUSE_ERR_BATCH;
  switch (choose_path(h, batch)) {
    case Path::B1:
    case Path::B1Split: return 1;
    case Path::TensorCore: return 2;   // activation-package prep + tcgen05 kernel
    default: return with_norm ? 2 : 1;  // generic: RMSNorm pre-pass + GEMV
  }
}

const char *muse_lmhead_path_name(const muse_lmhead *h, int batch) {
  if (!h || batch < 1 || batch > h->max_batch) return nullptr;
  switch (choose_path(h, batch)) {
    case Path::B1: return "gemv_b1";
    case Path::B1Split: return "gemv_b1_split";
    case Path::TensorCore: return "gemm_tc";
    default: return "gemv_generic";
  }
}

int muse_lmhead_device_status(muse_lmhead *h, uint32_t *status_out) {
  if (!h || !status_out) return MUSE_ERR_NULL;
  DeviceGuard g(h->device);
  if (!g.ok) return MUSE_ERR_DEVICE;
  cudaError_t e = cudaMemcpy(status_out, h->ws.status, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? MUSE_OK : cuda_fail(e);
}

int muse_lmhead_clear_device_status(muse_lmhead *h, void *stream) {
  if (!h) return MUSE_ERR_NULL;
  DeviceGuard g(h->device);
  if (!g.ok) return MUSE_ERR_DEVICE;
  cudaError_t e = cudaMemsetAsync(h->ws.status, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream));
  // a forward that gave up may have left a shared-tile or chunk counter counted in
  if (e == cudaSuccess && h->ws.split_cnt)
    e = cudaMemsetAsync(h->ws.split_cnt, 0, h->ws_split_cnt_bytes, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess && h->ws.b1_cnt)
    e = cudaMemsetAsync(h->ws.b1_cnt, 0, h->ws_b1_cnt_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MUSE_OK : cuda_fail(e);
}

int muse_lmhead_selftest_wait_timeout(muse_lmhead *h, void *stream) {
  if (!h) return MUSE_ERR_NULL;
  DeviceGuard g(h->device);
  if (!g.ok) return MUSE_ERR_DEVICE;
  const cudaError_t e = muse::launch_wait_timeout_selftest(h->ws.status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MUSE_OK : cuda_fail(e);
}

void muse_lmhead_destroy(muse_lmhead *h) {
  if (!h) return;
  DeviceGuard g(h->device);
  if (h->ws_base) cudaFree(h->ws_base);
  if (h->stage_hidden) cudaFree(h->stage_hidden);
  if (h->stage_logits) cudaFree(h->stage_logits);
  if (h->stage_argmax) cudaFree(h->stage_argmax);
  if (h->stage_group) cudaFree(h->stage_group);
  delete h;
}

const char *muse_lmhead_status_string(int status) {
  switch (status) {
    case MUSE_OK: return "ok";
    case MUSE_ERR_NULL: return "a required pointer is NULL";
    case MUSE_ERR_SHAPE: return "bad shape: need n_rows >= 1 and k a positive multiple of 256";
    case MUSE_ERR_BATCH: return "batch outside 1..max_batch (max_batch at most 32)";
    case MUSE_ERR_ALIGN: return "misaligned pointer: 16 bytes for hidden/gamma/weights/logits, 4 for argmax";
    case MUSE_ERR_VALUE: return "non-finite scale or cap, or bad eps";
    case MUSE_ERR_DEVICE: return "bad device index or not an sm_103 GPU";
    case MUSE_ERR_CUDA: return g_cuda_msg;
    case MUSE_ERR_NOMEM: return "out of memory";
    default: return "unknown status";
  }
}

}  // extern "C"
