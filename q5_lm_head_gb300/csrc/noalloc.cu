// Handle-free batch-1 forward that allocates no device memory.
//
// Some callers cannot call cudaMalloc at the moment they need a forward: code
// running while a CUDA graph is being captured (an allocation there is not
// captured, and cudaMalloc may synchronise the device), runtimes that reserve
// all device memory up front through their own allocator and forbid further
// allocations, and latency-critical serving loops that must not risk the
// implicit synchronisation of an allocation.  For them this entry point keeps
// the small scratch the fused batch-1 kernel needs (the packed argmax key, the
// CTA completion ticket and the status word) in a fixed array in the
// library's own device memory, instead of in a handle's workspace.
//
// Costs and limits: every GPU that loads the library holds kScratchBytes of
// it until the process exits; all calls on a device share the array, so two
// calls that may overlap on the GPU race on it and must be serialised by the
// caller (one stream, or events).
//
// Failure reporting: the kernel ORs a status bit into the array when one of
// its bounded waits gives up (its logits and argmax are then invalid).  Each
// forward clears only the argmax key and the ticket, so that bit stays set
// across later forwards until muse_lmhead_noalloc_device_status reads and
// clears it.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "muse_lmhead.h"

namespace {

constexpr int kScratchBytes = 256;   // stated maximum; the kernel needs 16 of it
constexpr int kMaxDevices = 64;

// keys (u64) at 0, ticket (u32) at 8, status (u32) at kStatusOffset
constexpr int kStatusOffset = 12;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_setup_mutex;
std::atomic<unsigned char *> g_scratch_ptr[kMaxDevices];   // device address per device, set once

// Once per device, with that device current: the device address of g_scratch
// (host code only sees a host-side stand-in for the array's name).
int scratch_for_device(int device, unsigned char **out) {
  unsigned char *p = g_scratch_ptr[device].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_ptr[device].load(std::memory_order_relaxed);
    if (!p) {
      void *addr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&addr, g_scratch);
      if (e != cudaSuccess || !addr) return MUSE_ERR_CUDA;
      p = static_cast<unsigned char *>(addr);
      g_scratch_ptr[device].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return MUSE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int muse_lmhead_forward_b1_noalloc(int device, const float *hidden, const float *gamma, float eps,
                                              const void *weights, int64_t n_rows, int64_t k, float scale,
                                              float cap, float *logits, int32_t *argmax, void *stream) {
  if (!hidden || !weights || !logits) return MUSE_ERR_NULL;
  if (n_rows < 1 || n_rows > (int64_t{1} << 31) - 1 || k < 256 || k % 256 != 0) return MUSE_ERR_SHAPE;
  if (!muse::b1_supported(static_cast<int>(k))) return MUSE_ERR_SHAPE;   // the fused kernel's K only
  if (!std::isfinite(scale) || !std::isfinite(cap)) return MUSE_ERR_VALUE;
  if (gamma && (!std::isfinite(eps) || eps < 0.0f)) return MUSE_ERR_VALUE;
  if (!aligned16(hidden) || !aligned16(weights) || !aligned16(logits) || (gamma && !aligned16(gamma)))
    return MUSE_ERR_ALIGN;
  if (argmax && (reinterpret_cast<uintptr_t>(argmax) & 3u)) return MUSE_ERR_ALIGN;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return MUSE_ERR_CUDA;
  if (device < 0 || device >= ndev || device >= kMaxDevices) return MUSE_ERR_DEVICE;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return MUSE_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return MUSE_ERR_DEVICE;
  int st = MUSE_OK;
  int sms = 0;
  unsigned char *scratch = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  do {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      st = MUSE_ERR_CUDA;
      break;
    }
    if (major != 10 || minor != 3) {
      st = MUSE_ERR_DEVICE;
      break;
    }
    if ((st = scratch_for_device(device, &scratch)) != MUSE_OK) break;
    // key and ticket must start at zero; an earlier call leaves them re-armed,
    // this also covers one that gave up early.  The status word (bytes 12..15)
    // is left alone: it keeps a failure until the status call reads it.
    if (cudaMemsetAsync(scratch, 0, kStatusOffset, s) != cudaSuccess) {
      st = MUSE_ERR_CUDA;
      break;
    }
    muse::LaunchArgs a;
    a.hidden = hidden;
    a.gamma = gamma;
    a.eps = eps;
    a.w = static_cast<const uint8_t *>(weights);
    a.scale = scale;
    a.cap = cap;
    a.logits = logits;
    a.argmax = argmax;
    a.batch = 1;
    a.n_rows = n_rows;
    a.k = static_cast<int>(k);
    a.num_sms = sms;
    a.ws.keys = reinterpret_cast<unsigned long long *>(scratch);
    a.ws.ticket = reinterpret_cast<unsigned int *>(scratch + 8);
    a.ws.status = reinterpret_cast<uint32_t *>(scratch + kStatusOffset);
    a.ws.x = nullptr;   // the fused kernel normalises in registers and needs no activation buffer
    a.stream = s;
    if (muse::launch_b1(a) != cudaSuccess) st = MUSE_ERR_CUDA;
  } while (false);
  if (prev >= 0 && prev != device) cudaSetDevice(prev);
  return st;
}

extern "C" int muse_lmhead_noalloc_device_status(int device, void *stream, uint32_t *status) {
  if (!status) return MUSE_ERR_NULL;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return MUSE_ERR_CUDA;
  if (device < 0 || device >= ndev || device >= kMaxDevices) return MUSE_ERR_DEVICE;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return MUSE_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return MUSE_ERR_DEVICE;
  int st = MUSE_OK;
  unsigned char *scratch = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  do {
    if ((st = scratch_for_device(device, &scratch)) != MUSE_OK) break;
    // after the caller's earlier work on `stream`: copy the word out, clear it
    if (cudaMemcpyAsync(&word, scratch + kStatusOffset, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(scratch + kStatusOffset, 0, sizeof(word), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      st = MUSE_ERR_CUDA;
      break;
    }
    *status = word;
  } while (false);
  if (prev >= 0 && prev != device) cudaSetDevice(prev);
  return st;
}
