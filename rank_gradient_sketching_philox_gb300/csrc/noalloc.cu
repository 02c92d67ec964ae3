// Normalized-SGD update for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory: a plugin that a host
// framework calls with nothing but its input and output buffers, or a process
// that hands all free device memory to another pool up front (for example a
// rollout engine that gives HBM to its KV cache), where cudaMalloc either
// fails or stalls the device.  sketch_apply_update_normsgd_noalloc serves them:
// it runs exactly the computation of sketch_apply_update_normsgd, with the
// workspace taken from a fixed array in device memory that this file owns.
//
// The array is kNoAllocScratchBytes long.  It is reserved on a device when the
// library's device code is loaded there (under lazy module loading: when the
// first call looks up its address) and stays reserved until the process exits.
// The address found on a device is cached for the life of the process; a
// cudaDeviceReset() on that device invalidates it (and every other address the
// library keeps), so the library must not be called on a device after it has
// been reset.  Every call shares the array: two calls whose kernels overlap on
// the GPU (different streams, or different host threads) race on it and
// corrupt each other's results; order such calls on one stream.  No word of it
// needs to start at zero: each call writes every scratch value it reads before
// reading it, so the contents left by an earlier call do not matter.
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "sketch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the array on the current device.  In host code the name
// g_noalloc_scratch is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t sketch_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

sketch_status sketch_apply_update_normsgd_noalloc(uint16_t* W, int64_t d, int64_t k, int64_t ld_w,
                                                  const float* C, const float* P, int64_t r, float tau,
                                                  uint64_t seed, uint32_t layer, uint32_t step,
                                                  const double* wnorm2_in, double* wnorm2_out,
                                                  int32_t* dev_status, void* stream) {
  const size_t need = sketch_workspace_bytes(SKETCH_OP_UPDATE_NORMSGD, 0, d, k, r);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "the allocation-free update keeps its scratch in a fixed %zu-byte device array; "
             "d=%lld, k=%lld, r=%lld needs %zu bytes (use sketch_apply_update_normsgd with a workspace)",
             kNoAllocScratchBytes, (long long)d, (long long)k, (long long)r, need);
    rgs::set_last_error(msg);
    return SKETCH_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const cudaError_t err = scratch_address(&scratch);
  if (err != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "apply_update_normsgd_noalloc: %s", cudaGetErrorString(err));
    rgs::set_last_error(msg);
    return SKETCH_ERR_CUDA;
  }
  return sketch_apply_update_normsgd(W, d, k, ld_w, C, P, r, tau, seed, layer, step, wnorm2_in, wnorm2_out,
                                     dev_status, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
