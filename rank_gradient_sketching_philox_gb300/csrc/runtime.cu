// Host-side runtime helpers: TMA tensor-map encoding (through the driver entry
// point, so the library does not link libcuda) with a cache of encoded maps,
// the device error word that kernels set when a bounded wait gives up, the
// device count of exactly recomputed weights, and cached device properties.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include "internal.h"

namespace rgs {
namespace {

// Bits set by kernels whose bounded waits timed out (see tc.cuh).
__device__ int g_device_error = 0;
// Weights the update kernels recomputed on their exact path.
__device__ unsigned long long g_exact_count = 0;

constexpr int kMaxDevices = 64;
int* g_error_ptr[kMaxDevices] = {};
unsigned long long* g_exact_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::mutex g_mutex;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

cudaError_t encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                           uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// An encoded map is a pure function of its arguments and the device, so each
// encoding is kept: steps that reuse their buffers skip the driver call.
struct MapKey {
  int device;
  uintptr_t base;
  uint64_t inner, outer, stride;
  uint32_t box_inner, box_outer;
  bool operator==(const MapKey& o) const {
    return device == o.device && base == o.base && inner == o.inner && outer == o.outer &&
           stride == o.stride && box_inner == o.box_inner && box_outer == o.box_outer;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = 1469598103934665603ull;
    const uint64_t parts[6] = {(uint64_t)k.device, (uint64_t)k.base, k.inner, k.outer, k.stride,
                               ((uint64_t)k.box_inner << 32) | k.box_outer};
    for (uint64_t v : parts) h = (h ^ v) * 1099511628211ull;
    return (size_t)h;
  }
};
constexpr size_t kMapCacheMax = size_t(1) << 16;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;
std::mutex g_map_mutex;

}  // namespace

cudaError_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const MapKey key{dev, reinterpret_cast<uintptr_t>(base), inner, outer, row_stride_bytes, box_inner, box_outer};
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    auto it = g_map_cache.find(key);
    if (it != g_map_cache.end()) {
      *map = it->second;
      return cudaSuccess;
    }
  }
  cudaError_t err = encode_bf16_2d(map, base, inner, outer, row_stride_bytes, box_inner, box_outer);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
  g_map_cache.emplace(key, *map);
  return cudaSuccess;
}

cudaError_t device_error_word(int** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_error_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_device_error);
    if (err != cudaSuccess) return err;
    g_error_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_error_ptr[dev];
  return cudaSuccess;
}

cudaError_t device_exact_counter(unsigned long long** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_exact_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_exact_count);
    if (err != cudaSuccess) return err;
    g_exact_ptr[dev] = static_cast<unsigned long long*>(p);
  }
  *out = g_exact_ptr[dev];
  return cudaSuccess;
}

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
uint64_t launches_issued() { return g_launches.load(std::memory_order_relaxed); }

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_num_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

}  // namespace rgs
