// Status strings, version, per-device launch attributes and SM counts of libtreeverify.
#include <atomic>
#include <mutex>
#include <set>
#include <tuple>

#include "tv_common.cuh"

namespace tv {

bool smem_limit(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::tuple<const void*, int, int>> done;   // (kernel, device, bytes)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const auto key = std::make_tuple(kernel, dev, bytes);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(key)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  done.insert(key);
  return true;
}

int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices];   // 0: not read yet
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < kMaxDevices && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 148;
  }
  if (dev >= 0 && dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace tv

TV_API const char* tv_status_str(int status) {
  switch (status) {
    case TV_OK: return "TV_OK";
    case TV_EINVAL: return "TV_EINVAL: invalid argument, pointer or shape";
    case TV_EUNSUPPORTED: return "TV_EUNSUPPORTED: shape outside what the kernels implement";
    case TV_ECUDA: return "TV_ECUDA: a CUDA launch or runtime call failed";
    case TV_EWORKSPACE: return "TV_EWORKSPACE: workspace missing, misaligned or too small";
    default: return "unknown tv status";
  }
}

TV_API int tv_version(void) { return 100; }
