// Status strings, version and per-device launch attributes of libtreeverify.
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
