// Status strings and version of libtreeverify.
#include "tv_common.cuh"

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
