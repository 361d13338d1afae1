// Shared device/host helpers of libtreeverify (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tv.h"

#define TV_API extern "C" __attribute__((visibility("default")))

namespace tv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TV_OK : TV_ECUDA;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to the device, so it is set once per
// (kernel, device) and remembered; false when the runtime refuses.
bool smem_limit(const void* kernel, int bytes);
// Streaming multiprocessors of the current device (read once per device).
int sm_count();
template <typename... KArgs>
inline bool smem_limit(void (*kernel)(KArgs...), int bytes) {
  return smem_limit(reinterpret_cast<const void*>(kernel), bytes);
}

// Programmatic dependent launch.  Kernels of the verification step are
// launched with programmatic stream serialization: a kernel's CTAs may be
// scheduled while the previous kernel in the stream drains.  Each such
// kernel calls griddep_wait() before its first global-memory access (it
// returns once the previous grid has completed and its writes are visible;
// without the launch attribute it returns at once) and then
// griddep_release() so that the next kernel can be scheduled likewise.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // the stream's priority travels with the launch, so that a kernel captured
  // into a CUDA graph keeps it (the CTA scheduler serves higher priority first)
  int prio = 0;
  if (cudaStreamGetPriority(st, &prio) != cudaSuccess) {
    cudaGetLastError();
    prio = 0;
  }
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributePriority;
  attr[1].val.priority = prio;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess ? TV_OK : TV_ECUDA;
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_at(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(*p) << 16);
}

// float -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <typename T>
__device__ __forceinline__ T warp_max(T v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (value desc, index asc) total order used by every top-k / argmax.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

}  // namespace tv
