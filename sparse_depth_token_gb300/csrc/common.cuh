// Device-side helpers shared by the kernels of the sparse-depth layer library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "xmod.h"

namespace xmod {

// ---------------------------------------------------------------- element types

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

template <typename T> __device__ __forceinline__ float ld_f(const T* p) { return Elem<T>::to_f(*p); }
template <typename T> __device__ __forceinline__ void st_f(T* p, float v) { *p = Elem<T>::from_f(v); }

// 16-byte vector of elements: 8 bf16 or 4 fp32.
template <typename T> struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  uint4 raw;
  __device__ __forceinline__ float get(int i) const {
    const T* e = reinterpret_cast<const T*>(&raw);
    return Elem<T>::to_f(e[i]);
  }
  __device__ __forceinline__ void set(int i, float v) {
    T* e = reinterpret_cast<T*>(&raw);
    e[i] = Elem<T>::from_f(v);
  }
};

template <typename T>
__device__ __forceinline__ Vec16<T> ld_vec(const T* p) {
  Vec16<T> v;
  v.raw = *reinterpret_cast<const uint4*>(p);
  return v;
}
template <typename T>
__device__ __forceinline__ Vec16<T> ld_vec_stream(const T* p) {
  Vec16<T> v;
  v.raw = __ldcs(reinterpret_cast<const uint4*>(p));
  return v;
}
template <typename T>
__device__ __forceinline__ void st_vec(T* p, const Vec16<T>& v) {
  *reinterpret_cast<uint4*>(p) = v.raw;
}

// ---------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------- device status word

// First error wins; later errors do not overwrite it.
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float sigmoidf_acc(float s) { return 1.0f / (1.0f + expf(-s)); }

// ---------------------------------------------------------------- programmatic dependent launch
//
// Kernels launched with launch_pdl() may start while the previous kernel on the
// stream is still finishing. Each such kernel lets its own successor start early
// (pdl_trigger) and, before its first global-memory access, waits until every
// earlier grid on the stream has completed and its writes are visible (pdl_wait).
// Both are no-ops for an ordinary launch.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace xmod
