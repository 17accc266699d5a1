// Device helpers shared by the kernels: dtype unpacking, streaming loads, fast exp2, error flag.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

__device__ __forceinline__ void raise_error(unsigned* err, unsigned bit) {
  if (err != nullptr) atomicOr(err, bit);
}

// 16-byte load that bypasses L1 (K/V rows are read once per launch).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 32-bit read-only load issued where it stands (not moved by the compiler), so that a value loaded
// now and used much later has its latency hidden by the work in between.
__device__ __forceinline__ int ld_nc_s32(const int32_t* p) {
  int v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// 2^x with the hardware approximation (ex2.approx; -inf -> +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------------------------------------
// dtype traits: unpack a 16-byte vector into fp32, round fp32 back to the I/O type
// ------------------------------------------------------------------------------------------------
template <typename T>
struct Elt;

template <>
struct Elt<__nv_bfloat16> {
  static constexpr int kVec = 8;  // elements per 16 bytes
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static __nv_bfloat16 from_float(float x) { return __float2bfloat16_rn(x); }
};

template <>
struct Elt<__half> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static __half from_float(float x) { return __float2half_rn(x); }
};

template <>
struct Elt<float> {
  static constexpr int kVec = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static float from_float(float x) { return x; }
};

// Programmatic dependent launch: let the next kernel in the stream start its launch now (its CTAs
// still wait for this grid's completion before reading what it wrote).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Wait until the preceding grid in the stream has completed and its writes are visible (a no-op when
// the kernel was launched without programmatic serialization).
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Resolve which sequence a prefill query row belongs to: the largest b with qsl[b] <= row.
__device__ __forceinline__ int find_sequence(const int32_t* qsl, int batch, int64_t row) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(qsl + mid) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace pa
