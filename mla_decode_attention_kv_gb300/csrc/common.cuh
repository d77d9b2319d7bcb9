// Shared helpers of the CUDA kernels: dtype packing and row stores.
#pragma once
#include <cuda_runtime.h>
#include <algorithm>
#include <cmath>
#include <cstdint>
#include "ptx.cuh"

namespace mla {

enum Dtype : int { kBF16 = 0, kFP16 = 1, kFP32 = 2 };

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

__device__ __forceinline__ uint32_t pack2_dt(float a, float b, int dt) {
  return dt == kBF16 ? pack2<true>(a, b) : pack2<false>(a, b);
}

__device__ __forceinline__ float2 unpack2(uint32_t w, int dt) {
  if (dt == kBF16) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(v);
  }
  __half2 v = *reinterpret_cast<__half2*>(&w);
  return __half22float2(v);
}

// Store 32 consecutive fp32 accumulator values (raw bits in v) times `mul`
// at element offset e of a row-major tensor of dtype dt (16-byte aligned).
// 32 consecutive values of one row, scaled by mul, stored in dtype dt.  With
// a 32-byte aligned base (the row offsets e are multiples of 32 elements)
// each thread writes whole 32-byte sectors, which halves the store
// instructions of a row-per-thread epilogue.
__device__ __forceinline__ void store_row32(void* base, int64_t e, const uint32_t (&v)[32],
                                            float mul, int dt) {
  const bool wide = (reinterpret_cast<uintptr_t>(base) & 31u) == 0;
  if (dt == kFP32) {
    float* p = static_cast<float*>(base) + e;
    if (wide) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__uint_as_float(v[8 * q + k]) * mul);
        st_global_v8(p + 8 * q, w);
      }
    } else {
      float4* p4 = reinterpret_cast<float4*>(p);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        p4[q] = make_float4(__uint_as_float(v[4 * q]) * mul, __uint_as_float(v[4 * q + 1]) * mul,
                            __uint_as_float(v[4 * q + 2]) * mul, __uint_as_float(v[4 * q + 3]) * mul);
    }
  } else {
    uint16_t* p = static_cast<uint16_t*>(base) + e;
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
      w[k] = pack2_dt(__uint_as_float(v[2 * k]) * mul, __uint_as_float(v[2 * k + 1]) * mul, dt);
    if (wide) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t h[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) h[k] = w[8 * q + k];
        st_global_v8(p + 16 * q, h);
      }
    } else {
      uint4* p4 = reinterpret_cast<uint4*>(p);
#pragma unroll
      for (int q = 0; q < 4; ++q) p4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
  }
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

constexpr float kLn2 = 0.6931471805599453f;

}  // namespace mla
