// Device helpers shared by the libmla kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

typedef __nv_bfloat16 bf16;
typedef __nv_fp8_storage_t fp8;   // raw e4m3 byte

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxRopePairs = 64;     // d_r <= 128

// RoPE inverse frequencies theta^(-2k/d_r), computed on the host in double and passed by
// value so no table lives in device memory.
struct RopeTable {
  double inv_freq[kMaxRopePairs];
  int pairs;
};

// Rotation angle pos * inv_freq reduced to [-pi, pi] in double, then the hardware sin/cos
// approximation (absolute error about 2^-21 on [-pi, pi]): positions up to 2^17 stay
// accurate to about fp32 rounding, without a slow large-argument path.
__device__ __forceinline__ void rope_sincos(const RopeTable& rt, int k, int pos, float* s, float* c) {
  double a = (double)pos * rt.inv_freq[k];
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  a = fma(-two_pi, rint(a * inv_two_pi), a);
  __sincosf((float)a, s, c);
}

// ---- element conversion -------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float fp8_to_f32(uint8_t b) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
  return __half2float(__half(hr));
}
__device__ __forceinline__ uint8_t f32_to_fp8(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// Cache element codec: encode(value, inverse-free scale division) / decode.
template <typename CT> struct CacheCodec;
template <> struct CacheCodec<float> {
  __device__ __forceinline__ static float encode(float v, float) { return v; }
};
template <> struct CacheCodec<bf16> {
  __device__ __forceinline__ static bf16 encode(float v, float) { return __float2bfloat16_rn(v); }
};
template <> struct CacheCodec<uint8_t> {
  // IEEE division by the per-tensor scale, then round-to-nearest-even saturating e4m3.
  __device__ __forceinline__ static uint8_t encode(float v, float scale) { return f32_to_fp8(v / scale); }
};

// ---- warp reductions ----------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void flag_status(int32_t* status, int code) {
  if (status) atomicOr(status, 1 << code);
}

// Validates one append row; returns the destination row of the cache or -1.
__device__ __forceinline__ long long append_slot(const int32_t* req_ids, const int32_t* positions,
                                                 const int32_t* block_table, int batch,
                                                 int max_pages, int num_pages, int P, int r,
                                                 int32_t* status, int* pos_out) {
  const int b = req_ids[r], pos = positions[r];
  if (b < 0 || b >= batch || pos < 0 || pos / P >= max_pages) {
    flag_status(status, MLA_ERR_DEVICE_GUARD);
    return -1;
  }
  const int page = block_table[(long long)b * max_pages + pos / P];
  if (page < 0 || page >= num_pages) {
    flag_status(status, MLA_ERR_DEVICE_GUARD);
    return -1;
  }
  *pos_out = pos;
  return (long long)page * P + pos % P;
}

}  // namespace mla
