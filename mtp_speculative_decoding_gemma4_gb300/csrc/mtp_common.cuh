// Device helpers shared by the libmtp kernels: vector loads of bf16 / fp32 rows,
// element conversions, warp and block reductions, and order-preserving (value, id) keys for
// argmax / top-k with lowest-id tie-breaking.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mtp {

constexpr int kThreads = 256;  // every phase kernel runs 8 warps per CTA
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------- element types

template <typename T> struct Elem;
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;  // elements per 16-byte load
  __device__ static inline float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  // fp32 -> bf16, round to nearest even (storage conversion; activations stay fp32).
  __device__ static inline __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};
template <> struct Elem<float> {
  static constexpr int kVec = 4;
  __device__ static inline float to_f(float v) { return v; }
  __device__ static inline float from_f(float v) { return v; }
};


// 16-byte vector load of kVec elements, converted to fp32.
__device__ inline void load_vec(const __nv_bfloat16* p, float* out) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}
__device__ inline void load_vec(const float* p, float* out) {
  float4 f = *reinterpret_cast<const float4*>(p);
  out[0] = f.x; out[1] = f.y; out[2] = f.z; out[3] = f.w;
}
// Streaming variant for data read once per launch (weights, K): bypass L1 allocation.
__device__ inline void load_vec_stream(const __nv_bfloat16* p, float* out) {
  uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}
__device__ inline void load_vec_stream(const float* p, float* out) {
  float4 f = __ldcs(reinterpret_cast<const float4*>(p));
  out[0] = f.x; out[1] = f.y; out[2] = f.z; out[3] = f.w;
}

// ---------------------------------------------------------------- reductions

// Programmatic dependent launch (the tensor-core path's chain of launches): let the next
// kernel of the chain begin launching now, then wait until the kernels this one depends on
// have completed and their writes are visible. Both return at once for a launch that did
// not opt in, so every kernel of the library may call it first.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ inline float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ inline unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Sum over the CTA (kThreads threads). `red` holds kWarps floats. All threads get the sum.
__device__ inline float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) s += red[i];
  return s;
}

// ---------------------------------------------------------------- argmax keys

// Monotone map of fp32 to uint32 (larger float -> larger key); -0 is folded onto +0 so
// that equal values compare equal.
__device__ inline uint32_t ord_f32(float f) {
  if (f == 0.0f) f = 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ inline float unord_f32(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}
// (value, id) -> key whose maximum is the largest value, lowest id among equal values.
__device__ inline unsigned long long argmax_key(float v, int id) {
  return (static_cast<unsigned long long>(ord_f32(v)) << 32) | (0xffffffffu - static_cast<uint32_t>(id));
}
__device__ inline int key_id(unsigned long long k) { return static_cast<int>(0xffffffffu - static_cast<uint32_t>(k)); }
__device__ inline float key_val(unsigned long long k) { return unord_f32(static_cast<uint32_t>(k >> 32)); }

// RMSNorm factor 1/sqrt(mean(v^2) + eps) of a vector held in shared memory (fp32).
__device__ inline float rms_factor(const float* v, int n, float eps, float* red) {
  float s = 0.f;
  for (int i = threadIdx.x; i < n; i += kThreads) s += v[i] * v[i];
  s = block_sum(s, red);
  return rsqrtf(s / static_cast<float>(n) + eps);
}

__device__ inline float gelu_tanh(float x) {
  // 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
  const float k0 = 0.7978845608028654f;
  return 0.5f * x * (1.0f + tanhf(k0 * (x + 0.044715f * x * x * x)));
}

}  // namespace mtp
