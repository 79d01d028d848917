// gq_common.cuh -- shared device/host helpers of libgq (CUDA, sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gq.h"

#define GQ_TRY_CUDA(expr)                       \
  do {                                          \
    cudaError_t gq_e_ = (expr);                 \
    if (gq_e_ != cudaSuccess) return GQ_ERR_CUDA; \
  } while (0)

#define GQ_TRY(expr)              \
  do {                            \
    int gq_s_ = (expr);           \
    if (gq_s_ != GQ_OK) return gq_s_; \
  } while (0)

namespace gq {

constexpr unsigned FULL = 0xffffffffu;

inline int launch_status() { return cudaGetLastError() == cudaSuccess ? GQ_OK : GQ_ERR_CUDA; }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

inline int sm_count() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return v;
}

inline bool valid_bits(int b) { return b == 2 || b == 4 || b == 8; }

// Packed row layout (see gq.h): payload, pad to 8, {S, Z} fp32, pad to 16.
__host__ __device__ inline int64_t payload_bytes(int d, int bits) { return ((int64_t)d * bits + 7) / 8; }
__host__ __device__ inline int64_t header_offset(int d, int bits) { return (payload_bytes(d, bits) + 7) / 8 * 8; }
__host__ __device__ inline int64_t packed_pitch(int d, int bits) { return (header_offset(d, bits) + 8 + 15) / 16 * 16; }

// MurmurHash3's 32-bit finalizer.
__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  h *= 0xC2B2AE35u;
  h ^= h >> 16;
  return h;
}

// Per-row key of the stochastic-rounding stream.
__device__ __forceinline__ uint32_t row_key(uint32_t seed_key, uint32_t row) { return fmix32(row ^ seed_key); }
__host__ __device__ inline uint32_t seed_fold(uint64_t seed) { return (uint32_t)seed ^ (uint32_t)(seed >> 32); }

// fmix32(low32(seed) ^ high32(seed)), computed once on the host per call.
inline uint32_t seed_key_host(uint64_t seed) {
  uint32_t h = seed_fold(seed);
  h ^= h >> 16;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  h *= 0xC2B2AE35u;
  h ^= h >> 16;
  return h;
}

// u = (h >> 9) * 2^-23 in [0, 1 - 2^-23]: built as the float 1.m (exact)
// minus one (exact by Sterbenz), no integer-to-float conversion.
__device__ __forceinline__ float noise_u(uint32_t kr, uint32_t col) {
  const uint32_t h = fmix32(kr + col * 0x9E3779B9u);
  return __fsub_rn(__uint_as_float(0x3F800000u | (h >> 9)), 1.0f);
}

// Exact float of a small non-negative integer code (< 2^23) via the 2^23
// magic constant; `bits23` must already hold the code in its low bits.
__device__ __forceinline__ float code_to_float(uint32_t code) {
  return __fsub_rn(__uint_as_float(0x4B000000u | code), 8388608.0f);
}

// Byte k of w as an exact float (one PRMT + one FADD).
template <int K>
__device__ __forceinline__ float byte_to_float(uint32_t w) {
  return __fsub_rn(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | K)), 8388608.0f);
}

// Two floats as one bf16x2 word (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float4 ldg_f4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ void st_f4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

}  // namespace gq
