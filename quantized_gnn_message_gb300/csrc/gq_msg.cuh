// gq_msg.cuh -- reading one 8-column chunk of a message row: the
// de-quantized packed row of a marginal node (AdaQP Eqn 5, h^ = q*S + Z as
// one fused multiply-add) or the fp32 row of a central node (Sec. 3.1).
// Loads are split from decoding so callers can keep several rows in flight.
#pragma once

#include "gq_common.cuh"

namespace gq {

struct MsgSrc {
  const float* X;
  int64_t ldx;
  const uint8_t* packed;
  int64_t pitch;
  int hoff;
  const uint8_t* mask;  // null: every row packed (when BITS < 32)
  int d;
};

template <int BITS>
struct RawChunk {
  uint32_t w[8];  // fp32 bits, or the packed payload word(s) in w[0..1]
  float2 h;       // {S, Z} of a packed row
  bool quant;
};

template <int BITS>
__device__ __forceinline__ bool is_quant(const MsgSrc& m, int64_t x) {
  return BITS < 32 && (m.mask == nullptr || __ldg(m.mask + x) != 0);
}

template <int BITS>
__device__ __forceinline__ void load_raw(const MsgSrc& m, int64_t x, bool quant, int c, RawChunk<BITS>& r) {
  r.quant = quant;
  if (BITS < 32 && quant) {
    const uint8_t* row = m.packed + x * m.pitch;
    r.h = __ldg(reinterpret_cast<const float2*>(row + m.hoff));
    if constexpr (BITS == 8) {
      const uint2 t = __ldg(reinterpret_cast<const uint2*>(row + (int64_t)c * 8));
      r.w[0] = t.x;
      r.w[1] = t.y;
    } else if constexpr (BITS == 4) {
      r.w[0] = __ldg(reinterpret_cast<const uint32_t*>(row + (int64_t)c * 4));
    } else if constexpr (BITS == 2) {
      r.w[0] = __ldg(reinterpret_cast<const uint16_t*>(row + (int64_t)c * 2));
    }
  } else {
    const float* xr = m.X + x * m.ldx + c * 8;
    const float4 a = ldg_f4(xr);
    r.w[0] = __float_as_uint(a.x); r.w[1] = __float_as_uint(a.y);
    r.w[2] = __float_as_uint(a.z); r.w[3] = __float_as_uint(a.w);
    if (c * 8 + 4 < m.d) {
      const float4 b = ldg_f4(xr + 4);
      r.w[4] = __float_as_uint(b.x); r.w[5] = __float_as_uint(b.y);
      r.w[6] = __float_as_uint(b.z); r.w[7] = __float_as_uint(b.w);
    } else {
      r.w[4] = r.w[5] = r.w[6] = r.w[7] = 0u;
    }
  }
}

// The 8 message values of a chunk.
template <int BITS>
__device__ __forceinline__ void decode(const RawChunk<BITS>& r, float (&v)[8]) {
  if (BITS < 32 && r.quant) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float q;
      if constexpr (BITS == 8) {
        q = code_to_float((r.w[i >> 2] >> ((i & 3) * 8)) & 0xFFu);
      } else {
        q = code_to_float((r.w[0] >> (i * (BITS < 8 ? BITS : 1))) & ((1u << (BITS < 8 ? BITS : 1)) - 1u));
      }
      v[i] = __fmaf_rn(q, r.h.x, r.h.y);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r.w[i]);
  }
}

}  // namespace gq
