// gq_spmm.cu -- dequantization-fused CSR aggregation.
//
//   Y[r,:] = rowscale[r] * sum_{e in row r} w_e * m_{col[e]}
//
// with m_x = deq(packed row x) (AdaQP Sec. 2.3, Eqn 5) when node x is marginal
// and the fp32 row X[x,:] otherwise (AdaQP Sec. 3.1), and the coefficient of
// an edge either colscale[col[e]] (GCN / GraphSAGE-mean normalization,
// Sancus Sec. 2, split into a per-source and a per-destination factor) or a
// per-edge, per-head attention weight alpha[e, head] (Tango Sec. 2.1, step 5
// and its transposed backward form).
//
// Work decomposition (power-law degrees).  The graph's static schedule
// cuts every row of degree > hub_threshold into thread-block tasks (heaviest
// first, so they start before the light rows); a row cut into several tasks
// writes one partial row per task to the workspace and the last task to
// finish (arrival ticket) adds them in task order.  Four kernels share it:
//   - spmm_warp_kernel (packed and fp32 rows mixed by a mask, or fp32 rows
//     alone, with coefficients or with per-edge, per-head attention weights,
//     fp32 or 8-bit codes; 64 < d <= 256).  One warp per edge; lane l owns
//     4 or 8 columns and loads its part of the message row straight into
//     registers, 3-4 edges in flight per warp and 32 warps per SM.
//   - spmm_async_kernel (d <= 512: rows of one kind, all packed or all fp32;
//     packed and fp32 rows mixed by a mask; or rows of mixed widths for
//     d <= 128).  A group of LG lanes walks a stream of edges (a slice of a
//     heavy task, or one of the schedule's runs of consecutive light rows)
//     and gathers message rows into a shared-memory ring with cp.async,
//     kAS - 1 steps ahead of the step it consumes, so each SM keeps ~100 KB
//     of gathers in flight.
//   - spmm_bulk_kernel (rows of mixed widths, 128 < d <= 256).  One warp per
//     edge: the lane holding an edge's metadata copies the whole message row
//     into a slot of the warp's shared-memory ring with one bulk copy onto
//     the slot's mbarrier, and all 32 lanes consume it.
//   - spmm_kernel (attention weights outside 64 < d <= 256, or d > 512).  A light
//     row is one warp's job: lane groups of G lanes take one edge at a time,
//     each lane owning 8 consecutive columns (CPL chunks of 8 for d > 256);
//     edge metadata is loaded 32 edges at a time and broadcast with
//     shuffles, and U edges per group are gathered before any is consumed.
//     A heavy task's 8 warps split its edges into contiguous streams
//     (stream_row) whose partial rows are summed in shared memory in warp
//     order.
// An optional ReLU gate (one bit per output element) zeroes output elements
// as rows are written; in the warp and ring kernels it is a template
// parameter, since its code in the row flush changes the register
// allocation of their edge loops.
// Every sum runs in a fixed order, so results are identical run to run.
#include <cuda_bf16.h>

#include "gq_common.cuh"
#include "gq_internal.cuh"
#include "gq_sm100.cuh"

namespace gq {

struct SpmmParams {
  const int32_t* rowptr;
  const int32_t* col;
  const int32_t* eperm;     // edge id of each entry (transposed CSR), or null = identity
  const float* colscale;    // per gathered row, or null (= 1)
  const float* rowscale;    // per output row, or null (= 1)
  const float* alpha;       // per edge x heads (edge-weight mode 1)
  const uint8_t* acode;     // per edge x heads 8-bit codes (edge-weight mode 2)
  const float* ahdr;        // per output row x heads {S, Z} of those codes
  int heads, fshift;        // head of column j = j >> fshift
  const float* X;
  int64_t ldx;
  const uint8_t* packed;
  int64_t pitch;
  int hoff;
  const uint8_t* mask;      // null: every row packed (BITS < 32)
  float* Y;
  __nv_bfloat16* Yb;        // if set, the output is written in bf16 here instead
  int64_t ldy;
  const uint32_t* gate;     // if set, output element (r, c) is written as 0 unless bit c % 32 of
  int64_t ldg;              // word gate[r * ldg + c / 32] is set (a ReLU derivative as bits)
  int64_t n_rows;
  int d;
  const int32_t* tasks;     // heavy-row schedule (see gq_sched)
  const int32_t* groups;
  int64_t n_tasks;
  int hub_threshold;
  float* partial;           // [slot][d] partial rows of split heavy rows
  int* tickets;             // [group] arrivals, zero at launch
  const int32_t* light;     // runs of light rows {row_begin, row_end}
  int64_t n_light;
  int* err;                 // device status word (bounded waits that gave up)
  const uint8_t* rbits;     // per-row bit-widths (mixed packed rows), or null
  const int64_t* roff;      // byte offset of each packed row (mixed), or null
};

namespace {

constexpr int kSpmmThreads = 256;
constexpr int kSpmmWarps = kSpmmThreads / 32;

template <int BITS>
struct Chunk {
  uint32_t w[BITS == 32 ? 8 : (BITS == 8 ? 2 : 1)];
  float2 h;
};

// Load the message chunk `c` (columns 8c..8c+7) of gathered row x.
template <int BITS>
__device__ __forceinline__ void load_msg(const SpmmParams& p, int64_t x, bool quant, int c, Chunk<32>& f,
                                         Chunk<BITS>& q) {
  if (BITS < 32 && quant) {
    const uint8_t* row = p.packed + x * p.pitch;
    q.h = __ldg(reinterpret_cast<const float2*>(row + p.hoff));
    if constexpr (BITS == 8) {
      const uint2 t = __ldg(reinterpret_cast<const uint2*>(row + (int64_t)c * 8));
      q.w[0] = t.x;
      q.w[1] = t.y;
    } else if constexpr (BITS == 4) {
      q.w[0] = __ldg(reinterpret_cast<const uint32_t*>(row + (int64_t)c * 4));
    } else {
      q.w[0] = __ldg(reinterpret_cast<const uint16_t*>(row + (int64_t)c * 2));
    }
  } else {
    const float* xr = p.X + x * p.ldx + c * 8;
    const float4 a = ldg_f4(xr);
    f.w[0] = __float_as_uint(a.x); f.w[1] = __float_as_uint(a.y);
    f.w[2] = __float_as_uint(a.z); f.w[3] = __float_as_uint(a.w);
    if (c * 8 + 4 < p.d) {
      const float4 b = ldg_f4(xr + 4);
      f.w[4] = __float_as_uint(b.x); f.w[5] = __float_as_uint(b.y);
      f.w[6] = __float_as_uint(b.z); f.w[7] = __float_as_uint(b.w);
    } else {
      f.w[4] = f.w[5] = f.w[6] = f.w[7] = 0u;
    }
  }
}

template <int BITS>
__device__ __forceinline__ float code_at(const Chunk<BITS>& q, int i) {
  if constexpr (BITS == 8) {
    const uint32_t w = q.w[i >> 2];
    switch (i & 3) {
      case 0: return byte_to_float<0>(w);
      case 1: return byte_to_float<1>(w);
      case 2: return byte_to_float<2>(w);
      default: return byte_to_float<3>(w);
    }
  } else if constexpr (BITS < 8) {
    return code_to_float((q.w[0] >> (i * BITS)) & ((1u << BITS) - 1u));
  } else {
    return 0.0f;
  }
}

template <int BITS>
__device__ __forceinline__ void consume(bool quant, float coef, const Chunk<32>& f, const Chunk<BITS>& q,
                                        float (&acc)[8]) {
  if (BITS < 32 && quant) {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(coef, __fmaf_rn(code_at<BITS>(q, i), q.h.x, q.h.y), acc[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(coef, __uint_as_float(f.w[i]), acc[i]);
  }
}

// Accumulate, into this lane's chunks, the edges of batches
// [e_beg + 32*first, ...) with a stride of `stride` batches.
template <int BITS, int G, int CPL, int EW>
__device__ __forceinline__ void accumulate_row(const SpmmParams& p, int64_t row, int64_t e_beg, int64_t e_end,
                                               int first, int stride, float (&acc)[CPL][8]) {
  constexpr int NG = 32 / G;
  constexpr int U = CPL == 1 ? 4 : (CPL == 2 ? 2 : 1);
  const int lane = threadIdx.x & 31;
  const int g = lane / G;
  const int gl = lane % G;
  const int nchunks = (p.d + 7) >> 3;
  float2 az[CPL];  // mode 2: {S, Z} of the row's codes for the head of each chunk
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    az[i] = make_float2(0.0f, 0.0f);
    const int c = gl + G * i;
    if (EW == 2 && c < nchunks)
      az[i] = __ldg(reinterpret_cast<const float2*>(p.ahdr) + row * p.heads + ((c * 8) >> p.fshift));
  }
  for (int64_t base = e_beg + 32 * (int64_t)first; base < e_end; base += 32 * (int64_t)stride) {
    const int64_t e = base + lane;
    const bool valid = e < e_end;
    int32_t x = 0;
    float cf = 0.0f;
    int32_t eid = 0;
    bool qm = false;
    if (valid) {
      x = __ldg(p.col + e);
      if (EW) {
        eid = p.eperm ? __ldg(p.eperm + e) : (int32_t)e;
      } else {
        cf = p.colscale ? __ldg(p.colscale + x) : 1.0f;
      }
      qm = BITS < 32 && (p.mask == nullptr || __ldg(p.mask + x) != 0);
    }
    const int cnt = (int)min((int64_t)32, e_end - base);
    for (int jj = 0; jj < cnt; jj += NG * U) {
      Chunk<32> fb[U][CPL];
      Chunk<BITS> qb[U][CPL];
      bool act[U], qt[U];
      float cj[U][CPL];
#pragma unroll
      for (int t = 0; t < U; ++t) {
        const int j = jj + g + NG * t;
        const int src = j < cnt ? j : 0;
        const int32_t xj = __shfl_sync(FULL, x, src);
        const float cs = __shfl_sync(FULL, cf, src);
        const int32_t ej = __shfl_sync(FULL, eid, src);
        qt[t] = __shfl_sync(FULL, (int)qm, src) != 0;
        act[t] = j < cnt;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = gl + G * i;
          cj[t][i] = cs;
          if (act[t] && c < nchunks) {
            if (EW == 1) cj[t][i] = __ldg(p.alpha + (int64_t)ej * p.heads + ((c * 8) >> p.fshift));
            if (EW == 2)
              cj[t][i] = __fmaf_rn(code_to_float(__ldg(p.acode + (int64_t)ej * p.heads + ((c * 8) >> p.fshift))),
                                   az[i].x, az[i].y);
            load_msg<BITS>(p, xj, qt[t], c, fb[t][i], qb[t][i]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < U; ++t) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = gl + G * i;
          if (act[t] && c < nchunks) consume<BITS>(qt[t], cj[t][i], fb[t][i], qb[t][i], acc[i]);
        }
      }
    }
  }
}

template <int G, int CPL>
__device__ __forceinline__ void group_reduce(float (&acc)[CPL][8]) {
#pragma unroll
  for (int o = G; o < 32; o <<= 1)
#pragma unroll
    for (int i = 0; i < CPL; ++i)
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[i][k] += __shfl_xor_sync(FULL, acc[i][k], o);
}

// The output value of row r, column c after the optional ReLU gate (the
// derivative of the activation of the layer whose input this output is, one
// bit per element).
__device__ __forceinline__ float gated(const SpmmParams& p, int64_t r, int c, float v) {
  return (p.gate != nullptr && !((__ldg(p.gate + r * p.ldg + (c >> 5)) >> (c & 31)) & 1u)) ? 0.0f : v;
}
// columns c .. c+3 (c a multiple of 4)
__device__ __forceinline__ float4 gated4(const SpmmParams& p, int64_t r, int c, float4 v) {
  if (p.gate != nullptr) {
    const uint32_t b = __ldg(p.gate + r * p.ldg + (c >> 5)) >> (c & 31);
    if (!(b & 1u)) v.x = 0.0f;
    if (!(b & 2u)) v.y = 0.0f;
    if (!(b & 4u)) v.z = 0.0f;
    if (!(b & 8u)) v.w = 0.0f;
  }
  return v;
}

__device__ __forceinline__ void store_chunk(const SpmmParams& p, int64_t r, int c, float s, const float (&a_in)[8]) {
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = (c * 8 + k < p.d) ? gated(p, r, c * 8 + k, a_in[k]) : a_in[k];
  if (p.Yb != nullptr) {
    __nv_bfloat16* y = p.Yb + r * p.ldy + c * 8;
    if (c * 8 + 4 < p.d) {
      *reinterpret_cast<uint4*>(y) = make_uint4(pack_bf16x2(a[0] * s, a[1] * s), pack_bf16x2(a[2] * s, a[3] * s),
                                                pack_bf16x2(a[4] * s, a[5] * s), pack_bf16x2(a[6] * s, a[7] * s));
    } else {
      *reinterpret_cast<uint2*>(y) = make_uint2(pack_bf16x2(a[0] * s, a[1] * s), pack_bf16x2(a[2] * s, a[3] * s));
    }
    return;
  }
  float* y = p.Y + r * p.ldy;
  st_f4(y + c * 8, a[0] * s, a[1] * s, a[2] * s, a[3] * s);
  if (c * 8 + 4 < p.d) st_f4(y + c * 8 + 4, a[4] * s, a[5] * s, a[6] * s, a[7] * s);
}


// ---------------------------------------------------------------------------
// Edge streams of a heavy-row task: a group of LG lanes walks one
// contiguous stretch of the task's edges, lane j of the group owning columns
// [16 j, 16 j + 16), U edges per step, in a three-stage pipeline: column ids
// are loaded two steps ahead, the per-source coefficient and mask bit one
// step ahead, and the message rows of the current step are gathered before
// any is consumed.
// De-quantization is folded into the accumulation: with c = 2^(b-1),
//   a * (q S + Z) = (a S) (q - c) + a (Z + c S),
// so each element costs one FMA on the centred code and the per-edge term
// a (Z + c S) is summed once per lane.
// ---------------------------------------------------------------------------
constexpr int kLC = 16;  // columns per lane in an edge stream
constexpr int kLU = 2;   // edges per step

// One lane's 16-column chunk of one message row.  With ALLQ (every row
// packed) only the payload words are kept, which saves registers.
template <int BITS, bool ALLQ>
struct LMsg {
  static constexpr int PW = BITS < 32 ? (kLC * BITS + 31) / 32 : kLC;
  uint32_t w[ALLQ ? PW : kLC];  // fp32 bits (central row) or the packed payload words
  float2 h;                     // {S, Z}
  bool quant;
};

template <int BITS, bool ALLQ>
__device__ __forceinline__ void lload(const SpmmParams& p, int64_t x, bool quant, int c0, LMsg<BITS, ALLQ>& m) {
  m.quant = ALLQ || quant;
  if (BITS < 32 && (ALLQ || quant)) {
    const uint8_t* row = p.packed + x * p.pitch;
    m.h = __ldg(reinterpret_cast<const float2*>(row + p.hoff));
    const uint8_t* pl = row + (int64_t)c0 * BITS / 8;
    if constexpr (BITS == 8) {
      const uint4 t = __ldg(reinterpret_cast<const uint4*>(pl));
      m.w[0] = t.x; m.w[1] = t.y; m.w[2] = t.z; m.w[3] = t.w;
    } else if constexpr (BITS == 4) {
      const uint2 t = __ldg(reinterpret_cast<const uint2*>(pl));
      m.w[0] = t.x; m.w[1] = t.y;
    } else if constexpr (BITS == 2) {
      m.w[0] = __ldg(reinterpret_cast<const uint32_t*>(pl));
    }
  } else if constexpr (!ALLQ) {
    const float* xr = p.X + x * p.ldx + c0;
#pragma unroll
    for (int k = 0; k < kLC / 4; ++k) {
      if (c0 + 4 * k < p.d) {
        const float4 a = ldg_f4(xr + 4 * k);
        m.w[4 * k] = __float_as_uint(a.x); m.w[4 * k + 1] = __float_as_uint(a.y);
        m.w[4 * k + 2] = __float_as_uint(a.z); m.w[4 * k + 3] = __float_as_uint(a.w);
      } else {
        m.w[4 * k] = m.w[4 * k + 1] = m.w[4 * k + 2] = m.w[4 * k + 3] = 0u;
      }
    }
  }
}

// (q - c) as an exact float, for code k of the lane's payload.
template <int BITS, int K, int NW>
__device__ __forceinline__ float centred(const uint32_t (&w)[NW]) {
  if constexpr (BITS == 8) {
    return __fsub_rn(__uint_as_float(__byte_perm(w[K >> 2], 0x4B000000u, 0x7540u | (K & 3))), 8388608.0f + 128.0f);
  } else {
    constexpr int per = 32 / BITS;
    constexpr uint32_t mask = (1u << BITS) - 1u;
    const uint32_t code = (w[K / per] >> ((K % per) * BITS)) & mask;
    return __fsub_rn(__uint_as_float(0x4B000000u | code), 8388608.0f + (float)(1 << (BITS - 1)));
  }
}

template <int BITS, bool ALLQ, int K>
__device__ __forceinline__ void lconsume_q(const LMsg<BITS, ALLQ>& m, float cs, float (&acc)[kLC]) {
  if constexpr (K < kLC && BITS < 32) {
    acc[K] = __fmaf_rn(cs, centred<BITS, K>(m.w), acc[K]);
    lconsume_q<BITS, ALLQ, K + 1>(m, cs, acc);
  }
}

template <int BITS, bool ALLQ>
__device__ __forceinline__ void lconsume(const LMsg<BITS, ALLQ>& m, float coef, float (&acc)[kLC], float& accz) {
  if (BITS < 32 && (ALLQ || m.quant)) {
    constexpr float c = (float)(BITS < 32 ? (1 << (BITS - 1)) : 0);
    lconsume_q<BITS, ALLQ, 0>(m, coef * m.h.x, acc);
    accz = __fmaf_rn(coef, __fmaf_rn(c, m.h.x, m.h.y), accz);
  } else if constexpr (!ALLQ) {
#pragma unroll
    for (int k = 0; k < kLC; ++k) acc[k] = __fmaf_rn(coef, __uint_as_float(m.w[k]), acc[k]);
  }
}

// Per-edge metadata of U consecutive edges: column ids, then coefficients
// and mask bits.
template <int BITS, int EW, int U>
__device__ __forceinline__ void meta_cols(const SpmmParams& p, int64_t at, int64_t end, int32_t (&xs)[U]) {
#pragma unroll
  for (int t = 0; t < U; ++t) xs[t] = (at + t < end) ? __ldg(p.col + at + t) : 0;
}

template <int BITS, int EW, bool ALLQ, int U>
__device__ __forceinline__ void meta_coef(const SpmmParams& p, int64_t at, int64_t end, int head, float2 az,
                                          const int32_t (&xs)[U], float (&f)[U], bool (&q)[U]) {
#pragma unroll
  for (int t = 0; t < U; ++t) {
    f[t] = 1.0f;
    q[t] = ALLQ;
    if (at + t < end) {
      if (EW == 1) {
        const int64_t eid = p.eperm ? __ldg(p.eperm + at + t) : at + t;
        f[t] = __ldg(p.alpha + eid * p.heads + head);
      } else if (EW == 2) {  // forward only: the edge id is the CSR position
        f[t] = __fmaf_rn(code_to_float(__ldg(p.acode + (at + t) * p.heads + head)), az.x, az.y);
      } else if (p.colscale) {
        f[t] = __ldg(p.colscale + xs[t]);
      }
      if (!ALLQ) q[t] = BITS < 32 && (p.mask == nullptr || __ldg(p.mask + xs[t]) != 0);
    }
  }
}

// Accumulate the contiguous edges [e_beg, e_end) of one row into this
// lane's 16 columns, in the three-stage pipeline described above.
template <int BITS, int EW, bool ALLQ>
__device__ __forceinline__ void stream_row(const SpmmParams& p, int64_t e_beg, int64_t e_end, int c0, int head,
                                           float2 az, float (&acc)[kLC], float& accz) {
  constexpr int U = kLU;
  int32_t cx[U], nx[U];
  float cf[U];
  bool cq[U];
  meta_cols<BITS, EW, U>(p, e_beg, e_end, cx);
  meta_coef<BITS, EW, ALLQ, U>(p, e_beg, e_end, head, az, cx, cf, cq);
  meta_cols<BITS, EW, U>(p, e_beg + U, e_end, nx);
  for (int64_t e = e_beg; e < e_end; e += U) {
    LMsg<BITS, ALLQ> m[U];
#pragma unroll
    for (int t = 0; t < U; ++t)
      if (e + t < e_end && c0 < p.d) lload<BITS, ALLQ>(p, cx[t], cq[t], c0, m[t]);
    float nf[U];
    bool nq[U];
    meta_coef<BITS, EW, ALLQ, U>(p, e + U, e_end, head, az, nx, nf, nq);
    int32_t nnx[U];
    meta_cols<BITS, EW, U>(p, e + 2 * U, e_end, nnx);
#pragma unroll
    for (int t = 0; t < U; ++t)
      if (e + t < e_end && c0 < p.d) lconsume<BITS, ALLQ>(m[t], cf[t], acc, accz);
#pragma unroll
    for (int t = 0; t < U; ++t) {
      cx[t] = nx[t];
      cf[t] = nf[t];
      cq[t] = nq[t];
      nx[t] = nnx[t];
    }
  }
}

// Sum of the block's partial rows (one per warp in `part`) in warp order,
// written as the row's output, or as a split row's partial with the last
// task of the group adding all partials in task order.
__device__ __forceinline__ void finish_heavy(const SpmmParams& p, const int4& task, float* part) {
  __shared__ int last;
  const int64_t r = task.x;
  const float s = p.rowscale ? p.rowscale[r] : 1.0f;
  if (task.w < 0) {  // the whole row in this task
    for (int j = threadIdx.x; j < p.d; j += blockDim.x) {
      float t = 0.0f;
#pragma unroll
      for (int ww = 0; ww < kSpmmWarps; ++ww) t += part[ww * p.d + j];
      if (p.Yb != nullptr)
        p.Yb[r * p.ldy + j] = __float2bfloat16_rn(gated(p, r, j, t * s));
      else
        p.Y[r * p.ldy + j] = gated(p, r, j, t * s);
    }
    return;
  }
  const int4 grp = __ldg(reinterpret_cast<const int4*>(p.groups) + task.w);
  float* mine = p.partial + (int64_t)(grp.w + ((int)blockIdx.x - grp.y)) * p.d;
  for (int j = threadIdx.x; j < p.d; j += blockDim.x) {
    float t = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kSpmmWarps; ++ww) t += part[ww * p.d + j];
    mine[j] = t;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(&p.tickets[task.w], 1) == grp.z - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  const float* base = p.partial + (int64_t)grp.w * p.d;
  for (int j = threadIdx.x; j < p.d; j += blockDim.x) {
    float t = 0.0f;
    for (int k = 0; k < grp.z; ++k) t += __ldcg(base + (int64_t)k * p.d + j);
    if (p.Yb != nullptr)
      p.Yb[r * p.ldy + j] = __float2bfloat16_rn(gated(p, r, j, t * s));
    else
      p.Y[r * p.ldy + j] = gated(p, r, j, t * s);
  }
}

template <int BITS, int G, int CPL, int LG, int EW, bool ALLQ>
__global__ void __launch_bounds__(kSpmmThreads) spmm_kernel(const SpmmParams p) {
  extern __shared__ float part[];  // [kSpmmWarps][d] for heavy rows
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int gl = lane % G;
  const int nchunks = (p.d + 7) >> 3;

  if ((int64_t)blockIdx.x < p.n_tasks) {
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.tasks) + blockIdx.x);
    if constexpr (LG > 0) {
      // the task's edges cut into one contiguous stream per lane group
      constexpr int NG = 32 / LG;
      const int sid = w * NG + lane / LG;
      const int64_t len = task.z - task.y;
      int64_t chunk = (len + kSpmmWarps * NG - 1) / (kSpmmWarps * NG);
      chunk = (chunk + kLU - 1) / kLU * kLU;
      const int64_t b0 = task.y + (int64_t)sid * chunk;
      const int64_t b1 = min(b0 + chunk, (int64_t)task.z);
      const int c0 = (lane % LG) * kLC;
      const int head = EW ? (c0 >> p.fshift) : 0;
      float acc[kLC] = {};
      float accz = 0.0f;
      const float2 az = EW == 2 && c0 < p.d
                            ? __ldg(reinterpret_cast<const float2*>(p.ahdr) + (int64_t)task.x * p.heads + head)
                            : make_float2(0.0f, 0.0f);
      if (b0 < b1) stream_row<BITS, EW, ALLQ>(p, b0, b1, c0, head, az, acc, accz);
#pragma unroll
      for (int k = 0; k < kLC; ++k) acc[k] += accz;
#pragma unroll
      for (int o = LG; o < 32; o <<= 1)
#pragma unroll
        for (int k = 0; k < kLC; ++k) acc[k] += __shfl_xor_sync(FULL, acc[k], o);
      if (lane < LG && c0 < p.d)
#pragma unroll
        for (int k = 0; k < kLC; ++k)
          if (c0 + k < p.d) part[w * p.d + c0 + k] = acc[k];
    } else {
      float acc[CPL][8] = {};
      accumulate_row<BITS, G, CPL, EW>(p, task.x, task.y, task.z, w, kSpmmWarps, acc);
      group_reduce<G, CPL>(acc);
      if (lane < G) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = gl + G * i;
          if (c < nchunks)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (c * 8 + k < p.d) part[w * p.d + c * 8 + k] = acc[i][k];
        }
      }
    }
    __syncthreads();
    finish_heavy(p, task, part);
    return;
  }

  {
    // one warp per light row, lanes owning 8-column chunks
    const int64_t gw = ((int64_t)blockIdx.x - p.n_tasks) * kSpmmWarps + w;
    const int64_t nw = ((int64_t)gridDim.x - p.n_tasks) * kSpmmWarps;
    for (int64_t r = gw; r < p.n_rows; r += nw) {
      const int64_t a = p.rowptr[r], b = p.rowptr[r + 1];
      if (b - a > p.hub_threshold) continue;  // a block task handles it
      float acc[CPL][8] = {};
      accumulate_row<BITS, G, CPL, EW>(p, r, a, b, 0, 1, acc);
      group_reduce<G, CPL>(acc);
      if (lane < G) {
        const float s = p.rowscale ? p.rowscale[r] : 1.0f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = gl + G * i;
          if (c < nchunks) store_chunk(p, r, c, s, acc[i]);
        }
      }
    }
  }
}


// ---------------------------------------------------------------------------
// Asynchronous-copy aggregation (coefficient modes, d <= 512, every message
// row of one kind: all packed, or all fp32).
//
// A group of LG lanes walks a stream of edges (a slice of a heavy task, or
// one of the schedule's runs of consecutive light rows).  The message row of
// each edge is copied into the group's shared-memory ring with cp.async in
// contiguous 16-byte pieces spread over the lanes (a packed row whole,
// payload and {S, Z} together; an fp32 row as the pieces each lane will
// read), kAS - 1 steps of U edges ahead of the step being consumed.  Column
// ids are loaded two steps ahead and coefficients at issue time, into
// register rings indexed by the unrolled stage number.
//
// Packed rows: lane j owns columns [16 j, 16 j + 16) and reads its payload
// slice and the (broadcast) header from the slot.  De-quantization is
// folded into the accumulation:
//   a (q S + Z) = (a S)(q - c) + a (Z + c S),   c = 2^(b-1),
// so the per-edge term a (Z + c S) is summed once per lane.  The code q sits
// in the low mantissa bits of a float with exponent 2^23 (a byte permute for
// b = 8; a bit mask at offset o for b = 2, 4, giving 2^23 + q 2^o); one
// subtraction leaves (q - c) 2^o exactly, and the FMA takes a S 2^-o, so
// the product a S (q - c) is the same exact product as without the offset.
// fp32 rows: lane j owns the 4-column pieces j, j + LG, j + 2 LG, j + 3 LG.
// Pairs of columns go through the two-lane fp32 add and FMA of sm_100-class
// GPUs; each lane of those is an ordinary round-to-nearest fp32 operation.
// ---------------------------------------------------------------------------
constexpr int kAS = 4;  // pipeline stages

typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(f32x2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t sm_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// 16-byte pieces a lane copies per packed row: a row of d <= 16 LG columns
// has at most LG + 1 pieces at b = 8 and at most LG at b = 2, 4.
template <int BITS>
constexpr int kPiecesPerLane = BITS == 8 ? 2 : 1;

// Bytes of one edge slot: the largest row of the width bucket (d <= 16 LG),
// a packed row (payload rounded to 8 bytes, {S, Z}, rounded to 16) or an
// fp32 row (also when packed and fp32 rows mix: MX).  A compile-time stride
// keeps every slot address an immediate offset from the group's ring.
template <int BITS, int LG, bool MX>
constexpr int kSlot = BITS > 0 && BITS < 32 && !MX ? ((2 * BITS * LG + 7) / 8 * 8 + 8 + 15) / 16 * 16 : 64 * LG;

constexpr uint32_t kMagicBits = 0x4B000000u;  // 2^23 as fp32
constexpr float kMagic = 8388608.0f;

// The loop-invariant pair -(2^23 + c), c = 2^(b-1), for the subtraction.
template <int BITS>
__device__ __forceinline__ f32x2 a_bias() {
  constexpr float c = (float)(1 << (BITS > 0 && BITS < 32 ? BITS - 1 : 0));
  return f2_pack(-(kMagic + c), -(kMagic + c));
}

// The lane's place in its group's ring and in the row.
template <int LG>
struct ALane {
  const uint8_t* ring;  // group ring, for reading
  uint32_t sring;       // the same, shared-space address
  unsigned gmask;       // lanes of the group
  int gl;
  bool has0, has1;      // packed rows: pieces gl and gl + LG exist
  int c0;               // packed rows: first of the lane's 16 columns
  bool on;              // the lane owns at least one column
  int nv;               // fp32 rows: pieces gl + LG k, k < nv, are in range
  const uint8_t* src;   // the lane's first piece in message row 0
  uint32_t stride;      // bytes between message rows
  // mixed rows: an fp32 row's columns [c0, c0 + 16) as nvm 16-byte pieces,
  // piece k stored at 64 gl + 16 (k ^ swz) of the slot so that the pieces
  // of a quarter-warp fall in distinct banks
  const uint8_t* srcx;
  uint32_t stridex;
  int nvm, swz;
  // per-row widths (BITS == 0): bit 2i / 2i + 1 = pieces gl / gl + LG exist
  // in a row of width 2 << i
  uint32_t hasw;
};

// Column of accumulator entry i (acc[i / 2], half i % 2) of this lane.
template <int BITS, int LG>
__device__ __forceinline__ int a_col(const ALane<LG>& L, int i) {
  if constexpr (BITS < 32) return L.c0 + i;
  else return 4 * (L.gl + LG * (i >> 2)) + (i & 3);
}

// Accumulate a packed row of width BITS (header at hoff) from slot sl.
template <int BITS, int LG>
__device__ __forceinline__ void a_consume_packed(const ALane<LG>& L, const uint8_t* sl, int hoff, float cf,
                                                 f32x2 bias, f32x2 (&acc)[8], float& accz) {
  {
    constexpr float c = (float)(1 << (BITS - 1));
    const float2 h = *reinterpret_cast<const float2*>(sl + hoff);
    const float cs = cf * h.x;
    accz = __fmaf_rn(cf, __fmaf_rn(c, h.x, h.y), accz);
    const f32x2 cs2 = f2_pack(cs, cs);
    const uint8_t* pl = sl + L.gl * (2 * BITS);
    // the lane's 16 codes spread one per byte over four words, in column
    // order: byte a of sp[k] is code 4 a + k (b = 2), byte a of sp[2 h + k]
    // is code 8 h + 2 a + k (b = 4), byte a of sp[k] is code 4 k + a (b = 8)
    uint32_t sp[4];
    if constexpr (BITS == 8) {
      const uint4 t = *reinterpret_cast<const uint4*>(pl);
      sp[0] = t.x; sp[1] = t.y; sp[2] = t.z; sp[3] = t.w;
    } else if constexpr (BITS == 4) {
      const uint2 t = *reinterpret_cast<const uint2*>(pl);
      sp[0] = t.x & 0x0F0F0F0Fu; sp[1] = (t.x >> 4) & 0x0F0F0F0Fu;
      sp[2] = t.y & 0x0F0F0F0Fu; sp[3] = (t.y >> 4) & 0x0F0F0F0Fu;
    } else {
      const uint32_t t = *reinterpret_cast<const uint32_t*>(pl);
      sp[0] = t & 0x03030303u; sp[1] = (t >> 2) & 0x03030303u;
      sp[2] = (t >> 4) & 0x03030303u; sp[3] = (t >> 6) & 0x03030303u;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // columns 2i, 2i + 1: (word, byte) of each
      int w0, b0, w1, b1;
      if constexpr (BITS == 8) { w0 = i >> 1; b0 = (2 * i) & 3; w1 = w0; b1 = b0 + 1; }
      else if constexpr (BITS == 4) { w0 = 2 * (i >> 2); b0 = i & 3; w1 = w0 + 1; b1 = b0; }
      else { w0 = 2 * (i & 1); b0 = i >> 1; w1 = w0 + 1; b1 = b0; }
      const f32x2 v = f2_pack(__uint_as_float(__byte_perm(sp[w0], kMagicBits, 0x7540u | b0)),
                              __uint_as_float(__byte_perm(sp[w1], kMagicBits, 0x7540u | b1)));
      acc[i] = f2_fma(cs2, f2_add(v, bias), acc[i]);
    }
  }
}

// An fp32 row stored in the mixed layout (the lane's 16 columns as nvm
// swizzled 16-byte pieces).
template <int LG>
__device__ __forceinline__ void a_consume_fp32x(const ALane<LG>& L, const uint8_t* sl, float cf, f32x2 (&acc)[8]) {
  const f32x2 c2 = f2_pack(cf, cf);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < L.nvm) {
      const f32x2* xr = reinterpret_cast<const f32x2*>(sl + 64 * L.gl + 16 * (k ^ L.swz));
      acc[2 * k] = f2_fma(c2, xr[0], acc[2 * k]);
      acc[2 * k + 1] = f2_fma(c2, xr[1], acc[2 * k + 1]);
    }
  }
}

// Accumulate one edge from its slot sl with coefficient cf.  BITS == 0: the
// row's kind (0 = fp32, else its width) is `kind`.
template <int BITS, int LG, bool MX>
__device__ __forceinline__ void a_consume(const SpmmParams& p, const ALane<LG>& L, const uint8_t* sl, bool quant,
                                          int kind, float cf, f32x2 bias, f32x2 (&acc)[8], float& accz) {
  if constexpr (BITS == 0) {
    if (kind == 8)
      a_consume_packed<8, LG>(L, sl, (int)header_offset(p.d, 8), cf, a_bias<8>(), acc, accz);
    else if (kind == 4)
      a_consume_packed<4, LG>(L, sl, (int)header_offset(p.d, 4), cf, a_bias<4>(), acc, accz);
    else if (kind == 2)
      a_consume_packed<2, LG>(L, sl, (int)header_offset(p.d, 2), cf, a_bias<2>(), acc, accz);
    else
      a_consume_fp32x<LG>(L, sl, cf, acc);
  } else if (MX && !quant) {
    a_consume_fp32x<LG>(L, sl, cf, acc);
  } else if constexpr (BITS < 32) {
    a_consume_packed<BITS, LG>(L, sl, p.hoff, cf, bias, acc, accz);
  } else {
    const f32x2 c2 = f2_pack(cf, cf);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (k < L.nv) {
        const f32x2* xr = reinterpret_cast<const f32x2*>(sl + 16 * (L.gl + LG * k));
        acc[2 * k] = f2_fma(c2, xr[0], acc[2 * k]);
        acc[2 * k + 1] = f2_fma(c2, xr[1], acc[2 * k + 1]);
      }
    }
  }
}

// Write the lane's columns of row r: (acc + accz) * rs, through the ReLU
// gate when GATE (a separate instantiation: the gate's code changes the
// register allocation of the whole streaming loop).
template <int BITS, int LG, bool GATE>
__device__ __forceinline__ void a_flush(const SpmmParams& p, const ALane<LG>& L, int64_t r, float rs,
                                        const f32x2 (&acc)[8], float accz) {
  float o[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 v = f2_unpack(acc[i]);
    o[2 * i] = (v.x + accz) * rs;
    o[2 * i + 1] = (v.y + accz) * rs;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int col = a_col<BITS, LG>(L, 4 * k);
    if (col < p.d) {
      if (GATE) {
        const float4 g = gated4(p, r, col, make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]));
        o[4 * k] = g.x; o[4 * k + 1] = g.y; o[4 * k + 2] = g.z; o[4 * k + 3] = g.w;
      }
      if (p.Yb != nullptr)
        *reinterpret_cast<uint2*>(p.Yb + r * p.ldy + col) =
            make_uint2(pack_bf16x2(o[4 * k], o[4 * k + 1]), pack_bf16x2(o[4 * k + 2], o[4 * k + 3]));
      else
        st_f4(p.Y + r * p.ldy + col, o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
    }
  }
}

// Stream the edges [eb, eb + n) through the group's ring.  LIGHT: they are
// the edges of rows [row0, row1) and each row is written once its last edge
// has been consumed; otherwise the sums are left in acc / accz.
template <int BITS, int LG, int U, bool LIGHT, bool MX, bool GATE>
__device__ __forceinline__ void a_stream(const SpmmParams& p, const ALane<LG>& L, f32x2 bias, int eb, int n,
                                         int row0, int row1, f32x2 (&acc)[8], float& accz) {
  const float* __restrict__ colscale = p.colscale;
  const int nsteps = (n + U - 1) / U;
  uint32_t cx[kAS][U];
  float cf[kAS][U];
  bool mq[kAS][U];  // mixed rows: the gathered row is packed
  int kd[kAS][U];   // per-row widths (BITS == 0): the gathered row's kind
  // column ids two steps ahead: cp points at edge 2 U of the current step,
  // rem counts the edges from there to the end of the stream
  const int32_t* __restrict__ cp = p.col + eb;
#pragma unroll
  for (int t = 0; t < U; ++t) {
    cx[0][t] = t < n ? (uint32_t)__ldg(cp + t) : 0u;
    cx[1][t] = U + t < n ? (uint32_t)__ldg(cp + U + t) : 0u;
  }
  cp += 2 * U;
  int rem = n - 2 * U;
  // mixed rows: mask bits of the next step to issue, loaded one step ahead
  bool mqn[U];
#pragma unroll
  for (int t = 0; t < U; ++t) mqn[t] = MX && t < n && __ldg(p.mask + cx[0][t]) != 0;
  // light rows: end of the current row and of the next (relative to eb),
  // and their output scales, one row ahead
  int row = row0;
  int rend = 0, rnext = 0;
  float rs = 1.0f, rsn = 1.0f;
  if (LIGHT) {
    rend = __ldg(p.rowptr + row0 + 1) - eb;
    rnext = row0 + 2 <= row1 ? __ldg(p.rowptr + row0 + 2) - eb : 0x7fffffff;
    if (p.rowscale) {
      rs = __ldg(p.rowscale + row0);
      rsn = row0 + 1 < row1 ? __ldg(p.rowscale + row0 + 1) : 1.0f;
    }
  }
  for (int s0 = 0; s0 < nsteps + kAS - 1; s0 += kAS) {
#pragma unroll
    for (int j = 0; j < kAS; ++j) {
      const int s = s0 + j;
      __syncwarp(L.gmask);  // stage j was consumed in the previous step
      if (s < nsteps) {
#pragma unroll
        for (int t = 0; t < U; ++t) cx[(j + 2) % kAS][t] = t < rem ? (uint32_t)__ldg(cp + t) : 0u;
        if (MX) {
#pragma unroll
          for (int t = 0; t < U; ++t) {
            mq[j][t] = mqn[t];
            mqn[t] = t < rem + U && __ldg(p.mask + cx[(j + 1) % kAS][t]) != 0;  // edge (s + 1) U + t
          }
        }
        cp += U;
        rem -= U;
#pragma unroll
        for (int t = 0; t < U; ++t) {
          if (U == 1 || t < rem + 3 * U) {  // edge s U + t exists
            const uint32_t x = cx[j][t];
            cf[j][t] = colscale != nullptr ? __ldg(colscale + x) : 1.0f;
            const uint32_t dst = L.sring + (j * U + t) * kSlot<BITS, LG, MX>;
            const uint8_t* src = L.src + (size_t)x * L.stride;
            if constexpr (BITS == 0) {
              // the row's own width: the whole packed row at its offset, or the fp32 row
              const uint32_t b = __ldg(p.rbits + x);
              const int kind = (b == 2u || b == 4u || b == 8u) ? (int)b : 0;
              kd[j][t] = kind;
              if (kind == 0) {
                const uint8_t* sx = L.srcx + (size_t)x * L.stridex;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  if (k < L.nvm) cp_async16(dst + 64 * L.gl + 16 * (k ^ L.swz), sx + 16 * k);
              } else {
                const int sh = 2 * (kind == 2 ? 0 : (kind == 4 ? 1 : 2));
                const uint8_t* sp = p.packed + __ldg(p.roff + x) + 16 * L.gl;
                if ((L.hasw >> sh) & 1u) cp_async16(dst + 16 * L.gl, sp);
                if ((L.hasw >> (sh + 1)) & 1u) cp_async16(dst + 16 * (L.gl + LG), sp + 16 * LG);
              }
            } else if (MX && !mq[j][t]) {
              const uint8_t* sx = L.srcx + (size_t)x * L.stridex;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                if (k < L.nvm) cp_async16(dst + 64 * L.gl + 16 * (k ^ L.swz), sx + 16 * k);
            } else if constexpr (BITS < 32) {
              if (L.has0) cp_async16(dst + 16 * L.gl, src);
              if (kPiecesPerLane<BITS> > 1 && L.has1) cp_async16(dst + 16 * (L.gl + LG), src + 16 * LG);
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                if (k < L.nv) cp_async16(dst + 16 * (L.gl + LG * k), src + 16 * LG * k);
            }
          }
        }
      }
      cp_commit();
      const int c = s - (kAS - 1);
      if (c >= 0 && c < nsteps) {
        cp_wait<kAS - 1>();
        __syncwarp(L.gmask);  // every lane's pieces of the slot have landed
        const int jc = (j + 1) % kAS;
#pragma unroll
        for (int t = 0; t < U; ++t) {
          const int e = c * U + t;
          if (U == 1 || e < n) {
            if (LIGHT) {
              while (e >= rend) {
                if (L.on) a_flush<BITS, LG, GATE>(p, L, row, rs, acc, accz);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0ull;
                accz = 0.0f;
                ++row;
                rend = rnext;
                rnext = row + 2 <= row1 ? __ldg(p.rowptr + row + 2) - eb : 0x7fffffff;
                rs = rsn;
                if (p.rowscale) rsn = row + 1 < row1 ? __ldg(p.rowscale + row + 1) : 1.0f;
              }
            }
            if (L.on)
              a_consume<BITS, LG, MX>(p, L, L.ring + (jc * U + t) * kSlot<BITS, LG, MX>, MX && mq[jc][t],
                                      BITS == 0 ? kd[jc][t] : 0, cf[jc][t], bias, acc, accz);
          }
        }
      }
    }
  }
  if (LIGHT) {
    for (; row < row1; ++row) {
      if (L.on) a_flush<BITS, LG, GATE>(p, L, row, p.rowscale ? __ldg(p.rowscale + row) : 1.0f, acc, accz);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0ull;
      accz = 0.0f;
    }
  }
}

template <int BITS, int LG, int U, bool MX, bool GATE>
__global__ void __launch_bounds__(kSpmmThreads) spmm_async_kernel(const SpmmParams p) {
  extern __shared__ __align__(16) uint8_t asm_[];
  constexpr int NG = 32 / LG;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane / LG;
  ALane<LG> L;
  L.gl = lane % LG;
  constexpr int SLOT = kSlot<BITS, LG, MX>;
  L.ring = asm_ + (w * NG + g) * (kAS * U * SLOT);
  L.sring = sm_addr(L.ring);
  L.gmask = (LG == 32 ? 0xffffffffu : ((1u << LG) - 1u)) << (g * LG);
  const int pieces = BITS > 0 && BITS < 32 ? (int)(p.pitch / 16) : 0;
  L.has0 = L.gl < pieces;
  L.has1 = L.gl + LG < pieces;
  L.c0 = 16 * L.gl;
  L.hasw = 0u;
  if constexpr (BITS == 0) {
    // per-row widths: packed rows of any width and fp32 rows in the mixed layout
    L.on = L.c0 < p.d;
    L.nv = 0;
    L.src = nullptr;
    L.stride = 0u;
    L.srcx = reinterpret_cast<const uint8_t*>(p.X + L.c0);
    L.stridex = (uint32_t)(p.ldx * 4);
    L.nvm = max(0, min(4, (p.d - L.c0) / 4));
    L.swz = (L.gl >> 1) & 3;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int pw = (int)(packed_pitch(p.d, 2 << i) / 16);
      L.hasw |= (uint32_t)(L.gl < pw) << (2 * i) | (uint32_t)(L.gl + LG < pw) << (2 * i + 1);
    }
  } else if constexpr (BITS < 32) {
    L.on = L.c0 < p.d;
    L.nv = 0;
    L.src = p.packed + 16 * L.gl;
    L.stride = (uint32_t)p.pitch;
    L.srcx = MX ? reinterpret_cast<const uint8_t*>(p.X + L.c0) : nullptr;
    L.stridex = MX ? (uint32_t)(p.ldx * 4) : 0u;
    L.nvm = MX ? max(0, min(4, (p.d - L.c0) / 4)) : 0;
    L.swz = (L.gl >> 1) & 3;
  } else {
    L.src = reinterpret_cast<const uint8_t*>(p.X + 4 * L.gl);
    L.stride = (uint32_t)(p.ldx * 4);
    const int nq = p.d / 4;  // 4-column pieces of a row
    L.nv = L.gl < nq ? min(4, (nq - L.gl + LG - 1) / LG) : 0;
    L.on = L.nv > 0;
  }
  const f32x2 bias = a_bias<BITS>();
  f32x2 acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0ull;
  float accz = 0.0f;
  if ((int64_t)blockIdx.x < p.n_tasks) {
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.tasks) + blockIdx.x);
    const int sid = w * NG + g;
    const int len = task.z - task.y;
    int chunk = (len + kSpmmWarps * NG - 1) / (kSpmmWarps * NG);
    chunk = (chunk + U - 1) / U * U;
    const int b0 = task.y + sid * chunk;
    const int b1 = min(b0 + chunk, task.z);
    if (b0 < b1) a_stream<BITS, LG, U, false, MX, GATE>(p, L, bias, b0, b1 - b0, 0, 0, acc, accz);
    float o[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 v = f2_unpack(acc[i]);
      o[2 * i] = v.x + accz;
      o[2 * i + 1] = v.y + accz;
    }
#pragma unroll
    for (int off = LG; off < 32; off <<= 1)
#pragma unroll
      for (int k = 0; k < 16; ++k) o[k] += __shfl_xor_sync(FULL, o[k], off);
    __syncthreads();  // every ring is drained: reuse the space for the warp partials
    float* part = reinterpret_cast<float*>(asm_);
    if (lane < LG && L.on)
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int col = a_col<BITS, LG>(L, k);
        if (col < p.d) part[w * p.d + col] = o[k];
      }
    __syncthreads();
    finish_heavy(p, task, part);
    return;
  }
  const int64_t gid = ((int64_t)blockIdx.x - p.n_tasks) * kSpmmWarps * NG + w * NG + g;
  const int64_t ngroups = ((int64_t)gridDim.x - p.n_tasks) * kSpmmWarps * NG;
  for (int64_t t = gid; t < p.n_light; t += ngroups) {
    const int2 run = __ldg(reinterpret_cast<const int2*>(p.light) + t);
    const int eb = __ldg(p.rowptr + run.x), ee = __ldg(p.rowptr + run.y);
    a_stream<BITS, LG, U, true, MX, GATE>(p, L, bias, eb, ee - eb, run.x, run.y, acc, accz);
  }
}

template <int BITS, int LG, int U, bool MX, bool GATE>
int launch_async_g(const SpmmParams& p, cudaStream_t s) {
  constexpr int NG = 32 / LG;
  constexpr int SLOT = kSlot<BITS, LG, MX>;
  static_assert(BITS == 32 || BITS == 0 || kSlot<BITS, LG, false> / 16 <= kPiecesPerLane<BITS> * LG,
                "row pieces exceed the lanes' share");
  if (BITS > 0 && BITS < 32 && p.pitch > kSlot<BITS, LG, false>) return GQ_ERR_UNSUPPORTED;
  if ((BITS == 32 || BITS == 0 || MX) && 4 * p.d > SLOT) return GQ_ERR_UNSUPPORTED;
  // per-row widths: a row of width 8 (the widest) takes at most two pieces per lane
  if (BITS == 0 && packed_pitch(p.d, 8) > 32 * LG) return GQ_ERR_UNSUPPORTED;
  size_t smem = (size_t)kSpmmWarps * NG * kAS * U * SLOT;
  const size_t part = sizeof(float) * kSpmmWarps * p.d;
  if (smem < part) smem = part;
  auto kern = spmm_async_kernel<BITS, LG, U, MX, GATE>;
  // (the kernel also holds a few bytes of static shared memory)
  if (smem > 32 * 1024) GQ_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSpmmThreads, smem) != cudaSuccess || per_sm < 1)
    return GQ_ERR_UNSUPPORTED;
  int64_t light = (int64_t)sm_count() * per_sm;
  const int64_t need = (p.n_light + kSpmmWarps * NG - 1) / (kSpmmWarps * NG);
  if (light > need) light = need;
  if (light < 1) light = 1;
  const int64_t grid = p.n_tasks + light;
  if (grid > 0x7fffffff) return GQ_ERR_UNSUPPORTED;
  kern<<<(unsigned)grid, kSpmmThreads, smem, s>>>(p);
  return launch_status();
}

template <int BITS, int LG, int U, bool MX>
int launch_async(const SpmmParams& p, cudaStream_t s) {
  return p.gate != nullptr ? launch_async_g<BITS, LG, U, MX, true>(p, s) : launch_async_g<BITS, LG, U, MX, false>(p, s);
}

template <int BITS, int U, bool MX>
int launch_async_d(const SpmmParams& p, cudaStream_t s) {
  if (p.d <= 16) return launch_async<BITS, 1, U, MX>(p, s);
  if (p.d <= 32) return launch_async<BITS, 2, U, MX>(p, s);
  if (p.d <= 64) return launch_async<BITS, 4, U, MX>(p, s);
  if (p.d <= 128) return launch_async<BITS, 8, U, MX>(p, s);
  if (p.d <= 256) return launch_async<BITS, 16, U, MX>(p, s);
  return launch_async<BITS, 32, U, MX>(p, s);
}

// Coefficient-mode aggregation with d <= 512.  One kind of message row
// (all packed, or all fp32): packed rows keep two edges per stage; a mask
// mixing packed and fp32 rows: one edge per stage in fp32-sized slots.
int launch_async_any(const SpmmParams& p, int bits, cudaStream_t s) {
  const bool mx = bits < 32 && p.mask != nullptr;
  switch (bits) {
    case 2: return mx ? launch_async_d<2, 1, true>(p, s) : launch_async_d<2, 2, false>(p, s);
    case 4: return mx ? launch_async_d<4, 1, true>(p, s) : launch_async_d<4, 2, false>(p, s);
    case 8: return mx ? launch_async_d<8, 1, true>(p, s) : launch_async_d<8, 2, false>(p, s);
    default: return launch_async_d<32, 1, false>(p, s);
  }
}

template <int BITS, int G, int CPL, int LG, int EW, bool ALLQ>
int launch_cfg(SpmmParams p, cudaStream_t s) {
  const size_t smem = sizeof(float) * kSpmmWarps * p.d;
  const int64_t rows_blocks = (p.n_rows + kSpmmWarps - 1) / kSpmmWarps;
  int64_t grid = (int64_t)sm_count() * 8;
  if (grid > rows_blocks) grid = rows_blocks;
  if (grid < 1) grid = 1;
  grid += p.n_tasks;
  if (grid > 0x7fffffff) return GQ_ERR_UNSUPPORTED;
  spmm_kernel<BITS, G, CPL, LG, EW, ALLQ><<<(unsigned)grid, kSpmmThreads, smem, s>>>(p);
  return launch_status();
}

template <int BITS, int EW, bool ALLQ>
int launch_bits(const SpmmParams& p, cudaStream_t s) {
  if (p.d <= 16) return launch_cfg<BITS, 4, 1, 1, EW, ALLQ>(p, s);
  if (p.d <= 32) return launch_cfg<BITS, 4, 1, 2, EW, ALLQ>(p, s);
  if (p.d <= 64) return launch_cfg<BITS, 8, 1, 4, EW, ALLQ>(p, s);
  if (p.d <= 128) return launch_cfg<BITS, 16, 1, 8, EW, ALLQ>(p, s);
  if (p.d <= 256) return launch_cfg<BITS, 32, 1, 16, EW, ALLQ>(p, s);
  if (p.d <= 512) return launch_cfg<BITS, 32, 2, 32, EW, ALLQ>(p, s);
  return launch_cfg<BITS, 32, 4, 0, EW, ALLQ>(p, s);
}

template <int EW>
int launch_any(const SpmmParams& p, int bits, cudaStream_t s) {
  switch (bits) {
    case 2: return launch_bits<2, EW, false>(p, s);
    case 4: return launch_bits<4, EW, false>(p, s);
    case 8: return launch_bits<8, EW, false>(p, s);
    default: return launch_bits<32, EW, false>(p, s);
  }
}


// Bytes of an edge slot of the bulk-copy ring: a whole fp32 row of the width
// bucket (d <= 32 CPL), which also holds any packed row of that bucket.
template <int CPL>
constexpr int kBSlot = 128 * CPL;

// Four 8-bit codes (one word, column order) as the floats 2^23 + q.
__device__ __forceinline__ void codes4_b8(uint32_t w, float (&v)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(__byte_perm(w, kMagicBits, 0x7540u | i));
}

// Coefficient and row kind of the lane's edge of a batch: kind 0 = an fp32
// row, else the packed row's bit-width.  BITS == 0: every row has its own
// width (mixed packed rows; widths other than 2, 4, 8 mean fp32), and `off`
// is the packed row's byte offset.
template <int BITS, bool MX>
__device__ __forceinline__ void r_meta(const SpmmParams& p, uint32_t x, bool valid, float& cf, uint32_t& kind,
                                       int64_t& off) {
  cf = 1.0f;
  kind = (BITS > 0 && BITS < 32 && !MX) ? BITS : 0;
  off = 0;
  if (valid) {
    if (p.colscale != nullptr) cf = __ldg(p.colscale + x);
    if constexpr (BITS == 0) {
      const uint32_t b = __ldg(p.rbits + x);
      kind = (b == 2 || b == 4 || b == 8) ? b : 0;
      if (kind != 0) off = __ldg(p.roff + x);
    } else if (MX) {
      kind = __ldg(p.mask + x) != 0 ? BITS : 0;
    }
  }
}

// acc[2 k], acc[2 k + 1] += cs * (q - c) for piece k (4 columns) of a packed
// row in a slot: the lane's codes of the piece (one byte for b = 2, two for
// b = 4, four for b = 8) become the floats 2^23 + q (a byte permute, or a
// mask and an or), and one paired subtraction of 2^23 + c leaves q - c.
template <int BITS, int CPL>
__device__ __forceinline__ void bf_packed(const uint8_t* sl, f32x2 cs2, f32x2 bias, f32x2 (&acc)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < CPL / 4; ++k) {
    float v[4];
    if constexpr (BITS == 2) {
      const uint32_t w = sl[32 * k + lane];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(kMagicBits | ((w >> (2 * i)) & 3u));
    } else if constexpr (BITS == 4) {
      const uint32_t w = *reinterpret_cast<const uint16_t*>(sl + 64 * k + 2 * lane);
      const uint32_t lo = w & 0x0F0Fu, hi = (w >> 4) & 0x0F0Fu;  // codes 0, 2 / 1, 3 in bytes 0, 1
      v[0] = __uint_as_float(__byte_perm(lo, kMagicBits, 0x7540u));
      v[1] = __uint_as_float(__byte_perm(hi, kMagicBits, 0x7540u));
      v[2] = __uint_as_float(__byte_perm(lo, kMagicBits, 0x7541u));
      v[3] = __uint_as_float(__byte_perm(hi, kMagicBits, 0x7541u));
    } else {
      codes4_b8(*reinterpret_cast<const uint32_t*>(sl + 128 * k + 4 * lane), v);
    }
    acc[2 * k] = f2_fma(cs2, f2_add(f2_pack(v[0], v[1]), bias), acc[2 * k]);
    acc[2 * k + 1] = f2_fma(cs2, f2_add(f2_pack(v[2], v[3]), bias), acc[2 * k + 1]);
  }
}

// The lane's columns of (acc + accz) * s, written to row r of Y / Yb, or to
// `part` (an fp32 partial row) when it is not null.
template <int CPL>
__device__ __forceinline__ void bf_write(const SpmmParams& p, bool a_on, bool b_on, int64_t r, float s, float* part,
                                         const f32x2 (&acc)[4], float accz) {
  const int c0 = 4 * (threadIdx.x & 31);
#pragma unroll
  for (int k = 0; k < CPL / 4; ++k) {
    if (k == 0 ? a_on : b_on) {
      const float2 u = f2_unpack(acc[2 * k]), v = f2_unpack(acc[2 * k + 1]);
      float o0 = (u.x + accz) * s, o1 = (u.y + accz) * s, o2 = (v.x + accz) * s, o3 = (v.y + accz) * s;
      const int c = c0 + 128 * k;
      if (part == nullptr && p.gate != nullptr) {
        const float4 g = gated4(p, r, c, make_float4(o0, o1, o2, o3));
        o0 = g.x; o1 = g.y; o2 = g.z; o3 = g.w;
      }
      if (part != nullptr)
        st_f4(part + c, o0, o1, o2, o3);
      else if (p.Yb != nullptr)
        *reinterpret_cast<uint2*>(p.Yb + r * p.ldy + c) = make_uint2(pack_bf16x2(o0, o1), pack_bf16x2(o2, o3));
      else
        st_f4(p.Y + r * p.ldy + c, o0, o1, o2, o3);
    }
  }
}

// ---------------------------------------------------------------------------
// Bulk-copy ring aggregation (rows of mixed widths, 64 < d <= 256).
//
// Warp-per-edge consumption as in spmm_warp_kernel, with the gathers
// done by the bulk-copy engine: the lane that holds an edge's metadata
// copies the whole message row (d*4 bytes of an fp32 row, or the packed row
// with its header) into one of the warp's R shared-memory slots with a
// single cp.async.bulk that completes on the slot's mbarrier, and stores the
// edge's coefficient and kind beside the slot.  The warp consumes the edges
// in order, waiting on each slot's barrier (a bounded wait: on timeout it
// records a code in the graph's status word, waits again, boundedly, for the
// copies it still has in flight and gives up the rest of its work); after
// every H edges consumed, the H freed slots are refilled with the edges R
// ahead, one lane each.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
struct BLane {
  const uint8_t* xb;   // fp32 rows (row 0)
  const uint8_t* pb;   // packed rows (row 0)
  uint32_t xstride, xbytes, pitch;
  int d;
  uint32_t sring;      // the warp's slots (shared address)
  const uint8_t* ring;
  uint32_t sbar;       // the warp's R barriers
  float2* meta;        // the warp's R {coefficient, kind} entries
  uint32_t used;       // edges this warp streamed before (slot use count)
  bool a_on, b_on;
  bool failed;
};

// Issue the wave of edges [f0, f0 + H) (f0 a multiple of H) from the batch
// registers of the lanes holding them.
template <int BITS, bool MX, int R, int H, int SLOT>
__device__ __forceinline__ void b_issue(BLane& L, int f0, int n, uint32_t x, uint32_t kind, float cf, int64_t off) {
  const int lane = threadIdx.x & 31;
  const int l0 = f0 & 31;
  const int f = f0 - l0 + lane;
  if (lane >= l0 && lane < l0 + H && f < n) {
    const uint32_t slot = (L.used + (uint32_t)f) & (R - 1);
    const bool quant = BITS < 32 && kind != 0;
    L.meta[slot] = make_float2(cf, (float)kind);
    uint32_t bytes = L.xbytes;
    const uint8_t* src = L.xb + (size_t)(x * (uint64_t)L.xstride);
    if (quant) {
      if constexpr (BITS == 0) {
        bytes = (uint32_t)packed_pitch(L.d, (int)kind);
        src = L.pb + off;
      } else {
        bytes = L.pitch;
        src = L.pb + (size_t)(x * (uint64_t)L.pitch);
      }
    }
    const uint32_t bar = L.sbar + 8 * slot;
    bar_expect_tx(bar, bytes);
    bulk_g2s(L.sring + slot * SLOT, src, bytes, bar);
  }
}

// Stream the edges [eb, eb + n).  LIGHT: they are the edges of rows
// [row0, row1), each row written once its last edge is consumed; otherwise
// the sums are left in acc / accz.
template <int BITS, int CPL, bool MX, int R, int H, bool LIGHT>
__device__ __forceinline__ void b_stream(const SpmmParams& p, BLane& L, f32x2 bias, int eb, int n, int row0,
                                         int row1, f32x2 (&acc)[4], float& accz) {
  static_assert(R <= 32 && 32 % H == 0 && R % H == 0 && (R & (R - 1)) == 0, "ring shape");
  constexpr int SLOT = kBSlot<CPL>;
  const int lane = threadIdx.x & 31;
  const int32_t* __restrict__ col = p.col + eb;
  // lane i: edge kb + i (x0, q0, cf0) and kb + 32 + i (x1, q1, cf1); the
  // column id of kb + 64 + i (x2)
  uint32_t x0 = lane < n ? (uint32_t)__ldg(col + lane) : 0u;
  uint32_t x1 = 32 + lane < n ? (uint32_t)__ldg(col + 32 + lane) : 0u;
  uint32_t x2 = 64 + lane < n ? (uint32_t)__ldg(col + 64 + lane) : 0u;
  float cf0, cf1;
  uint32_t q0, q1;
  int64_t o0, o1;
  r_meta<BITS, MX>(p, x0, lane < n, cf0, q0, o0);
  r_meta<BITS, MX>(p, x1, 32 + lane < n, cf1, q1, o1);
  int kb = 0;
  int rb = row0, ri = 0, rend = 0x7fffffff, rpl = 0x7fffffff;
  float rsl = 1.0f;
  if (LIGHT) {
    if (row0 + lane < row1) {
      rpl = __ldg(p.rowptr + row0 + 1 + lane) - eb;
      if (p.rowscale) rsl = __ldg(p.rowscale + row0 + lane);
    }
    rend = __shfl_sync(FULL, rpl, 0);
  }
  // fill the ring (the first R edges are all in batch 0)
#pragma unroll
  for (int f0 = 0; f0 < R; f0 += H)
    if (f0 < n) b_issue<BITS, MX, R, H, SLOT>(L, f0, n, x0, q0, cf0, o0);
  int issued = min(R, n);
  int e = 0;
  for (; e < n; ++e) {
    if (e == kb + 32) {  // the consumer enters the next batch
      kb += 32;
      x0 = x1;
      q0 = q1;
      cf0 = cf1;
      o0 = o1;
      x1 = x2;
      r_meta<BITS, MX>(p, x1, kb + 32 + lane < n, cf1, q1, o1);
      x2 = kb + 64 + lane < n ? (uint32_t)__ldg(col + kb + 64 + lane) : 0u;
    }
    const uint32_t u = L.used + (uint32_t)e;
    const uint32_t slot = u & (R - 1);
    if (!__all_sync(FULL, mbar_wait_u32(L.sbar + 8 * slot, (u / R) & 1u))) {  // a warp-wide verdict
      L.failed = true;
      break;
    }
    const float2 mt = L.meta[slot];
    if (LIGHT) {
      while (e >= rend) {
        bf_write<CPL>(p, L.a_on, L.b_on, rb + ri, __shfl_sync(FULL, rsl, ri), nullptr, acc, accz);
#pragma unroll
        for (int i = 0; i < CPL / 2; ++i) acc[i] = 0ull;
        accz = 0.0f;
        if (++ri == 32) {
          rb += 32;
          ri = 0;
          rpl = 0x7fffffff;
          rsl = 1.0f;
          if (rb + lane < row1) {
            rpl = __ldg(p.rowptr + rb + 1 + lane) - eb;
            if (p.rowscale) rsl = __ldg(p.rowscale + rb + lane);
          }
        }
        rend = __shfl_sync(FULL, rpl, ri);
      }
    }
    const uint8_t* sl = L.ring + slot * SLOT;
    if (BITS == 0 && mt.y != 0.0f) {
      // a packed row of its own width b: header at its own offset, c = 2^(b-1)
      const int b = (int)mt.y;
      const float c = (float)(1 << (b - 1));
      const float2 h = *reinterpret_cast<const float2*>(sl + header_offset(p.d, b));
      accz = __fmaf_rn(mt.x, __fmaf_rn(c, h.x, h.y), accz);
      const float cs = mt.x * h.x;
      const f32x2 bz = f2_pack(-(kMagic + c), -(kMagic + c));
      if (b == 2)
        bf_packed<2, CPL>(sl, f2_pack(cs, cs), bz, acc);
      else if (b == 4)
        bf_packed<4, CPL>(sl, f2_pack(cs, cs), bz, acc);
      else
        bf_packed<8, CPL>(sl, f2_pack(cs, cs), bz, acc);
    } else if (BITS > 0 && BITS < 32 && mt.y != 0.0f) {
      constexpr float c = (float)(1 << ((BITS > 0 && BITS < 32 ? BITS : 8) - 1));
      const float2 h = *reinterpret_cast<const float2*>(sl + p.hoff);
      accz = __fmaf_rn(mt.x, __fmaf_rn(c, h.x, h.y), accz);
      const float cs = mt.x * h.x;
      bf_packed<BITS, CPL>(sl, f2_pack(cs, cs), bias, acc);
    } else {
      const f32x2 c2 = f2_pack(mt.x, mt.x);
      const f32x2* a = reinterpret_cast<const f32x2*>(sl + 16 * lane);
      acc[0] = f2_fma(c2, a[0], acc[0]);
      acc[1] = f2_fma(c2, a[1], acc[1]);
      if (CPL == 8) {
        acc[2] = f2_fma(c2, a[64], acc[2]);
        acc[3] = f2_fma(c2, a[65], acc[3]);
      }
    }
    const int f0 = e + 1 - H + R;  // refill wave, once H slots are free
    if (((e + 1) & (H - 1)) == 0 && f0 < n) {
      __syncwarp();  // every lane is done with the freed slots
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (f0 >= kb + 32)
        b_issue<BITS, MX, R, H, SLOT>(L, f0, n, x1, q1, cf1, o1);
      else
        b_issue<BITS, MX, R, H, SLOT>(L, f0, n, x0, q0, cf0, o0);
      issued = min(f0 + H, n);
    }
  }
  if (L.failed) {
    // record the failure, then wait (boundedly) for the copies still in flight
    if (lane == 0 && p.err != nullptr) atomicCAS(p.err, 0, kWaitCodeAggregation);
    for (int f = e; f < issued; ++f) {
      const uint32_t u = L.used + (uint32_t)f;
      mbar_wait_u32(L.sbar + 8 * (u & (R - 1)), (u / R) & 1u);
    }
    return;
  }
  L.used += (uint32_t)n;
  if (LIGHT) {
    // the last row, and any rows without edges after it
    while (rb + ri < row1) {
      bf_write<CPL>(p, L.a_on, L.b_on, rb + ri, __shfl_sync(FULL, rsl, ri), nullptr, acc, accz);
#pragma unroll
      for (int i = 0; i < CPL / 2; ++i) acc[i] = 0ull;
      accz = 0.0f;
      if (++ri == 32) {
        rb += 32;
        ri = 0;
        rsl = 1.0f;
        if (rb + lane < row1 && p.rowscale) rsl = __ldg(p.rowscale + rb + lane);
      }
    }
  }
}

template <int BITS, int CPL, bool MX, int R, int H>
__global__ void __launch_bounds__(kSpmmThreads, 3) spmm_bulk_kernel(const SpmmParams p) {
  extern __shared__ __align__(128) uint8_t bsm[];
  constexpr int SLOT = kBSlot<CPL>;
  constexpr int HDR = kSpmmWarps * R * 16;  // barriers and {coefficient, kind} entries of all warps
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  BLane L;
  L.xb = reinterpret_cast<const uint8_t*>(p.X);
  L.pb = p.packed;
  L.xstride = (uint32_t)(p.ldx * 4);
  L.xbytes = (uint32_t)(p.d * 4);
  L.pitch = (uint32_t)p.pitch;
  L.d = p.d;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bsm) + w * R;
  L.sbar = sm_addr(bars);
  L.meta = reinterpret_cast<float2*>(bsm + kSpmmWarps * R * 8) + w * R;
  L.ring = bsm + HDR + w * (R * SLOT);
  L.sring = sm_addr(L.ring);
  L.used = 0;
  L.a_on = 4 * lane < p.d;
  L.b_on = CPL == 8 && 128 + 4 * lane < p.d;
  L.failed = false;
  if (lane < R) bar_init(L.sbar + 8 * lane, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  const f32x2 bias = a_bias<BITS>();
  f32x2 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0ull;
  float accz = 0.0f;
  if ((int64_t)blockIdx.x < p.n_tasks) {
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.tasks) + blockIdx.x);
    const int len = task.z - task.y;
    const int chunk = (len + kSpmmWarps - 1) / kSpmmWarps;
    const int b0 = task.y + w * chunk;
    const int b1 = min(b0 + chunk, task.z);
    if (b0 < b1) b_stream<BITS, CPL, MX, R, H, false>(p, L, bias, b0, b1 - b0, 0, 0, acc, accz);
    __syncthreads();  // every ring is drained: reuse the slots for the warp partials
    float* part = reinterpret_cast<float*>(bsm + HDR);
#pragma unroll
    for (int i = 0; i < CPL / 2; ++i) {
      const float2 v = f2_unpack(acc[i]);
      const int c = 4 * lane + 128 * (i >> 1) + 2 * (i & 1);
      if ((i >> 1) == 0 ? L.a_on : L.b_on) {
        part[w * p.d + c] = v.x + accz;
        part[w * p.d + c + 1] = v.y + accz;
      }
    }
    __syncthreads();
    finish_heavy(p, task, part);
    return;
  }
  const int64_t gw = ((int64_t)blockIdx.x - p.n_tasks) * kSpmmWarps + w;
  const int64_t nw = ((int64_t)gridDim.x - p.n_tasks) * kSpmmWarps;
  for (int64_t t = gw; t < p.n_light && !L.failed; t += nw) {
    const int2 run = __ldg(reinterpret_cast<const int2*>(p.light) + t);
    const int eb = __ldg(p.rowptr + run.x), ee = __ldg(p.rowptr + run.y);
    b_stream<BITS, CPL, MX, R, H, true>(p, L, bias, eb, ee - eb, run.x, run.y, acc, accz);
  }
}

template <int BITS, int CPL, bool MX, int R, int H>
int launch_bulk(const SpmmParams& p, cudaStream_t s) {
  constexpr int SLOT = kBSlot<CPL>;
  if (BITS < 32 && p.pitch > SLOT) return GQ_ERR_UNSUPPORTED;
  if (4 * p.d > SLOT) return GQ_ERR_UNSUPPORTED;
  auto kern = spmm_bulk_kernel<BITS, CPL, MX, R, H>;
  size_t smem = (size_t)kSpmmWarps * R * (16 + SLOT);
  const size_t part = kSpmmWarps * R * 16 + sizeof(float) * kSpmmWarps * p.d;
  if (smem < part) smem = part;
  if (smem > 48 * 1024) GQ_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSpmmThreads, smem) != cudaSuccess || per_sm < 1)
    return GQ_ERR_UNSUPPORTED;
  int64_t light = (int64_t)sm_count() * per_sm;
  const int64_t need = (p.n_light + kSpmmWarps - 1) / kSpmmWarps;
  if (light > need) light = need;
  if (light < 1) light = 1;
  const int64_t grid = p.n_tasks + light;
  if (grid > 0x7fffffff) return GQ_ERR_UNSUPPORTED;
  kern<<<(unsigned)grid, kSpmmThreads, smem, s>>>(p);
  return launch_status();
}


// ---------------------------------------------------------------------------
// Warp-per-edge register aggregation (coefficient modes, 64 < d <= 256).
//
// The whole warp takes one edge at a time (so the packed-or-fp32 choice of
// a mixing mask is uniform across it); lane l owns the C = 4 or 8 columns
// [C l, C l + C) and loads its part of the gathered message row straight
// into registers with plain loads: C b / 8 bytes of codes plus the row's
// {S, Z}, or C floats.  U edges are loaded before any is consumed, and the
// kernel keeps few registers so that many warps per SM cover the latency
// (plain loads at high occupancy gather random rows several times faster
// than the bulk-copy and cp.async rings above).  Per batch of 32 edges,
// lane j loads edge j's column id, coefficient and kind once (the next
// batch's column ids one batch ahead) and the warp broadcasts them with
// shuffles; the kind rides in the sign of the coefficient.
// De-quantization as in the kernels above: a (q S + Z) = (a S)(q - c) +
// a (Z + c S), the code placed at bit offset o of the float 2^23 (one
// bitwise op), one paired subtraction of 2^23 + c 2^o and a paired FMA
// with a S 2^-o.
// ---------------------------------------------------------------------------

template <int BITS, bool MX, int C>
struct WSlot {
  static constexpr int NW = (BITS == 32 || MX) ? C : (C * BITS + 31) / 32;
  uint32_t w[NW];
  float2 h;
};

template <int C>
struct WLane {
  int c0;    // first owned column
  int nv;    // owned columns inside the row (a multiple of 4)
};

template <int BITS, bool MX, int C>
__device__ __forceinline__ void w_load(const SpmmParams& p, const WLane<C>& L, uint32_t x, bool packed,
                                       WSlot<BITS, MX, C>& s) {
  if constexpr (BITS < 32) {
    if (!MX || packed) {
      const uint8_t* row = p.packed + (size_t)x * (size_t)p.pitch;
      s.h = __ldg(reinterpret_cast<const float2*>(row + p.hoff));
      const uint8_t* pl = row + L.c0 * BITS / 8;
      // the lane's C * BITS / 8 bytes (2 .. 8, aligned to their size); a
      // partial last lane reads the same span, which stays inside the
      // payload padded to 8 bytes
      if constexpr (C * BITS == 64) {
        const uint2 t = __ldg(reinterpret_cast<const uint2*>(pl));
        s.w[0] = t.x;
        s.w[1] = t.y;
      } else if constexpr (C * BITS == 32) {
        s.w[0] = __ldg(reinterpret_cast<const uint32_t*>(pl));
      } else if constexpr (C * BITS == 16) {
        s.w[0] = __ldg(reinterpret_cast<const uint16_t*>(pl));
      } else {
        s.w[0] = __ldg(pl);
      }
      return;
    }
  }
  if constexpr (BITS == 32 || MX) {
    const float* xr = p.X + (size_t)x * (size_t)p.ldx + L.c0;
#pragma unroll
    for (int k = 0; k < C / 4; ++k) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (4 * k < L.nv) a = ldg_f4(xr + 4 * k);
      s.w[4 * k] = __float_as_uint(a.x); s.w[4 * k + 1] = __float_as_uint(a.y);
      s.w[4 * k + 2] = __float_as_uint(a.z); s.w[4 * k + 3] = __float_as_uint(a.w);
    }
  }
}

// acc += cf * m over the lane's C columns (acc[i] holds columns 2i, 2i + 1).
template <int BITS, bool MX, int C>
__device__ __forceinline__ void w_consume(const WSlot<BITS, MX, C>& s, bool packed, float cf, f32x2 (&acc)[C / 2],
                                          float& accz) {
  if constexpr (BITS < 32) {
    if (!MX || packed) {
      constexpr float c = (float)(1 << (BITS - 1));
      const float cs = cf * s.h.x;
      accz = __fmaf_rn(cf, __fmaf_rn(c, s.h.x, s.h.y), accz);
      if constexpr (BITS == 8) {
        const f32x2 cs2 = f2_pack(cs, cs);
        const f32x2 bias = f2_pack(-(kMagic + c), -(kMagic + c));
#pragma unroll
        for (int k = 0; k < C / 4; ++k) {
          const uint32_t w = s.w[k];
          const f32x2 v0 = f2_pack(__uint_as_float(__byte_perm(w, kMagicBits, 0x7540u)),
                                   __uint_as_float(__byte_perm(w, kMagicBits, 0x7541u)));
          const f32x2 v1 = f2_pack(__uint_as_float(__byte_perm(w, kMagicBits, 0x7542u)),
                                   __uint_as_float(__byte_perm(w, kMagicBits, 0x7543u)));
          acc[2 * k] = f2_fma(cs2, f2_add(v0, bias), acc[2 * k]);
          acc[2 * k + 1] = f2_fma(cs2, f2_add(v1, bias), acc[2 * k + 1]);
        }
      } else {
        // code i of the lane sits at bit BITS * i of w[0]; columns 2j, 2j + 1
        // at offsets o0 = 2 j BITS and o0 + BITS within their 16-bit half
        // word (a pair never straddles two halves), so q 2^o < 2^23
        constexpr uint32_t M = (1u << BITS) - 1u;
#pragma unroll
        for (int j = 0; j < C / 2; ++j) {
          const int o0 = (2 * j * BITS) & 15, o1 = o0 + BITS;
          const uint32_t hw = (2 * j * BITS) >= 16 ? (s.w[0] >> 16) : s.w[0];
          const f32x2 v = f2_pack(__uint_as_float(kMagicBits | (hw & (M << o0))),
                                  __uint_as_float(kMagicBits | (hw & (M << o1))));
          const f32x2 bias = f2_pack(-(kMagic + c * (float)(1 << o0)), -(kMagic + c * (float)(1 << o1)));
          const f32x2 sc = f2_pack(cs * (1.0f / (float)(1 << o0)), cs * (1.0f / (float)(1 << o1)));
          acc[j] = f2_fma(sc, f2_add(v, bias), acc[j]);
        }
      }
      return;
    }
  }
  if constexpr (BITS == 32 || MX) {
    const f32x2 c2 = f2_pack(cf, cf);
#pragma unroll
    for (int k = 0; k < C / 2; ++k)
      acc[k] = f2_fma(c2, f2_pack(__uint_as_float(s.w[2 * k]), __uint_as_float(s.w[2 * k + 1])), acc[k]);
  }
}

// The lane's columns of (acc + accz) * rs to row r of Y / Yb, or to the
// fp32 partial row `part`.
template <int C, bool GATE>
__device__ __forceinline__ void w_flush(const SpmmParams& p, const WLane<C>& L, int64_t r, float rs, float* part,
                                        const f32x2 (&acc)[C / 2], float accz, uint32_t gw = 0u) {
#pragma unroll
  for (int k = 0; k < C / 4; ++k) {
    if (4 * k < L.nv) {
      const float2 u = f2_unpack(acc[2 * k]), v = f2_unpack(acc[2 * k + 1]);
      float o0 = (u.x + accz) * rs, o1 = (u.y + accz) * rs, o2 = (v.x + accz) * rs, o3 = (v.y + accz) * rs;
      const int col = L.c0 + 4 * k;
      if (GATE && part == nullptr) {  // gw: the gate word of the lane's columns
        const uint32_t b = gw >> (col & 31);
        if (!(b & 1u)) o0 = 0.0f;
        if (!(b & 2u)) o1 = 0.0f;
        if (!(b & 4u)) o2 = 0.0f;
        if (!(b & 8u)) o3 = 0.0f;
      }
      if (part != nullptr)
        st_f4(part + col, o0, o1, o2, o3);
      else if (p.Yb != nullptr)
        *reinterpret_cast<uint2*>(p.Yb + r * p.ldy + col) = make_uint2(pack_bf16x2(o0, o1), pack_bf16x2(o2, o3));
      else
        st_f4(p.Y + r * p.ldy + col, o0, o1, o2, o3);
    }
  }
}

// The gate word holding the lane's columns of row r (C <= 8 columns, inside
// one 32-column word), loaded when the row becomes current so that its
// flush, many edges later, does not wait on it.
template <int C>
__device__ __forceinline__ uint32_t w_gate_word(const SpmmParams& p, const WLane<C>& L, int64_t r) {
  return L.nv > 0 ? __ldg(p.gate + r * p.ldg + (L.c0 >> 5)) : 0u;
}

// The coefficient of gathered row x with the row's kind in its sign bit
// (set: a packed row of a mixing mask); coefficients are >= 0.
template <int BITS, bool MX>
__device__ __forceinline__ float w_cfk(const SpmmParams& p, uint32_t x) {
  const float cf = p.colscale != nullptr ? __ldg(p.colscale + x) : 1.0f;
  if (MX && __ldg(p.mask + x) != 0) return __uint_as_float(__float_as_uint(cf) | 0x80000000u);
  return cf;
}
__device__ __forceinline__ bool w_packed_kind(float cfk) { return (__float_as_uint(cfk) >> 31) != 0; }
__device__ __forceinline__ float w_coef(float cfk) { return __uint_as_float(__float_as_uint(cfk) & 0x7fffffffu); }

// Stream the edges [eb, ee).  LIGHT: the edges of rows [row0, row1), each
// row written once its last edge is consumed; otherwise the sums are left
// in acc / accz.
template <int BITS, bool MX, int C, int U, bool LIGHT, int EW, bool GATE>
__device__ __forceinline__ void w_stream(const SpmmParams& p, const WLane<C>& L, int eb, int ee, int row0, int row1,
                                         f32x2 (&acc)[C / 2], float& accz) {
  const int lane = threadIdx.x & 31;
  const int32_t* __restrict__ col = p.col;
  const int head = EW ? (L.c0 >> p.fshift) : 0;  // the lane's columns lie in one head (F >= 16 >= C)
  // EW = 2 (8-bit attention codes, forward): {S, Z} of the current row's head
  float2 az = make_float2(0.0f, 0.0f);
  if (EW == 2 && L.nv > 0 && row0 < p.n_rows)
    az = __ldg(reinterpret_cast<const float2*>(p.ahdr) + (int64_t)row0 * p.heads + head);
  uint32_t xn = eb + lane < ee ? (uint32_t)__ldg(col + eb + lane) : 0u;  // column ids of the next batch
  int row = row0, rend = 0x7fffffff, rnext = 0x7fffffff;
  float rs = 1.0f, rsn = 1.0f;
  uint32_t gw = 0u;  // GATE: the gate word of the current row
  if (LIGHT) {
    if (GATE) gw = w_gate_word(p, L, row0);
    rend = __ldg(p.rowptr + row0 + 1);
    rnext = row0 + 1 < row1 ? __ldg(p.rowptr + row0 + 2) : 0x7fffffff;
    if (p.rowscale) {
      rs = __ldg(p.rowscale + row0);
      rsn = row0 + 1 < row1 ? __ldg(p.rowscale + row0 + 1) : 1.0f;
    }
  }
  for (int base = eb; base < ee; base += 32) {
    const uint32_t xb = xn;
    // coefficient (edge-weight modes: +-1) with the row's kind in its sign bit
    const float cb = base + lane < ee ? w_cfk<BITS, MX>(p, xb) : 1.0f;
    // edge-weight modes: the CSR edge id of each edge of the batch
    const int32_t eidb = EW && p.eperm != nullptr && base + lane < ee ? __ldg(p.eperm + base + lane) : base + lane;
    xn = base + 32 + lane < ee ? (uint32_t)__ldg(col + base + 32 + lane) : 0u;
    const int cnt = min(32, ee - base);
    for (int t0 = 0; t0 < cnt; t0 += U) {
      WSlot<BITS, MX, C> m[U];
      float cf[U];
      float aw[U];  // edge-weight modes: the attention weight (EW = 1) or code (EW = 2) of the lane's head
#pragma unroll
      for (int t = 0; t < U; ++t) {
        const uint32_t x = __shfl_sync(FULL, xb, (t0 + t) & 31);
        cf[t] = __shfl_sync(FULL, cb, (t0 + t) & 31);
        aw[t] = 0.0f;
        if (EW == 1) {
          const int32_t eid = __shfl_sync(FULL, eidb, (t0 + t) & 31);
          if (t0 + t < cnt && L.nv > 0) aw[t] = __ldg(p.alpha + (int64_t)eid * p.heads + head);
        } else if (EW == 2) {  // forward only: the edge id is the CSR position
          if (t0 + t < cnt && L.nv > 0)
            aw[t] = code_to_float(__ldg(p.acode + (int64_t)(base + t0 + t) * p.heads + head));
        }
        if (t0 + t < cnt && L.nv > 0) w_load<BITS, MX, C>(p, L, x, w_packed_kind(cf[t]), m[t]);
      }
#pragma unroll
      for (int t = 0; t < U; ++t) {
        if (t0 + t < cnt) {
          if (LIGHT) {
            while (base + t0 + t >= rend) {
              if (L.nv > 0) w_flush<C, GATE>(p, L, row, rs, nullptr, acc, accz, gw);
#pragma unroll
              for (int i = 0; i < C / 2; ++i) acc[i] = 0ull;
              accz = 0.0f;
              ++row;
              if (GATE && row < row1) gw = w_gate_word(p, L, row);
              rend = rnext;
              rnext = row + 1 < row1 ? __ldg(p.rowptr + row + 2) : 0x7fffffff;
              rs = rsn;
              if (p.rowscale) rsn = row + 1 < row1 ? __ldg(p.rowscale + row + 1) : 1.0f;
              if (EW == 2 && L.nv > 0 && row < row1)
                az = __ldg(reinterpret_cast<const float2*>(p.ahdr) + (int64_t)row * p.heads + head);
            }
          }
          const float coef = EW == 1 ? aw[t] : (EW == 2 ? __fmaf_rn(aw[t], az.x, az.y) : w_coef(cf[t]));
          if (L.nv > 0) w_consume<BITS, MX, C>(m[t], w_packed_kind(cf[t]), coef, acc, accz);
        }
      }
    }
  }
  if (LIGHT) {
    for (; row < row1; ++row) {
      if (L.nv > 0) w_flush<C, GATE>(p, L, row, p.rowscale ? __ldg(p.rowscale + row) : 1.0f, nullptr, acc, accz,
                                     GATE ? w_gate_word(p, L, row) : 0u);
#pragma unroll
      for (int i = 0; i < C / 2; ++i) acc[i] = 0ull;
      accz = 0.0f;
    }
  }
}

template <int BITS, bool MX, int C, int U, int MINB, int EW, bool GATE>
__global__ void __launch_bounds__(kSpmmThreads, MINB) spmm_warp_kernel(const SpmmParams p) {
  extern __shared__ __align__(16) float wpart[];  // [kSpmmWarps][d] for heavy rows
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  WLane<C> L;
  L.c0 = C * lane;
  L.nv = min(C, max(0, p.d - L.c0));
  f32x2 acc[C / 2];
#pragma unroll
  for (int i = 0; i < C / 2; ++i) acc[i] = 0ull;
  float accz = 0.0f;
  if ((int64_t)blockIdx.x < p.n_tasks) {
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.tasks) + blockIdx.x);
    const int len = task.z - task.y;
    const int chunk = (len + kSpmmWarps - 1) / kSpmmWarps;
    const int b0 = min(task.y + w * chunk, task.z);
    const int b1 = min(b0 + chunk, task.z);
    if (b0 < b1) w_stream<BITS, MX, C, U, false, EW, GATE>(p, L, b0, b1, task.x, task.x + 1, acc, accz);
    if (L.nv > 0) w_flush<C, GATE>(p, L, 0, 1.0f, wpart + w * p.d, acc, accz);
    __syncthreads();
    finish_heavy(p, task, wpart);
    return;
  }
  const int64_t gw = ((int64_t)blockIdx.x - p.n_tasks) * kSpmmWarps + w;
  const int64_t nw = ((int64_t)gridDim.x - p.n_tasks) * kSpmmWarps;
  for (int64_t t = gw; t < p.n_light; t += nw) {
    const int2 run = __ldg(reinterpret_cast<const int2*>(p.light) + t);
    const int eb = __ldg(p.rowptr + run.x), ee = __ldg(p.rowptr + run.y);
    w_stream<BITS, MX, C, U, true, EW, GATE>(p, L, eb, ee, run.x, run.y, acc, accz);
  }
}

template <int BITS, bool MX, int C, int U, int MINB, int EW, bool GATE>
int launch_warp_g(const SpmmParams& p, cudaStream_t s) {
  if (p.d > 32 * C || p.d % 4 != 0) return GQ_ERR_UNSUPPORTED;
  const size_t smem = sizeof(float) * kSpmmWarps * p.d;
  auto kern = spmm_warp_kernel<BITS, MX, C, U, MINB, EW, GATE>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSpmmThreads, smem) != cudaSuccess || per_sm < 1)
    return GQ_ERR_UNSUPPORTED;
  int64_t light = (int64_t)sm_count() * per_sm;
  const int64_t need = (p.n_light + kSpmmWarps - 1) / kSpmmWarps;
  if (light > need) light = need;
  if (light < 1) light = 1;
  const int64_t grid = p.n_tasks + light;
  if (grid > 0x7fffffff) return GQ_ERR_UNSUPPORTED;
  kern<<<(unsigned)grid, kSpmmThreads, smem, s>>>(p);
  return launch_status();
}

// The gate (coefficient mode only) is its own instantiation: its code in the
// row flush changes the register allocation of the whole edge loop.
template <int BITS, bool MX, int C, int U, int MINB, int EW = 0>
int launch_warp(const SpmmParams& p, cudaStream_t s) {
  if constexpr (EW == 0) {
    if (p.gate != nullptr) return launch_warp_g<BITS, MX, C, U, MINB, 0, true>(p, s);
  }
  return launch_warp_g<BITS, MX, C, U, MINB, EW, false>(p, s);
}

// 64 < d <= 256 on the warp-per-edge register kernel: 4 columns per lane and
// 4 edges in flight up to d = 128, 8 columns and 3 edges above; 4 blocks
// per SM (each measured the fastest of its range on the large GCN graph).
template <int BITS, bool MX, int EW>
int launch_warp_d(const SpmmParams& p, cudaStream_t s) {
  return p.d <= 128 ? launch_warp<BITS, MX, 4, 4, 4, EW>(p, s) : launch_warp<BITS, MX, 8, 3, 4, EW>(p, s);
}

// EW = 1: per-edge, per-head attention weights (fp32) instead of the
// per-source coefficient.
template <int EW>
int launch_warp_any(const SpmmParams& p, int bits, cudaStream_t s) {
  const bool mx = bits < 32 && p.mask != nullptr;
  switch (bits) {
    case 2: return mx ? launch_warp_d<2, true, EW>(p, s) : launch_warp_d<2, false, EW>(p, s);
    case 4: return mx ? launch_warp_d<4, true, EW>(p, s) : launch_warp_d<4, false, EW>(p, s);
    case 8: return mx ? launch_warp_d<8, true, EW>(p, s) : launch_warp_d<8, false, EW>(p, s);
    default: return launch_warp_d<32, false, EW>(p, s);
  }
}


}  // namespace

// Common argument checks and message-source setup.
size_t ws_bytes_for(const gq_sched& sc, int d) {
  if (sc.n_groups == 0) return 0;
  return ((size_t)sc.n_slots * d * sizeof(float) + 255) / 256 * 256 + (size_t)sc.n_groups * sizeof(int) + 256;
}

// The argument checks of the aggregation entry points (nothing launched).
int spmm_check(const gq_graph* g, const float* X, int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d,
               int bits, const float* Y, int64_t ldy, const void* Yb) {
  if (g == nullptr || (Y == nullptr && Yb == nullptr) || d < 1 || ldy < d) return GQ_ERR_INVALID_ARG;
  if (!(bits == 32 || valid_bits(bits))) return GQ_ERR_INVALID_ARG;
  if (d > 1024) return GQ_ERR_UNSUPPORTED;
  const bool all_packed = bits < 32 && mask == nullptr;
  if (!all_packed) {
    if (X == nullptr || ldx < d || d % 4 != 0 || ldx % 4 != 0 || !aligned(X, 16)) return GQ_ERR_INVALID_ARG;
  }
  if (bits < 32 && (packed == nullptr || !aligned(packed, 16))) return GQ_ERR_INVALID_ARG;
  if (Yb != nullptr) {
    if (d % 4 != 0 || ldy % 8 != 0 || !aligned(Yb, 16)) return GQ_ERR_INVALID_ARG;
  } else if (d % 4 != 0 || ldy % 4 != 0 || !aligned(Y, 16)) {
    return GQ_ERR_INVALID_ARG;
  }
  return GQ_OK;
}

int spmm_setup(const gq_graph* g, int transpose, const float* X, int64_t ldx, const uint8_t* packed,
               const uint8_t* mask, int d, int bits, float* Y, int64_t ldy, void* ws, size_t ws_bytes,
               cudaStream_t s, SpmmParams& p, void* Yb = nullptr) {
  GQ_TRY(spmm_check(g, X, ldx, packed, mask, d, bits, Y, ldy, Yb));
  p = SpmmParams{};
  p.rowptr = transpose ? g->tr_rowptr : g->rowptr;
  p.col = transpose ? g->tr_col : g->col;
  const gq_sched& sc = transpose ? g->tr_sched : g->sched;
  p.tasks = sc.tasks;
  p.groups = sc.groups;
  p.n_tasks = sc.n_tasks;
  p.light = sc.light;
  p.n_light = sc.n_light;
  p.hub_threshold = g->hub_threshold;
  p.err = g->status;
  if (sc.n_groups > 0) {
    if (ws == nullptr || ws_bytes < ws_bytes_for(sc, d) || !aligned(ws, 256)) return GQ_ERR_WORKSPACE;
    p.partial = static_cast<float*>(ws);
    p.tickets = reinterpret_cast<int*>(static_cast<char*>(ws) + ((size_t)sc.n_slots * d * sizeof(float) + 255) / 256 * 256);
    GQ_TRY_CUDA(cudaMemsetAsync(p.tickets, 0, (size_t)sc.n_groups * sizeof(int), s));
  }
  p.n_rows = g->n;
  p.X = X;
  p.ldx = ldx;
  p.packed = packed;
  p.pitch = bits < 32 ? packed_pitch(d, bits) : 0;
  p.hoff = bits < 32 ? (int)header_offset(d, bits) : 0;
  p.mask = mask;
  p.Y = Y;
  p.Yb = static_cast<__nv_bfloat16*>(Yb);
  p.ldy = ldy;
  p.d = d;
  return GQ_OK;
}

size_t spmm_workspace(const gq_graph* g, int transpose, int d) {
  if (g == nullptr || d < 1) return 0;
  return ws_bytes_for(transpose ? g->tr_sched : g->sched, d);
}

int dequant_spmm(const gq_graph* g, int transpose, int coef, const float* X, int64_t ldx, const uint8_t* packed,
                 const uint8_t* mask, int d, int bits, float* Y, int64_t ldy, void* ws, size_t ws_bytes,
                 cudaStream_t s, void* Yb, const uint32_t* gate, int64_t ldg) {
  if (gate != nullptr && (ldg < (d + 31) / 32 || !aligned(gate, 4))) return GQ_ERR_INVALID_ARG;
  SpmmParams p;
  GQ_TRY(spmm_setup(g, transpose, X, ldx, packed, mask, d, bits, Y, ldy, ws, ws_bytes, s, p, Yb));
  p.gate = gate;
  p.ldg = ldg;
  if (coef == GQ_COEF_GCN) {
    // a_{u,v} = dinv_out[u] * dinv_in[v]
    p.colscale = transpose ? g->dinv_in : g->dinv_out;
    p.rowscale = transpose ? g->dinv_out : g->dinv_in;
  } else if (coef == GQ_COEF_SAGE) {
    // a_{u,v} = 1/deg_in(v)
    p.colscale = transpose ? g->inv_in : nullptr;
    p.rowscale = transpose ? nullptr : g->inv_in;
  } else if (coef != GQ_COEF_ONE) {
    return GQ_ERR_INVALID_ARG;
  }
  // packed and fp32 rows mixed by a mask, or fp32 rows alone, with
  // 64 < d <= 256: warp per edge, plain loads into registers; otherwise,
  // d <= 512 and an fp32 row stride under 2^31 bytes: asynchronous ring
  // pipeline; otherwise warp per light row
  if ((bits == 32 || mask != nullptr) && d > 64 && d <= 256 && ldx <= (int64_t)1 << 29)
    return launch_warp_any<0>(p, bits, s);
  if (d <= 512 && ldx <= (int64_t)1 << 29) return launch_async_any(p, bits, s);
  return launch_any<0>(p, bits, s);
}

// Mixed bit-widths per row (rbits, roff from gq_packed_row_offsets).
int dequant_spmm_mixed(const gq_graph* g, int transpose, int coef, const float* X, int64_t ldx, const uint8_t* packed,
                       const int64_t* roff, const uint8_t* rbits, int d, float* Y, int64_t ldy, void* ws,
                       size_t ws_bytes, cudaStream_t s) {
  if (packed == nullptr || roff == nullptr || rbits == nullptr || !aligned(packed, 16)) return GQ_ERR_INVALID_ARG;
  if (d > 256) return GQ_ERR_UNSUPPORTED;
  SpmmParams p;
  GQ_TRY(spmm_setup(g, transpose, X, ldx, nullptr, nullptr, d, 32, Y, ldy, ws, ws_bytes, s, p));
  if (ldx > (int64_t)1 << 29) return GQ_ERR_UNSUPPORTED;
  if (coef == GQ_COEF_GCN) {
    p.colscale = transpose ? g->dinv_in : g->dinv_out;
    p.rowscale = transpose ? g->dinv_out : g->dinv_in;
  } else if (coef == GQ_COEF_SAGE) {
    p.colscale = transpose ? g->inv_in : nullptr;
    p.rowscale = transpose ? nullptr : g->inv_in;
  } else if (coef != GQ_COEF_ONE) {
    return GQ_ERR_INVALID_ARG;
  }
  p.packed = packed;
  p.rbits = rbits;
  p.roff = roff;
  // d <= 128: lane groups of d/16 lanes per edge, each row copied whole at
  // its own width (cp.async ring); wider rows: one warp per edge, bulk copies
  // (each measured the faster of the two in its range)
  if (d <= 128) return launch_async_d<0, 1, false>(p, s);
  return d > 128 ? launch_bulk<0, 8, true, 4, 2>(p, s) : launch_bulk<0, 4, true, 8, 4>(p, s);
}

int edge_spmm(const gq_graph* g, int transpose, const float* alpha, int heads, const float* X, int64_t ldx,
              const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y, int64_t ldy, void* ws,
              size_t ws_bytes, cudaStream_t s) {
  SpmmParams p;
  GQ_TRY(spmm_setup(g, transpose, X, ldx, packed, mask, d, bits, Y, ldy, ws, ws_bytes, s, p));
  if ((alpha == nullptr && g->nnz > 0) || heads < 1 || d % heads != 0) return GQ_ERR_INVALID_ARG;
  const int F = d / heads;
  int fshift = 0;
  while ((1 << fshift) < F) ++fshift;
  if ((1 << fshift) != F || F < 16) return GQ_ERR_UNSUPPORTED;  // head width: power of two >= 16
  p.alpha = alpha;
  p.heads = heads;
  p.fshift = fshift;
  p.eperm = transpose ? g->tr_perm : nullptr;
  // 64 < d <= 256: warp per edge, plain loads into registers; otherwise a
  // warp per light row
  if (d > 64 && d <= 256 && (bits == 32 || mask != nullptr) && ldx <= (int64_t)1 << 29)
    return launch_warp_any<1>(p, bits, s);
  return launch_any<1>(p, bits, s);
}

// Edge-weight mode 2 (8-bit attention codes with per-row, per-head {S, Z})
// for widths up to 256, the GAT layer's range.
template <int BITS>
int launch_alpha8(const SpmmParams& p, cudaStream_t s) {
  if (p.d <= 16) return launch_cfg<BITS, 4, 1, 1, 2, false>(p, s);
  if (p.d <= 32) return launch_cfg<BITS, 4, 1, 2, 2, false>(p, s);
  if (p.d <= 64) return launch_cfg<BITS, 8, 1, 4, 2, false>(p, s);
  if (p.d <= 128) return launch_cfg<BITS, 16, 1, 8, 2, false>(p, s);
  return launch_cfg<BITS, 32, 1, 16, 2, false>(p, s);
}

int edge_spmm_alpha8(const gq_graph* g, const uint8_t* acode, const float* ahdr, int heads, const float* X,
                     int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y,
                     int64_t ldy, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (g == nullptr || ahdr == nullptr || (acode == nullptr && g->nnz > 0) || heads < 1 || d % heads != 0 ||
      !aligned(ahdr, 8))
    return GQ_ERR_INVALID_ARG;
  if (d > 256) return GQ_ERR_UNSUPPORTED;
  const int F = d / heads;
  int fshift = 0;
  while ((1 << fshift) < F) ++fshift;
  if ((1 << fshift) != F || F < 16) return GQ_ERR_UNSUPPORTED;  // head width: power of two >= 16
  SpmmParams p;
  GQ_TRY(spmm_setup(g, 0, X, ldx, packed, mask, d, bits, Y, ldy, ws, ws_bytes, s, p));
  p.acode = acode;
  p.ahdr = ahdr;
  p.heads = heads;
  p.fshift = fshift;
  p.eperm = nullptr;
  // 64 < d <= 256: warp per edge, plain loads into registers
  if (d > 64 && d <= 256 && (bits == 32 || mask != nullptr) && ldx <= (int64_t)1 << 29)
    return launch_warp_any<2>(p, bits, s);
  switch (bits) {
    case 2: return launch_alpha8<2>(p, s);
    case 4: return launch_alpha8<4>(p, s);
    case 8: return launch_alpha8<8>(p, s);
    default: return launch_alpha8<32>(p, s);
  }
}

}  // namespace gq

extern "C" size_t gq_spmm_workspace_bytes(const gq_graph* g, int transpose, int d) {
  return gq::spmm_workspace(g, transpose, d);
}

extern "C" int gq_dequant_spmm(const gq_graph* g, int transpose, int coef, const float* X, int64_t ldx,
                               const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y, int64_t ldy,
                               void* ws, size_t ws_bytes, gq_stream stream) {
  return gq::dequant_spmm(g, transpose, coef, X, ldx, packed, mask, d, bits, Y, ldy, ws, ws_bytes,
                          (cudaStream_t)stream, nullptr);
}

extern "C" int gq_dequant_spmm_mixed(const gq_graph* g, int transpose, int coef, const float* X, int64_t ldx,
                                     const uint8_t* packed, const int64_t* roff, const uint8_t* rbits, int d,
                                     float* Y, int64_t ldy, void* ws, size_t ws_bytes, gq_stream stream) {
  return gq::dequant_spmm_mixed(g, transpose, coef, X, ldx, packed, roff, rbits, d, Y, ldy, ws, ws_bytes,
                                (cudaStream_t)stream);
}

extern "C" int gq_edge_spmm_alpha8(const gq_graph* g, const uint8_t* acode, const float* ahdr, int heads,
                                   const float* X, int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d,
                                   int bits, float* Y, int64_t ldy, void* ws, size_t ws_bytes, gq_stream stream) {
  return gq::edge_spmm_alpha8(g, acode, ahdr, heads, X, ldx, packed, mask, d, bits, Y, ldy, ws, ws_bytes,
                              (cudaStream_t)stream);
}

extern "C" int gq_edge_spmm(const gq_graph* g, int transpose, const float* alpha, int heads, const float* X,
                            int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y,
                            int64_t ldy, void* ws, size_t ws_bytes, gq_stream stream) {
  return gq::edge_spmm(g, transpose, alpha, heads, X, ldx, packed, mask, d, bits, Y, ldy, ws, ws_bytes,
                       (cudaStream_t)stream);
}
