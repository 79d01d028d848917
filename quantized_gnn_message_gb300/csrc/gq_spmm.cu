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
// finish (arrival ticket) adds them in task order.  Two kernels share it:
//   - spmm_async_kernel (coefficient mode, d <= 512, every message row of one
//     kind: all packed or all fp32).  A group of LG lanes walks a stream of
//     edges (a slice of a heavy task, or one of the schedule's runs of
//     consecutive light rows) and gathers message rows into a shared-memory
//     ring with cp.async, kAS - 1 steps ahead of the step it consumes, so
//     each SM keeps ~100 KB of gathers in flight.
//   - spmm_kernel (attention weights, a mask mixing packed and fp32 rows, or
//     d > 512).  A light row is one warp's job: lane groups of G lanes take
//     one edge at a time, each lane owning 8 consecutive columns (CPL chunks
//     of 8 for d > 256); edge metadata is loaded 32 edges at a time and
//     broadcast with shuffles, and U edges per group are gathered before any
//     is consumed.  A heavy task's 8 warps split its edges into contiguous
//     streams (stream_row) whose partial rows are summed in shared memory in
//     warp order.
// Every sum runs in a fixed order, so results are identical run to run.
#include <cuda_bf16.h>

#include "gq_common.cuh"
#include "gq_internal.cuh"

namespace gq {

struct SpmmParams {
  const int32_t* rowptr;
  const int32_t* col;
  const int32_t* eperm;     // edge id of each entry (transposed CSR), or null = identity
  const float* colscale;    // per gathered row, or null (= 1)
  const float* rowscale;    // per output row, or null (= 1)
  const float* alpha;       // per edge x heads (edge-weight mode)
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
template <int BITS, int G, int CPL, bool EW>
__device__ __forceinline__ void accumulate_row(const SpmmParams& p, int64_t e_beg, int64_t e_end, int first,
                                               int stride, float (&acc)[CPL][8]) {
  constexpr int NG = 32 / G;
  constexpr int U = CPL == 1 ? 4 : (CPL == 2 ? 2 : 1);
  const int lane = threadIdx.x & 31;
  const int g = lane / G;
  const int gl = lane % G;
  const int nchunks = (p.d + 7) >> 3;
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
            if (EW) cj[t][i] = __ldg(p.alpha + (int64_t)ej * p.heads + ((c * 8) >> p.fshift));
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void store_chunk(const SpmmParams& p, int64_t r, int c, float s, const float (&a)[8]) {
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

__device__ __forceinline__ void lflush(const SpmmParams& p, int64_t r, int c0, const float (&acc)[kLC], float accz) {
  if (c0 >= p.d) return;
  const float s = p.rowscale ? __ldg(p.rowscale + r) : 1.0f;
  float o[kLC];
#pragma unroll
  for (int k = 0; k < kLC; ++k) o[k] = (acc[k] + accz) * s;
  if (p.Yb != nullptr) {
    __nv_bfloat16* y = p.Yb + r * p.ldy + c0;
#pragma unroll
    for (int k = 0; k < kLC; k += 8) {
      if (c0 + k + 8 <= p.d) {
        *reinterpret_cast<uint4*>(y + k) = make_uint4(pack_bf16x2(o[k], o[k + 1]), pack_bf16x2(o[k + 2], o[k + 3]),
                                                      pack_bf16x2(o[k + 4], o[k + 5]), pack_bf16x2(o[k + 6], o[k + 7]));
      } else if (c0 + k + 4 <= p.d) {
        *reinterpret_cast<uint2*>(y + k) = make_uint2(pack_bf16x2(o[k], o[k + 1]), pack_bf16x2(o[k + 2], o[k + 3]));
      }
    }
  } else {
    float* y = p.Y + r * p.ldy + c0;
#pragma unroll
    for (int k = 0; k < kLC; k += 4)
      if (c0 + k < p.d) st_f4(y + k, o[k], o[k + 1], o[k + 2], o[k + 3]);
  }
}

// Per-edge metadata of U consecutive edges: column ids, then coefficients
// and mask bits.
template <int BITS, bool EW, int U>
__device__ __forceinline__ void meta_cols(const SpmmParams& p, int64_t at, int64_t end, int32_t (&xs)[U]) {
#pragma unroll
  for (int t = 0; t < U; ++t) xs[t] = (at + t < end) ? __ldg(p.col + at + t) : 0;
}

template <int BITS, bool EW, bool ALLQ, int U>
__device__ __forceinline__ void meta_coef(const SpmmParams& p, int64_t at, int64_t end, int head,
                                          const int32_t (&xs)[U], float (&f)[U], bool (&q)[U]) {
#pragma unroll
  for (int t = 0; t < U; ++t) {
    f[t] = 1.0f;
    q[t] = ALLQ;
    if (at + t < end) {
      if (EW) {
        const int64_t eid = p.eperm ? __ldg(p.eperm + at + t) : at + t;
        f[t] = __ldg(p.alpha + eid * p.heads + head);
      } else if (p.colscale) {
        f[t] = __ldg(p.colscale + xs[t]);
      }
      if (!ALLQ) q[t] = BITS < 32 && (p.mask == nullptr || __ldg(p.mask + xs[t]) != 0);
    }
  }
}

// Accumulate the contiguous edges [e_beg, e_end) of one row into this
// lane's 16 columns, in the three-stage pipeline described above.
template <int BITS, bool EW, bool ALLQ>
__device__ __forceinline__ void stream_row(const SpmmParams& p, int64_t e_beg, int64_t e_end, int c0, int head,
                                           float (&acc)[kLC], float& accz) {
  constexpr int U = kLU;
  int32_t cx[U], nx[U];
  float cf[U];
  bool cq[U];
  meta_cols<BITS, EW, U>(p, e_beg, e_end, cx);
  meta_coef<BITS, EW, ALLQ, U>(p, e_beg, e_end, head, cx, cf, cq);
  meta_cols<BITS, EW, U>(p, e_beg + U, e_end, nx);
  for (int64_t e = e_beg; e < e_end; e += U) {
    LMsg<BITS, ALLQ> m[U];
#pragma unroll
    for (int t = 0; t < U; ++t)
      if (e + t < e_end && c0 < p.d) lload<BITS, ALLQ>(p, cx[t], cq[t], c0, m[t]);
    float nf[U];
    bool nq[U];
    meta_coef<BITS, EW, ALLQ, U>(p, e + U, e_end, head, nx, nf, nq);
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
        p.Yb[r * p.ldy + j] = __float2bfloat16_rn(t * s);
      else
        p.Y[r * p.ldy + j] = t * s;
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
      p.Yb[r * p.ldy + j] = __float2bfloat16_rn(t * s);
    else
      p.Y[r * p.ldy + j] = t * s;
  }
}

template <int BITS, int G, int CPL, int LG, bool EW, bool ALLQ>
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
      if (b0 < b1) stream_row<BITS, EW, ALLQ>(p, b0, b1, c0, head, acc, accz);
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
      accumulate_row<BITS, G, CPL, EW>(p, task.y, task.z, w, kSpmmWarps, acc);
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
      accumulate_row<BITS, G, CPL, EW>(p, a, b, 0, 1, acc);
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
// Asynchronous-copy aggregation (coefficient modes, d <= 512).
//
// Every message row a group needs is copied into a per-group ring of
// shared memory with cp.async (16-byte pieces spread over the group's
// lanes, the coefficient as one 4-byte copy), kAS steps of U edges deep,
// and consumed kAS - 1 steps later.  In-flight data lives in shared memory,
// not registers, so each SM keeps ~100 KB of gathers in flight at full
// occupancy.  Work units: heavy-row block tasks (each group streams a
// contiguous slice of the row) and runs of light rows (one group each,
// rows retired edge by edge as they are consumed).
// ---------------------------------------------------------------------------
constexpr int kAS = 4;  // pipeline stages

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t sm_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Bytes of one edge slot and of one group's ring.
__host__ __device__ inline int async_slot(int d, int bits, bool mixed) {
  int b = bits < 32 ? (int)packed_pitch(d, bits) : 4 * d;
  if (mixed && 4 * d > b) b = 4 * d;
  return (b + 15) / 16 * 16;
}
__host__ __device__ inline int async_ring(int slot, int U) { return kAS * U * slot + ((kAS * U * 5 + 15) / 16) * 16; }

template <int BITS, bool MIXED>
__device__ __forceinline__ void adecode(const SpmmParams& p, const uint8_t* sl, bool quant, float coef, int c0,
                                        float (&acc)[kLC], float& accz) {
  if (BITS < 32 && (!MIXED || quant)) {
    LMsg<BITS, true> m;
    m.quant = true;
    m.h = *reinterpret_cast<const float2*>(sl + p.hoff);
    const uint8_t* pl = sl + c0 * BITS / 8;
    if constexpr (BITS == 8) {
      const uint4 t = *reinterpret_cast<const uint4*>(pl);
      m.w[0] = t.x; m.w[1] = t.y; m.w[2] = t.z; m.w[3] = t.w;
    } else if constexpr (BITS == 4) {
      const uint2 t = *reinterpret_cast<const uint2*>(pl);
      m.w[0] = t.x; m.w[1] = t.y;
    } else if constexpr (BITS == 2) {
      m.w[0] = *reinterpret_cast<const uint32_t*>(pl);
    }
    lconsume<BITS, true>(m, coef, acc, accz);
  } else {
    const float* xr = reinterpret_cast<const float*>(sl) + c0;
#pragma unroll
    for (int k = 0; k < kLC; k += 4) {
      if (c0 + k < p.d) {
        const float4 a = *reinterpret_cast<const float4*>(xr + k);
        acc[k] = __fmaf_rn(coef, a.x, acc[k]);
        acc[k + 1] = __fmaf_rn(coef, a.y, acc[k + 1]);
        acc[k + 2] = __fmaf_rn(coef, a.z, acc[k + 2]);
        acc[k + 3] = __fmaf_rn(coef, a.w, acc[k + 3]);
      }
    }
  }
}

// Stream edges [eb, ee) through the group's ring.  LIGHT: the edges are
// those of rows [row0, row1) and each row is written when its last edge
// has been consumed; otherwise they all belong to one row and the sums are
// left in acc / accz.
template <int BITS, int LG, bool MIXED, int U, bool LIGHT>
__device__ __forceinline__ void async_stream(const SpmmParams& p, uint8_t* ring, int slot, unsigned gmask, int gl,
                                             int c0, int64_t eb, int64_t ee, int64_t row0, int64_t row1,
                                             float (&acc)[kLC], float& accz) {
  float* coefs = reinterpret_cast<float*>(ring + kAS * U * slot);
  uint8_t* flags = reinterpret_cast<uint8_t*>(coefs + kAS * U);
  const int64_t nsteps = (ee - eb + U - 1) / U;
  const int chunks_q = (int)(p.pitch / 16);
  const int chunks_x = p.d / 4;
  int32_t cx[U], nx[U];
  bool cq[U];
#pragma unroll
  for (int t = 0; t < U; ++t) {
    cx[t] = (eb + t < ee) ? __ldg(p.col + eb + t) : 0;
    cq[t] = BITS < 32 && (!MIXED || (p.mask == nullptr || __ldg(p.mask + cx[t]) != 0));
    nx[t] = (eb + U + t < ee) ? __ldg(p.col + eb + U + t) : 0;
  }
  int64_t row = row0, re = LIGHT ? __ldg(p.rowptr + row0 + 1) : 0;
  for (int64_t s = 0; s < nsteps + kAS - 1; ++s) {
    __syncwarp(gmask);  // the slots refilled below have been consumed
    if (s < nsteps) {
      const int st = (int)(s % kAS);
#pragma unroll
      for (int t = 0; t < U; ++t) {
        const int64_t e = eb + s * U + t;
        if (e < ee) {
          uint8_t* dst = ring + (st * U + t) * slot;
          if (BITS < 32 && (!MIXED || cq[t])) {
            const uint8_t* src = p.packed + (int64_t)cx[t] * p.pitch;
            for (int k = gl; k < chunks_q; k += LG) cp_async16(sm_addr(dst + 16 * k), src + 16 * k);
          } else {
            const float* src = p.X + (int64_t)cx[t] * p.ldx;
            for (int k = gl; k < chunks_x; k += LG) cp_async16(sm_addr(dst + 16 * k), src + 4 * k);
          }
          if (gl == 0) {
            if (p.colscale != nullptr) cp_async4(sm_addr(coefs + st * U + t), p.colscale + cx[t]);
            if (MIXED) flags[st * U + t] = cq[t] ? 1 : 0;
          }
        }
      }
      // column ids (and mask bits) of the next step are ready; fetch the one after
#pragma unroll
      for (int t = 0; t < U; ++t) {
        cx[t] = nx[t];
        const int64_t e1 = eb + (s + 1) * U + t, e2 = eb + (s + 2) * U + t;
        cq[t] = BITS < 32 && (!MIXED || (e1 < ee && (p.mask == nullptr || __ldg(p.mask + cx[t]) != 0)));
        nx[t] = (e2 < ee) ? __ldg(p.col + e2) : 0;
      }
    }
    cp_commit();
    if (s >= kAS - 1) {
      const int64_t c = s - (kAS - 1);
      cp_wait<kAS - 1>();
      __syncwarp(gmask);
      const int st = (int)(c % kAS);
#pragma unroll
      for (int t = 0; t < U; ++t) {
        const int64_t e = eb + c * U + t;
        if (e < ee) {
          if (LIGHT) {
            while (e >= re) {
              lflush(p, row, c0, acc, accz);
#pragma unroll
              for (int k = 0; k < kLC; ++k) acc[k] = 0.0f;
              accz = 0.0f;
              ++row;
              re = __ldg(p.rowptr + row + 1);
            }
          }
          if (c0 < p.d) {
            const float coef = p.colscale != nullptr ? coefs[st * U + t] : 1.0f;
            const bool quant = !MIXED || flags[st * U + t] != 0;
            adecode<BITS, MIXED>(p, ring + (st * U + t) * slot, quant, coef, c0, acc, accz);
          }
        }
      }
    }
  }
  if (LIGHT) {
    for (; row < row1; ++row) {
      lflush(p, row, c0, acc, accz);
#pragma unroll
      for (int k = 0; k < kLC; ++k) acc[k] = 0.0f;
      accz = 0.0f;
    }
  }
}

template <int BITS, int LG, bool MIXED, int U>
__global__ void __launch_bounds__(kSpmmThreads) spmm_async_kernel(const SpmmParams p, int slot, int ring) {
  extern __shared__ __align__(16) uint8_t asm_[];
  constexpr int NG = 32 / LG;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane / LG, gl = lane % LG;
  const unsigned gmask = (LG == 32 ? 0xffffffffu : ((1u << LG) - 1u)) << (g * LG);
  uint8_t* myring = asm_ + (size_t)(w * NG + g) * ring;
  const int c0 = gl * kLC;
  float acc[kLC] = {};
  float accz = 0.0f;
  if ((int64_t)blockIdx.x < p.n_tasks) {
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.tasks) + blockIdx.x);
    const int sid = w * NG + g;
    const int64_t len = task.z - task.y;
    int64_t chunk = (len + kSpmmWarps * NG - 1) / (kSpmmWarps * NG);
    chunk = (chunk + U - 1) / U * U;
    const int64_t b0 = task.y + (int64_t)sid * chunk;
    const int64_t b1 = min(b0 + chunk, (int64_t)task.z);
    if (b0 < b1) async_stream<BITS, LG, MIXED, U, false>(p, myring, slot, gmask, gl, c0, b0, b1, 0, 0, acc, accz);
#pragma unroll
    for (int k = 0; k < kLC; ++k) acc[k] += accz;
#pragma unroll
    for (int o = LG; o < 32; o <<= 1)
#pragma unroll
      for (int k = 0; k < kLC; ++k) acc[k] += __shfl_xor_sync(FULL, acc[k], o);
    __syncthreads();  // every ring is drained: reuse the space for the warp partials
    float* part = reinterpret_cast<float*>(asm_);
    if (lane < LG && c0 < p.d)
#pragma unroll
      for (int k = 0; k < kLC; ++k)
        if (c0 + k < p.d) part[w * p.d + c0 + k] = acc[k];
    __syncthreads();
    finish_heavy(p, task, part);
    return;
  }
  const int64_t gid = ((int64_t)blockIdx.x - p.n_tasks) * kSpmmWarps * NG + w * NG + g;
  const int64_t ngroups = ((int64_t)gridDim.x - p.n_tasks) * kSpmmWarps * NG;
  for (int64_t t = gid; t < p.n_light; t += ngroups) {
    const int2 run = __ldg(reinterpret_cast<const int2*>(p.light) + t);
    const int64_t eb = __ldg(p.rowptr + run.x), ee = __ldg(p.rowptr + run.y);
    async_stream<BITS, LG, MIXED, U, true>(p, myring, slot, gmask, gl, c0, eb, ee, run.x, run.y, acc, accz);
  }
}

template <int BITS, int LG, bool MIXED, int U>
int launch_async(SpmmParams p, cudaStream_t s) {
  const int slot = async_slot(p.d, BITS, MIXED);
  const int ring = async_ring(slot, U);
  constexpr int NG = 32 / LG;
  size_t smem = (size_t)kSpmmWarps * NG * ring;
  const size_t part = sizeof(float) * kSpmmWarps * p.d;
  if (smem < part) smem = part;
  auto kern = spmm_async_kernel<BITS, LG, MIXED, U>;
  if (smem > 48 * 1024) GQ_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSpmmThreads, smem) != cudaSuccess || per_sm < 1)
    return GQ_ERR_UNSUPPORTED;
  int64_t light = (int64_t)sm_count() * per_sm;
  const int64_t need = (p.n_light + kSpmmWarps * NG - 1) / (kSpmmWarps * NG);
  if (light > need) light = need;
  if (light < 1) light = 1;
  const int64_t grid = p.n_tasks + light;
  if (grid > 0x7fffffff) return GQ_ERR_UNSUPPORTED;
  kern<<<(unsigned)grid, kSpmmThreads, smem, s>>>(p, slot, ring);
  return launch_status();
}

template <int BITS, bool MIXED, int U>
int launch_async_d(const SpmmParams& p, cudaStream_t s) {
  if (p.d <= 16) return launch_async<BITS, 1, MIXED, U>(p, s);
  if (p.d <= 32) return launch_async<BITS, 2, MIXED, U>(p, s);
  if (p.d <= 64) return launch_async<BITS, 4, MIXED, U>(p, s);
  if (p.d <= 128) return launch_async<BITS, 8, MIXED, U>(p, s);
  if (p.d <= 256) return launch_async<BITS, 16, MIXED, U>(p, s);
  return launch_async<BITS, 32, MIXED, U>(p, s);
}

// Coefficient-mode aggregation with d <= 512 and one kind of message row
// (all packed, or all fp32); packed rows keep two edges per stage.
int launch_async_any(const SpmmParams& p, int bits, cudaStream_t s) {
  switch (bits) {
    case 2: return launch_async_d<2, false, 2>(p, s);
    case 4: return launch_async_d<4, false, 2>(p, s);
    case 8: return launch_async_d<8, false, 2>(p, s);
    default: return launch_async_d<32, false, 1>(p, s);
  }
}

template <int BITS, int G, int CPL, int LG, bool EW, bool ALLQ>
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

template <int BITS, bool EW, bool ALLQ>
int launch_bits(const SpmmParams& p, cudaStream_t s) {
  if (p.d <= 16) return launch_cfg<BITS, 4, 1, 1, EW, ALLQ>(p, s);
  if (p.d <= 32) return launch_cfg<BITS, 4, 1, 2, EW, ALLQ>(p, s);
  if (p.d <= 64) return launch_cfg<BITS, 8, 1, 4, EW, ALLQ>(p, s);
  if (p.d <= 128) return launch_cfg<BITS, 16, 1, 8, EW, ALLQ>(p, s);
  if (p.d <= 256) return launch_cfg<BITS, 32, 1, 16, EW, ALLQ>(p, s);
  if (p.d <= 512) return launch_cfg<BITS, 32, 2, 32, EW, ALLQ>(p, s);
  return launch_cfg<BITS, 32, 4, 0, EW, ALLQ>(p, s);
}

template <bool EW>
int launch_any(const SpmmParams& p, int bits, cudaStream_t s) {
  switch (bits) {
    case 2: return launch_bits<2, EW, false>(p, s);
    case 4: return launch_bits<4, EW, false>(p, s);
    case 8: return launch_bits<8, EW, false>(p, s);
    default: return launch_bits<32, EW, false>(p, s);
  }
}

}  // namespace

// Common argument checks and message-source setup.
size_t ws_bytes_for(const gq_sched& sc, int d) {
  if (sc.n_groups == 0) return 0;
  return ((size_t)sc.n_slots * d * sizeof(float) + 255) / 256 * 256 + (size_t)sc.n_groups * sizeof(int) + 256;
}

int spmm_setup(const gq_graph* g, int transpose, const float* X, int64_t ldx, const uint8_t* packed,
               const uint8_t* mask, int d, int bits, float* Y, int64_t ldy, void* ws, size_t ws_bytes,
               cudaStream_t s, SpmmParams& p, void* Yb = nullptr) {
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
                 cudaStream_t s, void* Yb) {
  SpmmParams p;
  GQ_TRY(spmm_setup(g, transpose, X, ldx, packed, mask, d, bits, Y, ldy, ws, ws_bytes, s, p, Yb));
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
  // every message row of one kind (all packed, or all fp32): asynchronous
  // pipeline; a mix of packed and fp32 rows (a mask): warp per light row,
  // whose registers hold the 1 KB fp32 rows more cheaply than 1 KB ring slots
  if (d <= 512 && !(bits < 32 && mask != nullptr)) return launch_async_any(p, bits, s);
  return launch_any<false>(p, bits, s);
}

int edge_spmm(const gq_graph* g, int transpose, const float* alpha, int heads, const float* X, int64_t ldx,
              const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y, int64_t ldy, void* ws,
              size_t ws_bytes, cudaStream_t s) {
  SpmmParams p;
  GQ_TRY(spmm_setup(g, transpose, X, ldx, packed, mask, d, bits, Y, ldy, ws, ws_bytes, s, p));
  if (alpha == nullptr || heads < 1 || d % heads != 0) return GQ_ERR_INVALID_ARG;
  const int F = d / heads;
  int fshift = 0;
  while ((1 << fshift) < F) ++fshift;
  if ((1 << fshift) != F || F < 16) return GQ_ERR_UNSUPPORTED;  // head width: power of two >= 16
  p.alpha = alpha;
  p.heads = heads;
  p.fshift = fshift;
  p.eperm = transpose ? g->tr_perm : nullptr;
  return launch_any<true>(p, bits, s);
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

extern "C" int gq_edge_spmm(const gq_graph* g, int transpose, const float* alpha, int heads, const float* X,
                            int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y,
                            int64_t ldy, void* ws, size_t ws_bytes, gq_stream stream) {
  return gq::edge_spmm(g, transpose, alpha, heads, X, ldx, packed, mask, d, bits, Y, ldy, ws, ws_bytes,
                       (cudaStream_t)stream);
}
