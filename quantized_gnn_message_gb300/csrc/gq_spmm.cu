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
// Work decomposition (power-law degrees):
//   - a row of degree <= hub_threshold is one warp's job.  The warp is split
//     into 32/G lane groups; a group takes one edge at a time and each lane
//     of the group owns 8 consecutive columns (CPL chunks of 8 for d > 256).
//     Edge metadata (column id, coefficient, mask bit) is loaded 32 edges at
//     a time, one per lane, and broadcast with shuffles; U edges per group
//     are gathered before any is consumed, to keep loads in flight.
//   - a heavy row is one or more thread-block tasks (the graph's static
//     schedule, heaviest first, so they start before the light rows): the 8
//     warps of a block interleave 32-edge batches and their partial rows are
//     summed in shared memory in warp order.  A row cut into several tasks
//     writes one partial row per task to the workspace; the last task to
//     finish (arrival ticket) adds them in task order.
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

template <int BITS, int G, int CPL, bool EW>
__global__ void __launch_bounds__(kSpmmThreads) spmm_kernel(const SpmmParams p) {
  extern __shared__ float part[];  // [kSpmmWarps][d] for hub rows
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int gl = lane % G;
  const int nchunks = (p.d + 7) >> 3;

  if ((int64_t)blockIdx.x < p.n_tasks) {
    __shared__ int last;
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.tasks) + blockIdx.x);
    const int64_t r = task.x;
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
    __syncthreads();
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
    return;
  }

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

template <int BITS, int G, int CPL, bool EW>
int launch_cfg(const SpmmParams& p, cudaStream_t s) {
  const size_t smem = sizeof(float) * kSpmmWarps * p.d;
  const int64_t rows_blocks = (p.n_rows + kSpmmWarps - 1) / kSpmmWarps;
  int64_t grid = (int64_t)sm_count() * 8;
  if (grid > rows_blocks) grid = rows_blocks;
  if (grid < 1) grid = 1;
  grid += p.n_tasks;
  if (grid > 0x7fffffff) return GQ_ERR_UNSUPPORTED;
  spmm_kernel<BITS, G, CPL, EW><<<(unsigned)grid, kSpmmThreads, smem, s>>>(p);
  return launch_status();
}

template <int BITS, bool EW>
int launch_bits(const SpmmParams& p, cudaStream_t s) {
  if (p.d <= 32) return launch_cfg<BITS, 4, 1, EW>(p, s);
  if (p.d <= 64) return launch_cfg<BITS, 8, 1, EW>(p, s);
  if (p.d <= 128) return launch_cfg<BITS, 16, 1, EW>(p, s);
  if (p.d <= 256) return launch_cfg<BITS, 32, 1, EW>(p, s);
  if (p.d <= 512) return launch_cfg<BITS, 32, 2, EW>(p, s);
  return launch_cfg<BITS, 32, 4, EW>(p, s);
}

template <bool EW>
int launch_any(const SpmmParams& p, int bits, cudaStream_t s) {
  switch (bits) {
    case 2: return launch_bits<2, EW>(p, s);
    case 4: return launch_bits<4, EW>(p, s);
    case 8: return launch_bits<8, EW>(p, s);
    default: return launch_bits<32, EW>(p, s);
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
  if ((1 << fshift) != F || F < 8) return GQ_ERR_UNSUPPORTED;  // head width: power of two >= 8
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
