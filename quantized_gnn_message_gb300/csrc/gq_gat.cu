// gq_gat.cu -- the edge kernels of the GAT layer (Tango Sec. 2.1, Fig. 1).
//
// edge_softmax_kernel  (Fig. 1a steps 3-4), per destination row v:
//     E_pre[e,k] = S[u,k] + D[v,k]            (SDDMM add, e = u -> v)
//     E[e,k]     = LeakyReLU(E_pre[e,k])
//     alpha[e,k] = exp(E[e,k] - max_v) / sum_{e' in in(v)} exp(E[e',k] - max_v)
//   one pass keeps an online (max, sum) per head, a second writes alpha;
//   a row of at most 32 edges is one thread's, rows up to the hub threshold
//   a warp's, heavier rows are cut into tasks of one warp each, whose
//   (max, sum) partials are merged in task order before their second pass.
// gat_edge_bwd_kernel + gat_edge_bwd_heavy_kernel  (Fig. 1b), per
// destination row v (light rows one warp each over the graph's light-row
// runs; heavy rows as block tasks, their P and dD merged in task order):
//     dalpha[e,k] = sum_f dOut[v,kF+f] m_u[kF+f]          (SDDMM dot)
//     P[v,k]      = sum_e alpha[e,k] dalpha[e,k]
//     dE_pre[e,k] = alpha (dalpha - P) * (E_pre > 0 ? 1 : slope)
//     dD[v,k]     = sum_e dE_pre[e,k]                      (in-edge sum)
// gat_node_heavy_kernel + gat_node_bwd_kernel  per source row u (transposed CSR):
//     dS[u,k]     = sum_{e in out(u)} dE_pre[e,k]          (out-edge sum; rows
//                   above the hub threshold as block tasks, the rest by lane
//                   or warp within groups of 32 rows)
//     dH'[u,c]    = dM[u,c] + dS[u,k] a_src[k,f] + dD[u,k] a_dst[k,f]
//     partial sums of da_src = sum_u dS[u,k] H'[u,:], da_dst likewise.
// edge_quant_kernel / edge_quant_heavy_kernel / edge_dequant_kernel
//   (Tango Sec. 3.3): the attention values as 8-bit codes, one AdaQP Eqn 4
//   vector per (destination, head) segment, and their de-quantized values.
// Heavy rows follow the graph's static schedule: the softmax and the
// quantizer cut them into warp tasks whose partials a second kernel merges;
// the edge and node backward use block tasks whose per-task partials are
// combined in task order (by a second kernel, or by the last block of the
// row to finish).  The softmax and the quantizer check
// each range and index they read against the graph and record an invalid
// one in the graph status word.
// Scores, attention and their gradients stay fp32 (Tango Sec. 3.2: full
// precision before the softmax).
#include <cuda_bf16.h>

#include "gq_common.cuh"
#include "gq_internal.cuh"
#include "gq_msg.cuh"

namespace gq {
namespace {

constexpr int kGatThreads = 256;
constexpr int kGatWarps = kGatThreads / 32;

constexpr float kNegInf = -__builtin_huge_valf();

// ------------------------------------------------------------ helpers ---
template <int K>
__device__ __forceinline__ void load_k(const float* __restrict__ p, float (&v)[K]) {
  if constexpr (K == 4) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  } else if constexpr (K == 8) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = __ldg(p + k);
  }
}

template <int K>
__device__ __forceinline__ void store_k(float* __restrict__ p, const float (&v)[K]) {
  if constexpr (K == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  } else if constexpr (K == 8) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
  } else if constexpr (K == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) p[k] = v[k];
  }
}

__device__ __forceinline__ float lrelu(float x, float slope) { return x > 0.0f ? x : slope * x; }

__device__ __forceinline__ void online_merge(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  if (M == kNegInf) return;  // both empty
  l = l * expf(m - M) + l2 * expf(m2 - M);
  m = M;
}

struct Sched {
  const int32_t* tasks;
  const int32_t* groups;
  int64_t n_tasks;
  int hub_threshold;
  float* partial;  // [slot][...]
  int* tickets;    // [group]
};

// Block-wide: publish this task's partial (n floats at `mine`), take a
// ticket; returns true in the last block of the group (after a fence).
__device__ __forceinline__ bool last_of_group(const Sched& sc, int group, int n_in_group) {
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(&sc.tickets[group], 1) == n_in_group - 1);
  __syncthreads();
  if (last) __threadfence();
  return last;
}

// ------------------------------------------------------- edge softmax ---
struct SoftmaxParams {
  const int32_t* rowptr;
  const int32_t* col;
  const float* S;
  const float* D;
  float slope;
  float* alpha;
  float* Epre;
  int64_t n_rows;
  int64_t n_edges;
  int64_t n_groups;
  int* err;  // graph status word
  Sched sc;
};

// Self-checks of the softmax: each row, task and group range is checked
// against the graph before it is walked, and each column id before its S
// row is read; an invalid one is recorded in the graph status word
// (kSoftmaxBadIndex) and the access is skipped (the row or task) or sent to
// row 0 (a column id), so no index read from memory can leave its buffer.
// The column check is one unsigned compare on the common path (n < 2^31).
constexpr int kSoftmaxBadIndex = 0x534D;
__device__ __forceinline__ int32_t sm_checked_col(int32_t x, int64_t n, int* err) {
  if ((uint32_t)x < (uint32_t)n) return x;
  atomicCAS(err, 0, kSoftmaxBadIndex);
  return 0;
}
__device__ __forceinline__ bool sm_range_ok(const SoftmaxParams& p, int64_t v, int64_t a, int64_t b) {
  const bool ok = v >= 0 && v < p.n_rows && a >= 0 && a <= b && b <= p.n_edges;
  if (!ok) atomicCAS(p.err, 0, kSoftmaxBadIndex);
  return ok;
}

// Scores of the thread's edges e, e + stride, e + 2 stride, e + 3 stride
// (those below end): their column ids, then their S rows, loaded before any
// is used.
template <int K>
__device__ __forceinline__ void sm_scores4s(const SoftmaxParams& p, int64_t e, int64_t end, int64_t stride,
                                            const float (&dv)[K], float (&ep)[4][K]) {
  int32_t x[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) x[t] = e + t * stride < end ? __ldg(p.col + e + t * stride) : 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    float s[K];
    load_k<K>(p.S + (int64_t)sm_checked_col(x[t], p.n_rows, p.err) * K, s);
#pragma unroll
    for (int k = 0; k < K; ++k) ep[t][k] = s[k] + dv[k];
  }
}

// (max, sum) of this thread's edges e = first, first + stride, ...
template <int K>
__device__ __forceinline__ void sm_pass1(const SoftmaxParams& p, int64_t first, int64_t end, int64_t stride,
                                         const float (&dv)[K], float (&m)[K], float (&l)[K]) {
#pragma unroll
  for (int k = 0; k < K; ++k) {
    m[k] = kNegInf;
    l[k] = 0.0f;
  }
  for (int64_t e = first; e < end; e += 4 * stride) {
    float ep[4][K];
    sm_scores4s<K>(p, e, end, stride, dv, ep);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (e + t * stride < end) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const float x = lrelu(ep[t][k], p.slope);
          const float mn = fmaxf(m[k], x);
          l[k] = l[k] * __expf(m[k] - mn) + __expf(x - mn);
          m[k] = mn;
        }
      }
    }
  }
}

template <int K>
__device__ __forceinline__ void sm_pass2(const SoftmaxParams& p, int64_t first, int64_t end, int64_t stride,
                                         const float (&dv)[K], const float (&M)[K], const float (&L)[K]) {
  float inv[K];
#pragma unroll
  for (int k = 0; k < K; ++k) inv[k] = 1.0f / L[k];
  for (int64_t e = first; e < end; e += 4 * stride) {
    float ep[4][K];
    sm_scores4s<K>(p, e, end, stride, dv, ep);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int64_t et = e + t * stride;
      if (et < end) {
        float al[K];
#pragma unroll
        for (int k = 0; k < K; ++k) al[k] = __expf(lrelu(ep[t][k], p.slope) - M[k]) * inv[k];
        store_k<K>(p.alpha + et * K, al);
        if (p.Epre != nullptr) store_k<K>(p.Epre + et * K, ep[t]);
      }
    }
  }
}

// One row [a, b) of at most 32 edges by one thread: scores, online max and
// sum per head, then alpha = exp(E - max) / sum.  Edges go four at a time
// (their column ids, then their S rows, loaded before any is used).
template <int K>
__device__ __forceinline__ void sm_scores4(const SoftmaxParams& p, int64_t e, int64_t b, const float (&dv)[K],
                                           float (&ep)[4][K]) {
  int32_t x[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) x[t] = e + t < b ? __ldg(p.col + e + t) : 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    float s[K];
    load_k<K>(p.S + (int64_t)sm_checked_col(x[t], p.n_rows, p.err) * K, s);
#pragma unroll
    for (int k = 0; k < K; ++k) ep[t][k] = s[k] + dv[k];
  }
}

template <int K>
__device__ __forceinline__ void sm_thread_row(const SoftmaxParams& p, int64_t r, int64_t a, int64_t b) {
  float dv[K];
  load_k<K>(p.D + r * K, dv);
  float m[K], l[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    m[k] = kNegInf;
    l[k] = 0.0f;
  }
  for (int64_t e = a; e < b; e += 4) {
    float ep[4][K];
    sm_scores4<K>(p, e, b, dv, ep);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (e + t < b) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const float x = lrelu(ep[t][k], p.slope);
          const float mn = fmaxf(m[k], x);
          l[k] = l[k] * __expf(m[k] - mn) + __expf(x - mn);
          m[k] = mn;
        }
      }
    }
  }
  float inv[K];
#pragma unroll
  for (int k = 0; k < K; ++k) inv[k] = 1.0f / l[k];
  for (int64_t e = a; e < b; e += 4) {
    float ep[4][K];
    sm_scores4<K>(p, e, b, dv, ep);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (e + t < b) {
        float al[K];
#pragma unroll
        for (int k = 0; k < K; ++k) al[k] = __expf(lrelu(ep[t][k], p.slope) - m[k]) * inv[k];
        store_k<K>(p.alpha + (e + t) * K, al);
        if (p.Epre != nullptr) store_k<K>(p.Epre + (e + t) * K, ep[t]);
      }
    }
  }
}

template <int K>
__device__ __forceinline__ void warp_merge(float (&m)[K], float (&l)[K]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const float m2 = __shfl_xor_sync(FULL, m[k], o);
      const float l2 = __shfl_xor_sync(FULL, l[k], o);
      online_merge(m[k], l[k], m2, l2);
    }
}

// Heavy rows (more edges than the hub threshold) are cut into the graph's
// tasks.  This kernel: one warp per task computes the online (max, sum) of
// its edges into part[task] (first pass); then the light rows.  The second
// pass of the heavy rows is edge_softmax_heavy_kernel.
template <int K>
__global__ void __launch_bounds__(kGatThreads) edge_softmax_kernel(const SoftmaxParams p) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t gw = (int64_t)blockIdx.x * kGatWarps + w;
  const int64_t nw = (int64_t)gridDim.x * kGatWarps;
  for (int64_t t = gw; t < p.sc.n_tasks; t += nw) {
    int4 task = __ldg(reinterpret_cast<const int4*>(p.sc.tasks) + t);
    if (!sm_range_ok(p, task.x, task.y, task.z)) task = make_int4(0, 0, 0, -1);
    float dv[K];
    load_k<K>(p.D + (int64_t)task.x * K, dv);
    float m[K], l[K];
    sm_pass1<K>(p, (int64_t)task.y + lane, task.z, 32, dv, m, l);
    warp_merge<K>(m, l);
    if (lane == 0) {
      float* mine = p.sc.partial + t * 2 * K;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        mine[2 * k] = m[k];
        mine[2 * k + 1] = l[k];
      }
    }
  }
  // light rows, in groups of 32 consecutive rows per warp: a row of at most
  // 32 edges is one thread's (two passes over its edges, the online max and
  // sum in registers); the group's rows of 33 .. hub_threshold edges are
  // then taken one at a time by the whole warp
  const int64_t groups = (p.n_rows + 31) / 32;
  for (int64_t grp = gw; grp < groups; grp += nw) {
    const int64_t r = grp * 32 + lane;
    int64_t a = 0, b = 0;
    if (r < p.n_rows) {
      a = __ldg(p.rowptr + r);
      b = __ldg(p.rowptr + r + 1);
      if (!sm_range_ok(p, r, a, b)) b = a;
    }
    if (r < p.n_rows && b - a <= 32) sm_thread_row<K>(p, r, a, b);
    unsigned mid = __ballot_sync(FULL, r < p.n_rows && b - a > 32 && b - a <= p.sc.hub_threshold);
    while (mid != 0) {
      const int l0 = __ffs(mid) - 1;
      mid &= mid - 1;
      const int64_t v = grp * 32 + l0;
      const int64_t va = __shfl_sync(FULL, a, l0), vb = __shfl_sync(FULL, b, l0);
      float dv[K];
      load_k<K>(p.D + v * K, dv);
      float m[K], l[K];
      sm_pass1<K>(p, va + lane, vb, 32, dv, m, l);
      warp_merge<K>(m, l);
      sm_pass2<K>(p, va + lane, vb, 32, dv, m, l);
    }
  }
}

// Second pass of the heavy rows: one warp per task merges the (max, sum)
// partials of its row's tasks in task order (its own alone when the row is
// one task) and writes alpha for the task's edges.
template <int K>
__global__ void __launch_bounds__(kGatThreads) edge_softmax_heavy_kernel(const SoftmaxParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= p.sc.n_tasks) return;
  const int4 task = __ldg(reinterpret_cast<const int4*>(p.sc.tasks) + t);
  int64_t t0 = t, nt = 1;
  if (task.w >= p.n_groups) {
    atomicCAS(p.err, 0, kSoftmaxBadIndex);
    return;
  }
  if (task.w >= 0) {
    const int4 grp = __ldg(reinterpret_cast<const int4*>(p.sc.groups) + task.w);
    t0 = grp.y;
    nt = grp.z;
  }
  if (!sm_range_ok(p, task.x, task.y, task.z) || t0 < 0 || nt < 1 || t0 + nt > p.sc.n_tasks || t < t0 ||
      t >= t0 + nt) {
    atomicCAS(p.err, 0, kSoftmaxBadIndex);
    return;
  }
  float m[K], l[K];
  const float* base = p.sc.partial + t0 * 2 * K;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    m[k] = __ldcg(base + 2 * k);
    l[k] = __ldcg(base + 2 * k + 1);
    for (int64_t i = 1; i < nt; ++i) online_merge(m[k], l[k], __ldcg(base + i * 2 * K + 2 * k), __ldcg(base + i * 2 * K + 2 * k + 1));
  }
  float dv[K];
  load_k<K>(p.D + (int64_t)task.x * K, dv);
  sm_pass2<K>(p, (int64_t)task.y + lane, task.z, 32, dv, m, l);
}

// ------------------------------------------- 8-bit attention values ---
// Tango Sec. 3.3: the SpMM reads quantized edge features.  Each (destination
// v, head k) segment alpha[rowptr[v] .. rowptr[v+1], k] is one vector of
// AdaQP Sec. 2.3 Eqn 4 at 8 bits: Z = min, S = (max - min) / 255,
// q = min(floor((alpha - Z) * (1/S) + u), 255) in fp32 round-to-nearest
// steps, u hashed from (seed, edge id, head); a segment with S below the
// smallest normal float codes as 0.  codes[e*K + k] bytes, hdr[(v*K + k)*2]
// = {S, Z}, {0, 0} for a row without edges.  Same schedule as the softmax:
// thread rows, warp rows, and heavy rows as warp tasks whose (min, max)
// partials merge in a second kernel (min and max are exact in any order).
struct EdgeQuantParams {
  const int32_t* rowptr;
  const float* alpha;
  uint8_t* codes;
  float* hdr;
  uint32_t seed_key;
  int64_t n_rows;
  int64_t n_edges;
  Sched sc;      // partial: [task][2K] {min, max}
  float* deq;    // de-quantized values (edge_dequant_kernel)
  int* err;      // graph status word: kEdgeQuantBadRange if a row or task range was invalid
};

// Every edge range is checked against the edge count before it is read or
// written; an invalid one is recorded in the status word and skipped.
constexpr int kEdgeQuantBadRange = 0x4551;
__device__ __forceinline__ bool eq_range_ok(const EdgeQuantParams& p, int64_t v, int64_t a, int64_t b) {
  const bool ok = v >= 0 && v < p.n_rows && a >= 0 && a <= b && b <= p.n_edges;
  if (!ok) atomicCAS(p.err, 0, kEdgeQuantBadRange);
  return ok;
}

template <int K>
__device__ __forceinline__ void eq_minmax(const EdgeQuantParams& p, int64_t first, int64_t end, int64_t stride,
                                          float (&mn)[K], float (&mx)[K]) {
#pragma unroll
  for (int k = 0; k < K; ++k) {
    mn[k] = __builtin_huge_valf();
    mx[k] = kNegInf;
  }
  int64_t e = first;
  for (; e + 3 * stride < end; e += 4 * stride) {
    float a[4][K];
#pragma unroll
    for (int t = 0; t < 4; ++t) load_k<K>(p.alpha + (e + t * stride) * K, a[t]);
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int k = 0; k < K; ++k) {
        mn[k] = fminf(mn[k], a[t][k]);
        mx[k] = fmaxf(mx[k], a[t][k]);
      }
  }
  for (; e < end; e += stride) {
    float a[K];
    load_k<K>(p.alpha + e * K, a);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      mn[k] = fminf(mn[k], a[k]);
      mx[k] = fmaxf(mx[k], a[k]);
    }
  }
}

template <int K>
__device__ __forceinline__ void warp_minmax(float (&mn)[K], float (&mx)[K]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int k = 0; k < K; ++k) {
      mn[k] = fminf(mn[k], __shfl_xor_sync(FULL, mn[k], o));
      mx[k] = fmaxf(mx[k], __shfl_xor_sync(FULL, mx[k], o));
    }
}

// Eqn 4 scale of each head's segment; writes the row's header when `head`.
template <int K>
__device__ __forceinline__ void eq_scale(const EdgeQuantParams& p, int64_t v, const float (&mn)[K],
                                         const float (&mx)[K], bool head, float (&S)[K], float (&inv)[K]) {
#pragma unroll
  for (int k = 0; k < K; ++k) {
    S[k] = __fdiv_rn(__fsub_rn(mx[k], mn[k]), 255.0f);
    inv[k] = S[k] >= 1.17549435e-38f ? __frcp_rn(S[k]) : 0.0f;  // 0: constant segment
    if (head) reinterpret_cast<float2*>(p.hdr)[v * K + k] = make_float2(S[k], mn[k]);
  }
}

template <int K>
__device__ __forceinline__ void store_codes(uint8_t* dst, const uint32_t (&q)[K]) {
  if constexpr (K == 1) {
    *dst = (uint8_t)q[0];
  } else if constexpr (K == 2) {
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(q[0] | (q[1] << 8));
  } else if constexpr (K == 4) {
    *reinterpret_cast<uint32_t*>(dst) = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
  } else {
    *reinterpret_cast<uint2*>(dst) = make_uint2(q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24),
                                                q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24));
  }
}

// Codes of this thread's edges e = first, first + stride, ...
template <int K>
__device__ __forceinline__ void eq_codes(const EdgeQuantParams& p, int64_t first, int64_t end, int64_t stride,
                                         const float (&mn)[K], const float (&inv)[K]) {
  for (int64_t e = first; e < end; e += stride) {
    float a[K];
    load_k<K>(p.alpha + e * K, a);
    const uint32_t kr = row_key(p.seed_key, (uint32_t)e);
    uint32_t q[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      q[k] = 0;
      if (inv[k] != 0.0f) {
        const float s = __fadd_rn(__fmul_rn(__fsub_rn(a[k], mn[k]), inv[k]), noise_u(kr, (uint32_t)k));
        // floor(s) for s in [0, 2^23): add 2^23 rounding down, read the mantissa
        q[k] = min(__float_as_uint(__fadd_rd(s, 8388608.0f)) - 0x4B000000u, 255u);
      }
    }
    store_codes<K>(p.codes + e * K, q);
  }
}

template <int K>
__global__ void __launch_bounds__(kGatThreads) edge_quant_kernel(const EdgeQuantParams p) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t gw = (int64_t)blockIdx.x * kGatWarps + w;
  const int64_t nw = (int64_t)gridDim.x * kGatWarps;
  // heavy rows: (min, max) of each task's edges into part[task]
  for (int64_t t = gw; t < p.sc.n_tasks; t += nw) {
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.sc.tasks) + t);
    float mn[K], mx[K];
    const bool ok = eq_range_ok(p, task.x, task.y, task.z);
    eq_minmax<K>(p, (int64_t)task.y + lane, ok ? task.z : task.y, 32, mn, mx);
    warp_minmax<K>(mn, mx);
    if (lane == 0) {
      float* mine = p.sc.partial + t * 2 * K;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        mine[2 * k] = mn[k];
        mine[2 * k + 1] = mx[k];
      }
    }
  }
  // light rows in groups of 32 consecutive rows per warp: a row of at most
  // 32 edges is one thread's; the group's rows of 33 .. hub_threshold edges
  // are then taken one at a time by the whole warp
  const int64_t groups = (p.n_rows + 31) / 32;
  for (int64_t grp = gw; grp < groups; grp += nw) {
    const int64_t r = grp * 32 + lane;
    int64_t a = 0, b = 0;
    if (r < p.n_rows) {
      a = __ldg(p.rowptr + r);
      b = __ldg(p.rowptr + r + 1);
    }
    if (r < p.n_rows && !eq_range_ok(p, r, a, b)) {
      b = a;  // skipped: neither a thread row nor a warp row
    } else if (r < p.n_rows && b == a) {
#pragma unroll
      for (int k = 0; k < K; ++k) reinterpret_cast<float2*>(p.hdr)[r * K + k] = make_float2(0.0f, 0.0f);
    } else if (r < p.n_rows && b - a <= 32) {
      float mn[K], mx[K], S[K], inv[K];
      eq_minmax<K>(p, a, b, 1, mn, mx);
      eq_scale<K>(p, r, mn, mx, true, S, inv);
      eq_codes<K>(p, a, b, 1, mn, inv);
    }
    unsigned mid = __ballot_sync(FULL, r < p.n_rows && b - a > 32 && b - a <= p.sc.hub_threshold);
    while (mid != 0) {
      const int l0 = __ffs(mid) - 1;
      mid &= mid - 1;
      const int64_t v = grp * 32 + l0;
      const int64_t va = __shfl_sync(FULL, a, l0), vb = __shfl_sync(FULL, b, l0);
      float mn[K], mx[K], S[K], inv[K];
      eq_minmax<K>(p, va + lane, vb, 32, mn, mx);
      warp_minmax<K>(mn, mx);
      eq_scale<K>(p, v, mn, mx, lane == 0, S, inv);
      eq_codes<K>(p, va + lane, vb, 32, mn, inv);
    }
  }
}

// Heavy rows, second kernel: one warp per task merges the (min, max) of its
// row's tasks, the row's first task writes the header, every task its codes.
template <int K>
__global__ void __launch_bounds__(kGatThreads) edge_quant_heavy_kernel(const EdgeQuantParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= p.sc.n_tasks) return;
  const int4 task = __ldg(reinterpret_cast<const int4*>(p.sc.tasks) + t);
  int64_t t0 = t, nt = 1;
  if (task.w >= 0) {
    const int4 grp = __ldg(reinterpret_cast<const int4*>(p.sc.groups) + task.w);
    t0 = grp.y;
    nt = grp.z;
  }
  if (!eq_range_ok(p, task.x, task.y, task.z) || t0 < 0 || t0 + nt > p.sc.n_tasks || t < t0 || t >= t0 + nt) {
    atomicCAS(p.err, 0, kEdgeQuantBadRange);
    return;
  }
  float mn[K], mx[K], S[K], inv[K];
  const float* base = p.sc.partial + t0 * 2 * K;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    mn[k] = __ldcg(base + 2 * k);
    mx[k] = __ldcg(base + 2 * k + 1);
    for (int64_t i = 1; i < nt; ++i) {
      mn[k] = fminf(mn[k], __ldcg(base + i * 2 * K + 2 * k));
      mx[k] = fmaxf(mx[k], __ldcg(base + i * 2 * K + 2 * k + 1));
    }
  }
  eq_scale<K>(p, task.x, mn, mx, t == t0 && lane == 0, S, inv);
  eq_codes<K>(p, (int64_t)task.y + lane, task.z, 32, mn, inv);
}

// AdaQP Eqn 5 on the attention codes: deq[e,k] = fmaf(q, S[v,k], Z[v,k]),
// one kernel over the same thread / warp rows and heavy-row warp tasks.
template <int K>
__device__ __forceinline__ void eq_expand(const EdgeQuantParams& p, int64_t v, int64_t first, int64_t end,
                                          int64_t stride) {
  float2 h[K];
#pragma unroll
  for (int k = 0; k < K; ++k) h[k] = __ldg(reinterpret_cast<const float2*>(p.hdr) + v * K + k);
  for (int64_t e = first; e < end; e += stride) {
    uint32_t w[(K + 3) / 4];
    if constexpr (K == 8) {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(p.codes + e * K));
      w[0] = x.x;
      w[1] = x.y;
    } else if constexpr (K == 4) {
      w[0] = __ldg(reinterpret_cast<const uint32_t*>(p.codes + e * K));
    } else if constexpr (K == 2) {
      w[0] = __ldg(reinterpret_cast<const uint16_t*>(p.codes + e * K));
    } else {
      w[0] = __ldg(p.codes + e);
    }
    float a[K];
#pragma unroll
    for (int k = 0; k < K; ++k) a[k] = __fmaf_rn(code_to_float((w[k >> 2] >> (8 * (k & 3))) & 0xFFu), h[k].x, h[k].y);
    store_k<K>(p.deq + e * K, a);
  }
}

template <int K>
__global__ void __launch_bounds__(kGatThreads) edge_dequant_kernel(const EdgeQuantParams p) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t gw = (int64_t)blockIdx.x * kGatWarps + w;
  const int64_t nw = (int64_t)gridDim.x * kGatWarps;
  for (int64_t t = gw; t < p.sc.n_tasks; t += nw) {
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.sc.tasks) + t);
    if (eq_range_ok(p, task.x, task.y, task.z)) eq_expand<K>(p, task.x, (int64_t)task.y + lane, task.z, 32);
  }
  const int64_t groups = (p.n_rows + 31) / 32;
  for (int64_t grp = gw; grp < groups; grp += nw) {
    const int64_t r = grp * 32 + lane;
    int64_t a = 0, b = 0;
    if (r < p.n_rows) {
      a = __ldg(p.rowptr + r);
      b = __ldg(p.rowptr + r + 1);
    }
    if (r < p.n_rows && !eq_range_ok(p, r, a, b)) b = a;
    if (r < p.n_rows && b - a <= 32) eq_expand<K>(p, r, a, b, 1);
    unsigned mid = __ballot_sync(FULL, r < p.n_rows && b - a > 32 && b - a <= p.sc.hub_threshold);
    while (mid != 0) {
      const int l0 = __ffs(mid) - 1;
      mid &= mid - 1;
      const int64_t va = __shfl_sync(FULL, a, l0), vb = __shfl_sync(FULL, b, l0);
      eq_expand<K>(p, grp * 32 + l0, va + lane, vb, 32);
    }
  }
}

// --------------------------------------------------- GAT edge backward ---
struct EdgeBwdParams {
  const int32_t* rowptr;
  const int32_t* col;
  const float* dOut;   // n x d, ld = d
  MsgSrc msg;          // forward messages m_u (H' or its de-quantized rows)
  const float* alpha;  // E x K
  const float* S;
  const float* D;      // n x K
  float slope;
  float* dEpre;        // E x K (holds dalpha of the rows of more than 32 edges between the passes)
  float* dD;           // n x K
  int64_t n_rows;
  int d, lph;          // lanes per head = F / 8
  const int32_t* light;  // runs of light rows
  int64_t n_light;
  Sched sc;            // heavy-row tasks
  float* Ppart;        // [task][K] sum of alpha dalpha over the task's edges
  float* dDpart;       // [task][K] sum of dE_pre over the task's edges
};

template <int K>
__device__ __forceinline__ void warp_sum(float (&x)[K]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int k = 0; k < K; ++k) x[k] += __shfl_xor_sync(FULL, x[k], o);
}

// The SDDMM dot of the 32 edges [c0, c0 + cnt) (cnt <= 32; lane j holds
// edge c0 + j's column id x): all lanes on one edge at a time, lane l owning
// columns 8l .. 8l+7, U gathers in flight; the per-head sum ends in
// sda[t * K + head] for edge c0 + t.
template <int BITS, int K, int U>
__device__ __forceinline__ void eb_dots(const EdgeBwdParams& p, int cnt, int32_t x, bool qx, const float (&g)[8],
                                        float* sda) {
  const int lane = threadIdx.x & 31;
  const bool live = lane < (p.d >> 3);
  const int head = live ? lane / p.lph : 0;
  const bool leader = live && lane % p.lph == 0;
  for (int t0 = 0; t0 < cnt; t0 += U) {
    RawChunk<BITS> r[U];
#pragma unroll
    for (int t = 0; t < U; ++t) {
      const int32_t xt = __shfl_sync(FULL, x, (t0 + t) & 31);
      const bool qt = BITS < 32 && __shfl_sync(FULL, (int)qx, (t0 + t) & 31) != 0;
      if (live && t0 + t < cnt) load_raw<BITS>(p.msg, xt, qt, lane, r[t]);
    }
#pragma unroll
    for (int t = 0; t < U; ++t) {
      float dot = 0.0f;
      if (live && t0 + t < cnt) {
        float v[8];
        decode<BITS>(r[t], v);
#pragma unroll
        for (int i = 0; i < 8; ++i) dot = __fmaf_rn(g[i], v[i], dot);
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1)
        if (o < p.lph) dot += __shfl_xor_sync(FULL, dot, o);
      if (leader && t0 + t < cnt) sda[(t0 + t) * K + head] = dot;
    }
  }
}

// dE_pre of one edge from dalpha, P and the LeakyReLU branch of its score.
template <int K>
__device__ __forceinline__ void eb_grad(const EdgeBwdParams& p, const float (&a)[K], const float (&da)[K],
                                        const float (&P)[K], const float (&s)[K], const float (&dv)[K],
                                        float (&dE)[K]) {
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const float t = a[k] * (da[k] - P[k]);
    dE[k] = (s[k] + dv[k]) > 0.0f ? t : p.slope * t;
  }
}

// Pass 1 over the edges [e0, e1) of one destination row (or a part of one):
// the SDDMM dots, stored to dEpre when `keep` (the pass 2 reads them back),
// and this lane's part of P = sum alpha dalpha.  For a single batch of at
// most 32 edges the lane's edge, alpha, dalpha and S row stay in registers.
template <int BITS, int K, int U>
__device__ __forceinline__ void eb_pass1(const EdgeBwdParams& p, int64_t e0, int64_t e1, const float (&g)[8],
                                         float* sda, bool keep, float (&P)[K], int32_t& x, float (&a)[K],
                                         float (&da)[K], float (&s)[K]) {
  const int lane = threadIdx.x & 31;
  x = 0;
#pragma unroll
  for (int k = 0; k < K; ++k) P[k] = a[k] = da[k] = s[k] = 0.0f;
  for (int64_t c0 = e0; c0 < e1; c0 += 32) {
    const int64_t e = c0 + lane;
    const bool has = e < e1;
    x = has ? __ldg(p.col + e) : 0;
    const bool qx = has && is_quant<BITS>(p.msg, x);
#pragma unroll
    for (int k = 0; k < K; ++k) a[k] = 0.0f;
    if (has) load_k<K>(p.alpha + e * K, a);
    if (!keep && has) load_k<K>(p.S + (int64_t)x * K, s);  // for pass 2, in flight during the dots
    eb_dots<BITS, K, U>(p, (int)min((int64_t)32, e1 - c0), x, qx, g, sda);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < K; ++k) da[k] = has ? sda[lane * K + k] : 0.0f;
    __syncwarp();  // sda is rewritten by the next batch
    if (keep && has) store_k<K>(p.dEpre + e * K, da);
#pragma unroll
    for (int k = 0; k < K; ++k) P[k] = __fmaf_rn(a[k], da[k], P[k]);
  }
}

// Pass 2 over [e0, e1) reading dalpha back from dEpre (thread per edge,
// `stride` threads); returns the thread's part of dD.
template <int K>
__device__ __forceinline__ void eb_pass2_mem(const EdgeBwdParams& p, int64_t v, int64_t first, int64_t e1,
                                             int64_t stride, const float (&P)[K], float (&dd)[K]) {
  float dv[K];
  load_k<K>(p.D + v * K, dv);
#pragma unroll
  for (int k = 0; k < K; ++k) dd[k] = 0.0f;
  for (int64_t e = first; e < e1; e += stride) {
    float s[K], a[K], da[K], dE[K];
    load_k<K>(p.S + (int64_t)__ldg(p.col + e) * K, s);
    load_k<K>(p.alpha + e * K, a);
#pragma unroll
    for (int k = 0; k < K; ++k) da[k] = __ldcg(p.dEpre + e * K + k);
    eb_grad<K>(p, a, da, P, s, dv, dE);
    store_k<K>(p.dEpre + e * K, dE);
#pragma unroll
    for (int k = 0; k < K; ++k) dd[k] += dE[k];
  }
}

// Light rows (at most the hub threshold in-edges), one warp per row over the
// graph's runs of light rows; heavy rows: first pass of each task, one block
// per task, its eight warps on contiguous parts of the task's edges, the
// task's P partial to Ppart.  gat_edge_bwd_heavy_kernel finishes them.
template <int BITS, int K>
__global__ void __launch_bounds__(kGatThreads, K <= 4 ? 4 : 3) gat_edge_bwd_kernel(const EdgeBwdParams p) {
  constexpr int U = 2;
  __shared__ float sda_all[kGatWarps][32 * K];
  __shared__ float red[kGatWarps][K];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const bool live = lane < (p.d >> 3);
  float* sda = sda_all[w];
  float g[8];
  float P[K], a[K], da[K], s[K];
  int32_t x;
  if ((int64_t)blockIdx.x < p.sc.n_tasks) {
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.sc.tasks) + blockIdx.x);
    const int64_t v = task.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = 0.0f;
    if (live) {
      const float4 u0 = ldg_f4(p.dOut + v * p.d + lane * 8), u1 = ldg_f4(p.dOut + v * p.d + lane * 8 + 4);
      g[0] = u0.x; g[1] = u0.y; g[2] = u0.z; g[3] = u0.w; g[4] = u1.x; g[5] = u1.y; g[6] = u1.z; g[7] = u1.w;
    }
    const int len = task.z - task.y;
    const int chunk = (len + kGatWarps - 1) / kGatWarps;
    const int64_t b0 = min(task.y + w * chunk, task.z), b1 = min(b0 + chunk, (int64_t)task.z);
    eb_pass1<BITS, K, U>(p, b0, b1, g, sda, true, P, x, a, da, s);
    warp_sum<K>(P);
    if (lane == 0)
#pragma unroll
      for (int k = 0; k < K; ++k) red[w][k] = P[k];
    __syncthreads();
    if (threadIdx.x < K) {
      float t = 0.0f;
      for (int ww = 0; ww < kGatWarps; ++ww) t += red[ww][threadIdx.x];
      p.Ppart[(int64_t)blockIdx.x * K + threadIdx.x] = t;
    }
    return;
  }
  const int64_t gw = ((int64_t)blockIdx.x - p.sc.n_tasks) * kGatWarps + w;
  const int64_t nw = ((int64_t)gridDim.x - p.sc.n_tasks) * kGatWarps;
  for (int64_t t = gw; t < p.n_light; t += nw) {
    const int2 run = __ldg(reinterpret_cast<const int2*>(p.light) + t);
    int64_t b = __ldg(p.rowptr + run.x);
    for (int64_t v = run.x; v < run.y; ++v) {
      const int64_t a0 = b;
      b = __ldg(p.rowptr + v + 1);
      const bool one = b - a0 <= 32;
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = 0.0f;
      if (live && b > a0) {
        const float4 u0 = ldg_f4(p.dOut + v * p.d + lane * 8), u1 = ldg_f4(p.dOut + v * p.d + lane * 8 + 4);
        g[0] = u0.x; g[1] = u0.y; g[2] = u0.z; g[3] = u0.w; g[4] = u1.x; g[5] = u1.y; g[6] = u1.z; g[7] = u1.w;
      }
      eb_pass1<BITS, K, U>(p, a0, b, g, sda, !one, P, x, a, da, s);
      float dv[K];
      load_k<K>(p.D + v * K, dv);
      warp_sum<K>(P);
      float dd[K];
      if (one) {
        const bool has = a0 + lane < b;
        float dE[K];
        eb_grad<K>(p, a, da, P, s, dv, dE);
        if (has) store_k<K>(p.dEpre + (a0 + lane) * K, dE);
#pragma unroll
        for (int k = 0; k < K; ++k) dd[k] = has ? dE[k] : 0.0f;
      } else {
        eb_pass2_mem<K>(p, v, a0 + lane, b, 32, P, dd);
      }
      warp_sum<K>(dd);
      if (lane == 0) store_k<K>(p.dD + v * K, dd);
    }
  }
}

// Second pass of the heavy rows, one block per task: P of the row (the
// row's task partials summed in task order), dE_pre of the task's edges
// (thread per edge), the task's dD partial; the last block of a split row
// sums the partials in task order into dD.
template <int K>
__global__ void __launch_bounds__(kGatThreads) gat_edge_bwd_heavy_kernel(const EdgeBwdParams p) {
  __shared__ float red[kGatWarps][K];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int4 task = __ldg(reinterpret_cast<const int4*>(p.sc.tasks) + blockIdx.x);
  int t0 = blockIdx.x, nt = 1;
  if (task.w >= 0) {
    const int4 grp = __ldg(reinterpret_cast<const int4*>(p.sc.groups) + task.w);
    t0 = grp.y;
    nt = grp.z;
  }
  float P[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    P[k] = 0.0f;
    for (int i = 0; i < nt; ++i) P[k] += __ldcg(p.Ppart + (int64_t)(t0 + i) * K + k);
  }
  float dd[K];
  eb_pass2_mem<K>(p, task.x, task.y + threadIdx.x, task.z, kGatThreads, P, dd);
  warp_sum<K>(dd);
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < K; ++k) red[w][k] = dd[k];
  __syncthreads();
  float t = 0.0f;
  if (threadIdx.x < K)
    for (int ww = 0; ww < kGatWarps; ++ww) t += red[ww][threadIdx.x];
  if (task.w < 0) {
    if (threadIdx.x < K) p.dD[(int64_t)task.x * K + threadIdx.x] = t;
    return;
  }
  if (threadIdx.x < K) p.dDpart[(int64_t)blockIdx.x * K + threadIdx.x] = t;
  if (!last_of_group(p.sc, task.w, nt)) return;
  if (threadIdx.x < K) {
    float r = 0.0f;
    for (int i = 0; i < nt; ++i) r += __ldcg(p.dDpart + (int64_t)(t0 + i) * K + threadIdx.x);
    p.dD[(int64_t)task.x * K + threadIdx.x] = r;
  }
}

// --------------------------------------------------- GAT node backward ---
struct NodeBwdParams {
  const int32_t* tr_rowptr;
  const int32_t* tr_perm;
  const float* dEpre;   // E x K (by CSR edge id)
  const float* dD;      // n x K
  const float* dM;      // n x d
  const float* Hp;      // n x d
  const float* a_src;   // d
  const float* a_dst;   // d
  __nv_bfloat16* dHp;   // n x ldb (bf16, for the GEMMs)
  int64_t ldb;
  float* dHp32;         // optional n x d fp32 copy
  float* dS;            // optional n x K
  float* dSh;           // n x K: dS of the rows above the hub threshold (gat_node_heavy_kernel)
  float* part;          // [block][2 d] partial da_src | da_dst
  int64_t n_rows;
  int d, fshift;
  Sched sc;             // the transposed graph's heavy-row tasks
};

__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// dS[u] = sum over the out-edges of u of dE_pre, for the rows above the hub
// threshold: one block per task of the transposed schedule, four edges per
// thread in flight; the tasks of a split row are summed in task order by
// the last block of the row.
template <int K>
__global__ void __launch_bounds__(kGatThreads) gat_node_heavy_kernel(const NodeBwdParams p) {
  __shared__ float red[kGatWarps][K];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int4 task = __ldg(reinterpret_cast<const int4*>(p.sc.tasks) + blockIdx.x);
  float ds[K];
#pragma unroll
  for (int k = 0; k < K; ++k) ds[k] = 0.0f;
  for (int64_t e = task.y + threadIdx.x; e < task.z; e += 4 * kGatThreads) {
    int32_t pe[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) pe[t] = e + t * kGatThreads < task.z ? __ldg(p.tr_perm + e + t * kGatThreads) : -1;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (pe[t] >= 0) {
        float x[K];
        load_k<K>(p.dEpre + (int64_t)pe[t] * K, x);
#pragma unroll
        for (int k = 0; k < K; ++k) ds[k] += x[k];
      }
    }
  }
  warp_sum<K>(ds);
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < K; ++k) red[w][k] = ds[k];
  __syncthreads();
  float t = 0.0f;
  if (threadIdx.x < K)
    for (int ww = 0; ww < kGatWarps; ++ww) t += red[ww][threadIdx.x];
  if (task.w < 0) {
    if (threadIdx.x < K) p.dSh[(int64_t)task.x * K + threadIdx.x] = t;
    return;
  }
  const int4 grp = __ldg(reinterpret_cast<const int4*>(p.sc.groups) + task.w);
  if (threadIdx.x < K) p.sc.partial[(int64_t)(grp.w + ((int)blockIdx.x - grp.y)) * K + threadIdx.x] = t;
  if (!last_of_group(p.sc, task.w, grp.z)) return;
  if (threadIdx.x < K) {
    float r = 0.0f;
    for (int i = 0; i < grp.z; ++i) r += __ldcg(p.sc.partial + (int64_t)(grp.w + i) * K + threadIdx.x);
    p.dSh[(int64_t)task.x * K + threadIdx.x] = r;
  }
}

// One warp per group of 32 consecutive source rows u:
//   dS[u]  : a row of at most 32 out-edges is one lane's (its edges in order,
//            four in flight, two for 8 heads); rows up to the hub threshold are the whole
//            warp's; heavier rows were summed by gat_node_heavy_kernel;
//   dH'[u] = dM[u] + dS[u,k] a_src + dD[u,k] a_dst, two rows at a time,
//            lane l owning columns 8l .. 8l+7, with the partial sums of
//            da_src = sum_u dS[u,k] H'[u] and da_dst = sum_u dD[u,k] H'[u].
template <int K>
__global__ void __launch_bounds__(kGatThreads, K == 8 ? 2 : 3) gat_node_bwd_kernel(const NodeBwdParams p) {
  constexpr int UE = K <= 4 ? 4 : 2;  // out-edges in flight per lane
  extern __shared__ float sm[];  // [kGatWarps][2 d]
  __shared__ float sds[kGatWarps][32 * K];
  __shared__ __align__(16) float sa[2][256];  // a_src | a_dst
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nchunks = p.d >> 3;
  const bool live = lane < nchunks;
  const int head = live ? (lane * 8) >> p.fshift : 0;
  for (int j = threadIdx.x; j < p.d; j += blockDim.x) {
    sa[0][j] = __ldg(p.a_src + j);
    sa[1][j] = __ldg(p.a_dst + j);
  }
  __syncthreads();
  float acc_s[8] = {}, acc_d[8] = {};
  float* myds = sds[w];
  const int64_t groups = (p.n_rows + 31) / 32;
  for (int64_t grp = (int64_t)blockIdx.x * kGatWarps + w; grp < groups; grp += (int64_t)gridDim.x * kGatWarps) {
    const int64_t u0 = grp * 32;
    const int rows = (int)min((int64_t)32, p.n_rows - u0);
    // dS of the group's rows
    int64_t a = 0, b = 0;
    if (lane < rows) {
      a = __ldg(p.tr_rowptr + u0 + lane);
      b = __ldg(p.tr_rowptr + u0 + lane + 1);
    }
    float ds[K];
#pragma unroll
    for (int k = 0; k < K; ++k) ds[k] = 0.0f;
    if (b - a > p.sc.hub_threshold) {
      load_k<K>(p.dSh + (u0 + lane) * K, ds);
    } else if (b - a <= 32) {
      for (int64_t e = a; e < b; e += UE) {
        int32_t pe[UE];
#pragma unroll
        for (int t = 0; t < UE; ++t) pe[t] = e + t < b ? __ldg(p.tr_perm + e + t) : -1;
#pragma unroll
        for (int t = 0; t < UE; ++t) {
          if (pe[t] >= 0) {
            float x[K];
            load_k<K>(p.dEpre + (int64_t)pe[t] * K, x);
#pragma unroll
            for (int k = 0; k < K; ++k) ds[k] += x[k];
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < K; ++k) myds[lane * K + k] = ds[k];
    __syncwarp();  // lane 0 overwrites the slots of the warp-summed rows below
    unsigned mid = __ballot_sync(FULL, b - a > 32 && b - a <= p.sc.hub_threshold);
    while (mid != 0) {
      const int l0 = __ffs(mid) - 1;
      mid &= mid - 1;
      const int64_t va = __shfl_sync(FULL, a, l0), vb = __shfl_sync(FULL, b, l0);
      float hs[K];
#pragma unroll
      for (int k = 0; k < K; ++k) hs[k] = 0.0f;
      for (int64_t e = va + lane; e < vb; e += UE * 32) {
        int32_t pe[UE];
#pragma unroll
        for (int t = 0; t < UE; ++t) pe[t] = e + 32 * t < vb ? __ldg(p.tr_perm + e + 32 * t) : -1;
#pragma unroll
        for (int t = 0; t < UE; ++t) {
          if (pe[t] >= 0) {
            float x[K];
            load_k<K>(p.dEpre + (int64_t)pe[t] * K, x);
#pragma unroll
            for (int k = 0; k < K; ++k) hs[k] += x[k];
          }
        }
      }
      warp_sum<K>(hs);
      if (lane == 0)
#pragma unroll
        for (int k = 0; k < K; ++k) myds[l0 * K + k] = hs[k];
    }
    __syncwarp();
    if (p.dS != nullptr)
      for (int j = lane; j < rows * K; j += 32) p.dS[u0 * K + j] = myds[j];
    // dH' and the da partials, two rows at a time
    for (int i = 0; i < rows; i += 2) {
      float4 m[2][2], h[2][2];
      float dsh[2], ddh[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int64_t u = u0 + i + r;
        if (live && i + r < rows) {
          m[r][0] = ldg_f4(p.dM + u * p.d + lane * 8);
          m[r][1] = ldg_f4(p.dM + u * p.d + lane * 8 + 4);
          h[r][0] = ldg_f4(p.Hp + u * p.d + lane * 8);
          h[r][1] = ldg_f4(p.Hp + u * p.d + lane * 8 + 4);
          ddh[r] = __ldg(p.dD + u * K + head);
          dsh[r] = myds[(i + r) * K + head];
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int64_t u = u0 + i + r;
        if (!live || i + r >= rows) continue;
        const float mv[8] = {m[r][0].x, m[r][0].y, m[r][0].z, m[r][0].w, m[r][1].x, m[r][1].y, m[r][1].z, m[r][1].w};
        const float hv[8] = {h[r][0].x, h[r][0].y, h[r][0].z, h[r][0].w, h[r][1].x, h[r][1].y, h[r][1].z, h[r][1].w};
        const float4 as0 = *reinterpret_cast<const float4*>(&sa[0][lane * 8]);
        const float4 as1 = *reinterpret_cast<const float4*>(&sa[0][lane * 8 + 4]);
        const float4 ad0 = *reinterpret_cast<const float4*>(&sa[1][lane * 8]);
        const float4 ad1 = *reinterpret_cast<const float4*>(&sa[1][lane * 8 + 4]);
        const float as[8] = {as0.x, as0.y, as0.z, as0.w, as1.x, as1.y, as1.z, as1.w};
        const float ad[8] = {ad0.x, ad0.y, ad0.z, ad0.w, ad1.x, ad1.y, ad1.z, ad1.w};
        float o[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          o[c] = mv[c] + dsh[r] * as[c] + ddh[r] * ad[c];
          acc_s[c] = __fmaf_rn(dsh[r], hv[c], acc_s[c]);
          acc_d[c] = __fmaf_rn(ddh[r], hv[c], acc_d[c]);
        }
        *reinterpret_cast<uint4*>(p.dHp + u * p.ldb + lane * 8) =
            make_uint4(bf2(o[0], o[1]), bf2(o[2], o[3]), bf2(o[4], o[5]), bf2(o[6], o[7]));
        if (p.dHp32 != nullptr) {
          st_f4(p.dHp32 + u * p.d + lane * 8, o[0], o[1], o[2], o[3]);
          st_f4(p.dHp32 + u * p.d + lane * 8 + 4, o[4], o[5], o[6], o[7]);
        }
      }
    }
    __syncwarp();  // the group's dS slots are rewritten by the next group
  }
  if (live)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sm[w * 2 * p.d + lane * 8 + i] = acc_s[i];
      sm[w * 2 * p.d + p.d + lane * 8 + i] = acc_d[i];
    }
  __syncthreads();
  for (int j = threadIdx.x; j < 2 * p.d; j += blockDim.x) {
    float t = 0.0f;
    for (int ww = 0; ww < kGatWarps; ++ww) t += sm[ww * 2 * p.d + j];
    p.part[(int64_t)blockIdx.x * 2 * p.d + j] = t;
  }
}

__global__ void sum_blocks_kernel(const float* __restrict__ part, int blocks, int n, float* out_a, float* out_b,
                                  int split) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= n) return;
  float t = 0.0f;
  for (int b = 0; b < blocks; ++b) t += part[(int64_t)b * n + j];
  if (j < split)
    out_a[j] = t;
  else
    out_b[j - split] = t;
}

Sched make_sched(const gq_sched& s, int hub_threshold, void* ws, int per_slot_floats) {
  Sched r{};
  r.tasks = s.tasks;
  r.groups = s.groups;
  r.n_tasks = s.n_tasks;
  r.hub_threshold = hub_threshold;
  if (s.n_groups > 0) {
    r.partial = static_cast<float*>(ws);
    r.tickets = reinterpret_cast<int*>(static_cast<char*>(ws) +
                                       ((size_t)s.n_slots * per_slot_floats * sizeof(float) + 255) / 256 * 256);
  }
  return r;
}

size_t sched_ws(const gq_sched& s, int per_slot_floats) {
  if (s.n_groups == 0) return 0;
  return ((size_t)s.n_slots * per_slot_floats * sizeof(float) + 255) / 256 * 256 + (size_t)s.n_groups * 4 + 256;
}

int light_grid(int64_t n_rows, int64_t n_tasks) {
  int64_t blocks = (n_rows + kGatWarps - 1) / kGatWarps;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)(blocks + n_tasks);
}

template <int K>
int launch_softmax(const SoftmaxParams& p, cudaStream_t s) {
  int64_t blocks = ((p.n_rows + 31) / 32 + p.sc.n_tasks + kGatWarps - 1) / kGatWarps;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  edge_softmax_kernel<K><<<(unsigned)blocks, kGatThreads, 0, s>>>(p);
  GQ_TRY(launch_status());
  if (p.sc.n_tasks > 0) {
    edge_softmax_heavy_kernel<K><<<(unsigned)((p.sc.n_tasks + kGatWarps - 1) / kGatWarps), kGatThreads, 0, s>>>(p);
    GQ_TRY(launch_status());
  }
  return GQ_OK;
}

template <int K>
int launch_edge_quant(const EdgeQuantParams& p, cudaStream_t s) {
  int64_t blocks = ((p.n_rows + 31) / 32 + p.sc.n_tasks + kGatWarps - 1) / kGatWarps;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  edge_quant_kernel<K><<<(unsigned)blocks, kGatThreads, 0, s>>>(p);
  GQ_TRY(launch_status());
  if (p.sc.n_tasks > 0) {
    edge_quant_heavy_kernel<K><<<(unsigned)((p.sc.n_tasks + kGatWarps - 1) / kGatWarps), kGatThreads, 0, s>>>(p);
    GQ_TRY(launch_status());
  }
  return GQ_OK;
}

template <int K>
int launch_edge_dequant(const EdgeQuantParams& p, cudaStream_t s) {
  int64_t blocks = ((p.n_rows + 31) / 32 + p.sc.n_tasks + kGatWarps - 1) / kGatWarps;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  edge_dequant_kernel<K><<<(unsigned)blocks, kGatThreads, 0, s>>>(p);
  return launch_status();
}

template <int BITS, int K>
int launch_edge_bwd(const EdgeBwdParams& p, cudaStream_t s) {
  int64_t light = (p.n_light + kGatWarps - 1) / kGatWarps;
  const int64_t cap = (int64_t)sm_count() * (K <= 4 ? 4 : 3);
  if (light > cap) light = cap;
  if (light < 1) light = 1;
  gat_edge_bwd_kernel<BITS, K><<<(unsigned)(light + p.sc.n_tasks), kGatThreads, 0, s>>>(p);
  GQ_TRY(launch_status());
  if (p.sc.n_tasks > 0) {
    gat_edge_bwd_heavy_kernel<K><<<(unsigned)p.sc.n_tasks, kGatThreads, 0, s>>>(p);
    GQ_TRY(launch_status());
  }
  return GQ_OK;
}

}  // namespace

// ---------------------------------------------------------------- API ---
// one (max, sum) pair per head for every heavy-row task
size_t edge_softmax_workspace(const gq_graph* g, int heads) {
  return ((size_t)g->sched.n_tasks * 2 * heads * sizeof(float) + 255) / 256 * 256;
}
// [task][K] P partials | [task][K] dD partials | tickets of the split rows
size_t edge_bwd_workspace(const gq_graph* g, int heads) {
  if (g->sched.n_tasks == 0) return 0;
  const size_t part = ((size_t)g->sched.n_tasks * heads * sizeof(float) + 255) / 256 * 256;
  return 2 * part + ((size_t)g->sched.n_groups * sizeof(int) + 255) / 256 * 256;
}

int edge_softmax(const gq_graph* g, const float* S, const float* D, int heads, float slope, float* Epre,
                 float* alpha, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (g == nullptr) return GQ_ERR_INVALID_ARG;
  if (!(heads == 1 || heads == 2 || heads == 4 || heads == 8)) return GQ_ERR_UNSUPPORTED;
  if (g->nnz == 0) return GQ_OK;  // no edges: nothing to score
  if (S == nullptr || D == nullptr || alpha == nullptr) return GQ_ERR_INVALID_ARG;
  if (!aligned(S, 16) || !aligned(D, 16) || !aligned(alpha, 16) || (Epre != nullptr && !aligned(Epre, 16)))
    return GQ_ERR_INVALID_ARG;
  SoftmaxParams p{};
  p.rowptr = g->rowptr;
  p.col = g->col;
  p.S = S;
  p.D = D;
  p.slope = slope;
  p.alpha = alpha;
  p.Epre = Epre;
  p.n_rows = g->n;
  p.n_edges = g->nnz;
  p.n_groups = g->sched.n_groups;
  p.err = g->status;
  const size_t need = edge_softmax_workspace(g, heads);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !aligned(ws, 256))) return GQ_ERR_WORKSPACE;
  p.sc = make_sched(g->sched, g->hub_threshold, nullptr, 2 * heads);
  p.sc.partial = static_cast<float*>(ws);
  switch (heads) {
    case 1: return launch_softmax<1>(p, s);
    case 2: return launch_softmax<2>(p, s);
    case 4: return launch_softmax<4>(p, s);
    default: return launch_softmax<8>(p, s);
  }
}

// 8-bit attention values: one (min, max) pair per head for every heavy-row task
size_t edge_quant_workspace(const gq_graph* g, int heads) { return edge_softmax_workspace(g, heads); }

int quantize_edge_values(const gq_graph* g, const float* alpha, int heads, uint64_t seed, uint8_t* codes, float* hdr,
                         void* ws, size_t ws_bytes, cudaStream_t s) {
  if (g == nullptr || hdr == nullptr) return GQ_ERR_INVALID_ARG;
  if (!(heads == 1 || heads == 2 || heads == 4 || heads == 8)) return GQ_ERR_UNSUPPORTED;
  // with no edges alpha and codes are empty (and may be NULL); the headers are still written
  if (g->nnz > 0 && (alpha == nullptr || codes == nullptr)) return GQ_ERR_INVALID_ARG;
  if (!aligned(alpha, 16) || !aligned(codes, 16) || !aligned(hdr, 16)) return GQ_ERR_INVALID_ARG;
  const size_t need = edge_quant_workspace(g, heads);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !aligned(ws, 256))) return GQ_ERR_WORKSPACE;
  EdgeQuantParams p{};
  p.rowptr = g->rowptr;
  p.alpha = alpha;
  p.codes = codes;
  p.hdr = hdr;
  p.seed_key = seed_key_host(seed);
  p.n_rows = g->n;
  p.n_edges = g->nnz;
  p.err = g->status;
  p.sc = make_sched(g->sched, g->hub_threshold, nullptr, 2 * heads);
  p.sc.partial = static_cast<float*>(ws);
  switch (heads) {
    case 1: return launch_edge_quant<1>(p, s);
    case 2: return launch_edge_quant<2>(p, s);
    case 4: return launch_edge_quant<4>(p, s);
    default: return launch_edge_quant<8>(p, s);
  }
}

int dequant_edge_values(const gq_graph* g, const uint8_t* codes, const float* hdr, int heads, float* out,
                        cudaStream_t s) {
  if (g == nullptr) return GQ_ERR_INVALID_ARG;
  if (!(heads == 1 || heads == 2 || heads == 4 || heads == 8)) return GQ_ERR_UNSUPPORTED;
  if (g->nnz == 0) return GQ_OK;  // no edges: no values
  if (codes == nullptr || hdr == nullptr || out == nullptr) return GQ_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(hdr, 16) || !aligned(out, 16)) return GQ_ERR_INVALID_ARG;
  EdgeQuantParams p{};
  p.rowptr = g->rowptr;
  p.codes = const_cast<uint8_t*>(codes);
  p.hdr = const_cast<float*>(hdr);
  p.deq = out;
  p.n_rows = g->n;
  p.n_edges = g->nnz;
  p.err = g->status;
  p.sc = make_sched(g->sched, g->hub_threshold, nullptr, 0);
  switch (heads) {
    case 1: return launch_edge_dequant<1>(p, s);
    case 2: return launch_edge_dequant<2>(p, s);
    case 4: return launch_edge_dequant<4>(p, s);
    default: return launch_edge_dequant<8>(p, s);
  }
}

int gat_edge_bwd(const gq_graph* g, const float* dOut, const float* Hp, const uint8_t* packed, const uint8_t* mask,
                 int bits, const float* alpha, const float* S, const float* D, int heads, int d, float slope,
                 float* dEpre, float* dD, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!(heads == 1 || heads == 2 || heads == 4 || heads == 8)) return GQ_ERR_UNSUPPORTED;
  if (d < 8 || d > 256 || d % heads) return GQ_ERR_UNSUPPORTED;
  const int F = d / heads;
  if (F % 8 || ((F / 8) & (F / 8 - 1))) return GQ_ERR_UNSUPPORTED;  // head width: 8 * power of two
  EdgeBwdParams p{};
  p.rowptr = g->rowptr;
  p.col = g->col;
  p.dOut = dOut;
  p.msg = MsgSrc{Hp, d, packed, bits < 32 ? packed_pitch(d, bits) : 0, bits < 32 ? (int)header_offset(d, bits) : 0,
                 mask, d};
  p.alpha = alpha;
  p.S = S;
  p.D = D;
  p.slope = slope;
  p.dEpre = dEpre;
  p.dD = dD;
  p.n_rows = g->n;
  p.d = d;
  p.lph = F / 8;
  p.light = g->sched.light;
  p.n_light = g->sched.n_light;
  const size_t need = edge_bwd_workspace(g, heads);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !aligned(ws, 256))) return GQ_ERR_WORKSPACE;
  p.sc = make_sched(g->sched, g->hub_threshold, nullptr, 0);
  if (g->sched.n_tasks > 0) {
    const size_t part = ((size_t)g->sched.n_tasks * heads * sizeof(float) + 255) / 256 * 256;
    p.Ppart = static_cast<float*>(ws);
    p.dDpart = reinterpret_cast<float*>(static_cast<char*>(ws) + part);
    p.sc.tickets = reinterpret_cast<int*>(static_cast<char*>(ws) + 2 * part);
    if (g->sched.n_groups > 0) GQ_TRY_CUDA(cudaMemsetAsync(p.sc.tickets, 0, g->sched.n_groups * sizeof(int), s));
  }
#define GQ_EB(B)                                       \
  switch (heads) {                                     \
    case 1: return launch_edge_bwd<B, 1>(p, s);        \
    case 2: return launch_edge_bwd<B, 2>(p, s);        \
    case 4: return launch_edge_bwd<B, 4>(p, s);        \
    default: return launch_edge_bwd<B, 8>(p, s);       \
  }
  switch (bits) {
    case 2: GQ_EB(2)
    case 4: GQ_EB(4)
    case 8: GQ_EB(8)
    default: GQ_EB(32)
  }
#undef GQ_EB
}

// the blocks resident at 85 registers a thread (at most 128 with 8 heads)
int node_bwd_blocks(int heads = 1) { return sm_count() * (heads == 8 ? 2 : 3); }

// [block][2 d] da partials | [n][K] dS of the heavy rows | their task partials and tickets
size_t node_bwd_workspace(const gq_graph* g, int heads, int d) {
  const size_t a = ((size_t)node_bwd_blocks() * 2 * d * sizeof(float) + 255) / 256 * 256;
  const size_t b = ((size_t)g->n * heads * sizeof(float) + 255) / 256 * 256;
  return a + b + sched_ws(g->tr_sched, heads) + 256;
}

int gat_node_bwd(const gq_graph* g, const float* dEpre, const float* dD, const float* dM, const float* Hp,
                 const float* a_src, const float* a_dst, int heads, int d, void* dHp_bf16, int64_t ldb, float* dHp32,
                 float* dS, float* da_src, float* da_dst, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (g == nullptr) return GQ_ERR_INVALID_ARG;
  if (d < 8 || d > 256 || d % 8 || d % heads) return GQ_ERR_UNSUPPORTED;
  if (!(heads == 1 || heads == 2 || heads == 4 || heads == 8)) return GQ_ERR_UNSUPPORTED;
  const int F = d / heads;
  int fshift = 0;
  while ((1 << fshift) < F) ++fshift;
  if ((1 << fshift) != F || F < 8) return GQ_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < node_bwd_workspace(g, heads, d) || !aligned(ws, 256)) return GQ_ERR_WORKSPACE;
  const int blocks = node_bwd_blocks(heads);
  char* wp = static_cast<char*>(ws);
  NodeBwdParams p{};
  p.tr_rowptr = g->tr_rowptr;
  p.tr_perm = g->tr_perm;
  p.dEpre = dEpre;
  p.dD = dD;
  p.dM = dM;
  p.Hp = Hp;
  p.a_src = a_src;
  p.a_dst = a_dst;
  p.dHp = static_cast<__nv_bfloat16*>(dHp_bf16);
  p.ldb = ldb;
  p.dHp32 = dHp32;
  p.dS = dS;
  p.part = reinterpret_cast<float*>(wp);
  wp += ((size_t)node_bwd_blocks() * 2 * d * sizeof(float) + 255) / 256 * 256;
  p.dSh = reinterpret_cast<float*>(wp);
  wp += ((size_t)g->n * heads * sizeof(float) + 255) / 256 * 256;
  p.n_rows = g->n;
  p.d = d;
  p.fshift = fshift;
  p.sc = make_sched(g->tr_sched, g->hub_threshold, wp, heads);
  const size_t smem = sizeof(float) * kGatWarps * 2 * d;
  if (g->tr_sched.n_groups > 0)
    GQ_TRY_CUDA(cudaMemsetAsync(p.sc.tickets, 0, g->tr_sched.n_groups * sizeof(int), s));
#define GQ_NB(KK)                                                                                             \
  if (p.sc.n_tasks > 0) {                                                                                     \
    gat_node_heavy_kernel<KK><<<(unsigned)p.sc.n_tasks, kGatThreads, 0, s>>>(p);                              \
    GQ_TRY(launch_status());                                                                                  \
  }                                                                                                           \
  gat_node_bwd_kernel<KK><<<blocks, kGatThreads, smem, s>>>(p);                                               \
  break;
  switch (heads) {
    case 1: GQ_NB(1)
    case 2: GQ_NB(2)
    case 4: GQ_NB(4)
    default: GQ_NB(8)
  }
#undef GQ_NB
  GQ_TRY(launch_status());
  sum_blocks_kernel<<<(2 * d + 255) / 256, 256, 0, s>>>(p.part, blocks, 2 * d, da_src, da_dst, d);
  return launch_status();
}

}  // namespace gq

extern "C" size_t gq_edge_softmax_workspace_bytes(const gq_graph* g, int heads) {
  if (g == nullptr || heads < 1) return 0;
  return gq::edge_softmax_workspace(g, heads);
}

extern "C" size_t gq_quantize_edge_values_workspace_bytes(const gq_graph* g, int heads) {
  if (g == nullptr || heads < 1) return 0;
  return gq::edge_quant_workspace(g, heads);
}

extern "C" int gq_quantize_edge_values(const gq_graph* g, const float* alpha, int heads, uint64_t seed,
                                       uint8_t* codes, float* hdr, void* ws, size_t ws_bytes, gq_stream stream) {
  return gq::quantize_edge_values(g, alpha, heads, seed, codes, hdr, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int gq_dequant_edge_values(const gq_graph* g, const uint8_t* codes, const float* hdr, int heads,
                                      float* out, gq_stream stream) {
  return gq::dequant_edge_values(g, codes, hdr, heads, out, (cudaStream_t)stream);
}

extern "C" int gq_sddmm_edge_softmax(const gq_graph* g, const float* S, const float* D, int heads, float slope,
                                     float* E_pre, float* alpha, void* ws, size_t ws_bytes, gq_stream stream) {
  return gq::edge_softmax(g, S, D, heads, slope, E_pre, alpha, ws, ws_bytes, (cudaStream_t)stream);
}
