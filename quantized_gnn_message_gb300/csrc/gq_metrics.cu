// gq_metrics.cu -- message-level quantization metrics.
//
// message_variance_weights (AdaQP Sec. 4.2, the weight beta_k of message k
// in Problem 11):
//   beta_k = sum_{v in N_T(k)} a_{k,v}^2 * D * (max h_k - min h_k)^2 / 6,
// where N_T(k) is every destination v of an edge k -> v (one GPU holds all
// of them) and a_{k,v} the aggregation coefficient; the variance of the
// aggregated error of message k quantized at b bits is beta_k / (2^b-1)^2.
// One warp per node: a min/max reduction over the row and a sum of a^2 over
// the node's out-edges (its row of the transposed CSR); a node with more
// out-edges than the graph's hub threshold is summed by blocks, one per
// task of the transposed heavy-row schedule, whose partials are added in
// task order.  Every sum has a fixed order.
//
// quant_error (Tango Sec. 3.2, Eq. 4):
//   Error_X = (1/N) sum_i |X_i - Xq_i| / (|X_i| + |Xq_i| + eps)
// over the N = n*d elements, Xq the de-quantized value (fmaf(q, S, Z)) of a
// quantized row; a row with mask 0 is not quantized and adds nothing.  The
// absolute values in the denominator read the page's X_i + Xq_i for an
// asymmetric quantizer (the page's values share one sign).  A warp per row
// sums its terms in fp32, each lane keeps an fp64 total; block partials are
// added in block order by a second kernel.
//
// assign_bits (AdaQP Sec. 4.2, Problems 10-12 on one device): each row's
// width in {2, 4, 8} minimizing lam * beta / (2^b - 1)^2 + (1 - lam) * gamma
// * d * b, in fp64 in a fixed operation order (ties to the fewer bits).
#include "gq_common.cuh"
#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr int kMetricThreads = 256;
constexpr int kMetricWarps = kMetricThreads / 32;

struct BetaParams {
  int64_t n;
  const int32_t* tr_rowptr;
  const int32_t* tr_col;
  const float* dinv_in;
  const float* dinv_out;
  const float* inv_in;
  int coef;
  const float* X;
  int64_t ldx;
  int d;
  float* beta;
  const int32_t* tasks;   // heavy rows of the transposed CSR (gq_sched)
  const int32_t* groups;
  int64_t n_tasks;
  int hub_threshold;
  float* part;            // [task] partial sums of a^2
};

// a_{k,v} of the edge k -> v (v = a destination of node k)
__device__ __forceinline__ float beta_coef(const BetaParams& p, float sk, int32_t v) {
  return p.coef == GQ_COEF_GCN ? sk * __ldg(p.dinv_in + v) : (p.coef == GQ_COEF_SAGE ? __ldg(p.inv_in + v) : 1.0f);
}

// (lane-strided) sum of a^2 over the edges [a, b) of node k's row
__device__ __forceinline__ float beta_s2(const BetaParams& p, float sk, int64_t a, int64_t b, int first, int stride) {
  float s2 = 0.0f;
  for (int64_t e = a + first; e < b; e += stride) {
    const float c = beta_coef(p, sk, __ldg(p.tr_col + e));
    s2 = __fmaf_rn(c, c, s2);
  }
  return s2;
}

// beta[k] from the warp's (lane 0) s2, after a min/max reduction over X[k]
__device__ __forceinline__ void beta_finish(const BetaParams& p, int64_t k, float s2) {
  const int lane = threadIdx.x & 31;
  const float* x = p.X + k * p.ldx;
  float mn = __int_as_float(0x7f800000), mx = -mn;  // +inf, -inf
  for (int j = lane; j < p.d; j += 32) {
    const float v = __ldg(x + j);
    mn = fminf(mn, v);
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(FULL, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
  }
  if (lane == 0) {
    const float r = mx - mn;
    p.beta[k] = s2 * (float)p.d * r * r * (1.0f / 6.0f);
  }
}

// Blocks [0, n_tasks): one heavy-row task each, its partial sum of a^2 to
// part[task].  Other blocks: one warp per light node (out-degree at most
// hub_threshold), beta written directly.
__global__ void __launch_bounds__(kMetricThreads) beta_kernel(const BetaParams p) {
  __shared__ float red[kMetricWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if ((int64_t)blockIdx.x < p.n_tasks) {
    const int4 task = __ldg(reinterpret_cast<const int4*>(p.tasks) + blockIdx.x);
    const float sk = p.coef == GQ_COEF_GCN ? __ldg(p.dinv_out + task.x) : 1.0f;
    float s2 = beta_s2(p, sk, task.y, task.z, threadIdx.x, blockDim.x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(FULL, s2, o);
    if (lane == 0) red[w] = s2;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int i = 0; i < kMetricWarps; ++i) t += red[i];
      p.part[blockIdx.x] = t;
    }
    return;
  }
  const int64_t gw = ((int64_t)blockIdx.x - p.n_tasks) * kMetricWarps + w;
  const int64_t nw = ((int64_t)gridDim.x - p.n_tasks) * kMetricWarps;
  for (int64_t k = gw; k < p.n; k += nw) {
    const int64_t a = __ldg(p.tr_rowptr + k), b = __ldg(p.tr_rowptr + k + 1);
    if (b - a > p.hub_threshold) continue;  // a heavy row: its tasks
    const float sk = p.coef == GQ_COEF_GCN ? __ldg(p.dinv_out + k) : 1.0f;
    float s2 = beta_s2(p, sk, a, b, lane, 32);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(FULL, s2, o);
    beta_finish(p, k, s2);
  }
}

// One warp per heavy-row task: the first task of each row adds the row's
// task partials in task order and writes beta.
__global__ void __launch_bounds__(kMetricThreads) beta_heavy_kernel(const BetaParams p) {
  const int64_t t = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  if (t >= p.n_tasks) return;
  const int4 task = __ldg(reinterpret_cast<const int4*>(p.tasks) + t);
  float s2;
  if (task.w < 0) {
    s2 = __ldcg(p.part + t);
  } else {
    const int4 grp = __ldg(reinterpret_cast<const int4*>(p.groups) + task.w);
    if (grp.y != t) return;  // not the group's first task
    s2 = 0.0f;
    for (int i = 0; i < grp.z; ++i) s2 += __ldcg(p.part + grp.y + i);
  }
  beta_finish(p, task.x, s2);
}

__global__ void __launch_bounds__(kMetricThreads) quant_error_kernel(const float* __restrict__ X, int64_t n, int d,
                                                                    int64_t ldx, const uint8_t* __restrict__ packed,
                                                                    int64_t pitch, int64_t hoff,
                                                                    const uint8_t* __restrict__ mask, int bits,
                                                                    float eps, double* __restrict__ part) {
  __shared__ double red[kMetricWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (gridDim.x * (int64_t)blockDim.x) >> 5;
  const uint32_t cmask = (1u << bits) - 1u;
  double tot = 0.0;
  for (int64_t r = gw; r < n; r += nw) {
    if (mask != nullptr && __ldg(mask + r) == 0) continue;
    const uint8_t* row = packed + r * pitch;
    const float2 h = __ldg(reinterpret_cast<const float2*>(row + hoff));  // {S, Z}
    const float* x = X + r * ldx;
    float s = 0.0f;
    for (int j = lane; j < d; j += 32) {
      const int bit = j * bits;
      const uint32_t q = ((uint32_t)__ldg(row + (bit >> 3)) >> (bit & 7)) & cmask;
      const float xq = __fmaf_rn((float)q, h.x, h.y);
      const float xv = __ldg(x + j);
      s += fabsf(xv - xq) / (fabsf(xv) + fabsf(xq) + eps);
    }
    tot += (double)s;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
  if (lane == 0) red[w] = tot;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < kMetricWarps; ++i) t += red[i];
    part[blockIdx.x] = t;
  }
}

__global__ void sum_parts_kernel(const double* __restrict__ part, int blocks, double inv_n, double* __restrict__ out) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < blocks; ++i) t += part[i];
    *out = t * inv_n;
  }
}

int error_blocks() { return sm_count() * 4; }

// Error_X of the quantizer at 2, 4 and 8 bits in one pass over X, and
// Tango's rule on top of it (Sec. 3.2, Eq. 4: the fewest bits whose error
// stays below the threshold).  A warp per row: the row's min and max once,
// then, per element, the noise u once and, for each width, the code the
// quantizer writes (the same fp32 operations: S = (max - min) / (2^b - 1),
// t = (x - Z) * (1/S), q = min(floor(t + u), 2^b - 1), Xq = fmaf(q, S, Z))
// and the term |x - Xq| / (|x| + |Xq| + eps).  Sums as in quant_error_kernel:
// fp32 per lane and row, fp64 across rows, block partials in block order.
__global__ void __launch_bounds__(kMetricThreads) error3_kernel(const float* __restrict__ X, int64_t n, int d,
                                                               int64_t ldx, const uint8_t* __restrict__ mask,
                                                               uint32_t seed_key, float eps,
                                                               double* __restrict__ part) {
  __shared__ double red[3][kMetricWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (gridDim.x * (int64_t)blockDim.x) >> 5;
  double tot[3] = {0.0, 0.0, 0.0};
  for (int64_t r = gw; r < n; r += nw) {
    if (mask != nullptr && __ldg(mask + r) == 0) continue;
    const float* x = X + r * ldx;
    float mn = __ldg(x), mx = mn;
    for (int j = lane; j < d; j += 32) {
      const float v = __ldg(x + j);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(FULL, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
    }
    float S[3], inv[3];
    bool constant[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      S[i] = __fdiv_rn(__fsub_rn(mx, mn), (float)((1u << (2 << i)) - 1u));
      constant[i] = !(S[i] >= 1.17549435e-38f);
      inv[i] = constant[i] ? 0.0f : __frcp_rn(S[i]);
    }
    const uint32_t kr = row_key(seed_key, (uint32_t)r);
    float s[3] = {0.0f, 0.0f, 0.0f};
    for (int j = lane; j < d; j += 32) {
      const float v = __ldg(x + j);
      const float u = noise_u(kr, (uint32_t)j);
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        uint32_t q = 0;
        if (!constant[i]) {
          const float t = __fmul_rn(__fsub_rn(v, mn), inv[i]);
          q = __float_as_uint(__fadd_rd(__fadd_rn(t, u), 8388608.0f)) - 0x4B000000u;
          q = min(q, (1u << (2 << i)) - 1u);
        }
        const float xq = __fmaf_rn((float)q, S[i], mn);
        s[i] += fabsf(v - xq) / (fabsf(v) + fabsf(xq) + eps);
      }
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) tot[i] += (double)s[i];
  }
#pragma unroll
  for (int i = 0; i < 3; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot[i] += __shfl_xor_sync(FULL, tot[i], o);
    if (lane == 0) red[i][w] = tot[i];
  }
  __syncthreads();
  if (threadIdx.x < 3) {
    double t = 0.0;
    for (int k = 0; k < kMetricWarps; ++k) t += red[threadIdx.x][k];
    part[(int64_t)threadIdx.x * gridDim.x + blockIdx.x] = t;
  }
}

// err3[i] = the block partials of width 2 << i, in block order, / (n d);
// *bits = the fewest of 2, 4, 8 whose error is below the threshold, else 8.
__global__ void error3_finish_kernel(const double* __restrict__ part, int blocks, double inv_n, double threshold,
                                     double* __restrict__ err3, int32_t* __restrict__ bits) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  int pick = 8;
  for (int i = 2; i >= 0; --i) {
    double t = 0.0;
    for (int k = 0; k < blocks; ++k) t += part[(int64_t)i * blocks + k];
    t *= inv_n;
    if (err3 != nullptr) err3[i] = t;
    if (t < threshold) pick = 2 << i;
  }
  *bits = pick;
}

// AdaQP Sec. 4.2, Problems 10-12 on one device: one device pair, so the
// time objective is theta + gamma * sum_k d b_k with theta constant, and the
// weighted sum with the variance objective separates per message.  Each row
// takes the width b in {2, 4, 8} minimizing
//   lam * (beta / (L * L)) + tw * (d * b),   L = 2^b - 1, tw = (1 - lam) * gamma
// in fp64 with each operation rounded to nearest in that order (ties to the
// fewer bits); rows with mask 0 stay full precision (width 0).
__global__ void assign_bits_kernel(const float* __restrict__ beta, const uint8_t* __restrict__ mask, int64_t n,
                                   double d, double lam, double tw, uint8_t* __restrict__ rbits) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride) {
    if (mask != nullptr && __ldg(mask + k) == 0) {
      rbits[k] = 0;
      continue;
    }
    const double bk = (double)__ldg(beta + k);
    int best = 2;
    double best_c = 0.0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int b = 2 << i;
      const double L = (double)((1 << b) - 1);
      const double c = __dadd_rn(__dmul_rn(lam, __ddiv_rn(bk, __dmul_rn(L, L))), __dmul_rn(tw, __dmul_rn(d, (double)b)));
      if (i == 0 || c < best_c) {
        best_c = c;
        best = b;
      }
    }
    rbits[k] = (uint8_t)best;
  }
}

}  // namespace
}  // namespace gq

extern "C" size_t gq_message_variance_weights_workspace_bytes(const gq_graph* g) {
  if (g == nullptr) return 0;
  return ((size_t)g->tr_sched.n_tasks * sizeof(float) + 255) / 256 * 256;
}

extern "C" int gq_message_variance_weights(const gq_graph* g, int coef, const float* X, int64_t ldx, int d,
                                           float* beta, void* ws, size_t ws_bytes, gq_stream stream) {
  using namespace gq;
  if (g == nullptr || X == nullptr || beta == nullptr || d < 1 || ldx < d) return GQ_ERR_INVALID_ARG;
  if (!(coef == GQ_COEF_GCN || coef == GQ_COEF_SAGE || coef == GQ_COEF_ONE)) return GQ_ERR_INVALID_ARG;
  const gq_sched& sc = g->tr_sched;
  if (sc.n_tasks > 0 && (ws == nullptr || ws_bytes < (size_t)sc.n_tasks * sizeof(float) || !aligned(ws, 4)))
    return GQ_ERR_WORKSPACE;
  BetaParams p{g->n, g->tr_rowptr, g->tr_col, g->dinv_in, g->dinv_out, g->inv_in, coef, X, ldx, d, beta,
               sc.tasks, sc.groups, sc.n_tasks, g->hub_threshold, static_cast<float*>(ws)};
  int64_t light = (g->n + kMetricWarps - 1) / kMetricWarps;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (light > cap) light = cap;
  if (light < 1) light = 1;
  const int64_t grid = sc.n_tasks + light;
  if (grid > 0x7fffffff) return GQ_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  beta_kernel<<<(unsigned)grid, kMetricThreads, 0, s>>>(p);
  GQ_TRY(launch_status());
  if (sc.n_tasks > 0) {
    beta_heavy_kernel<<<(unsigned)((sc.n_tasks + kMetricWarps - 1) / kMetricWarps), kMetricThreads, 0, s>>>(p);
    GQ_TRY(launch_status());
  }
  return GQ_OK;
}

extern "C" size_t gq_quant_error_workspace_bytes(void) { return (size_t)gq::error_blocks() * sizeof(double); }

extern "C" int gq_quant_error(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* packed,
                              const uint8_t* mask, int bits, float eps, double* err, void* ws, size_t ws_bytes,
                              gq_stream stream) {
  using namespace gq;
  if (err == nullptr || n < 0 || d < 1 || ldx < d || !valid_bits(bits) || !(eps > 0.0f)) return GQ_ERR_INVALID_ARG;
  if (n == 0) {  // an empty tensor: no elements, no error
    GQ_TRY_CUDA(cudaMemsetAsync(err, 0, sizeof(double), (cudaStream_t)stream));
    return GQ_OK;
  }
  if (X == nullptr || packed == nullptr || !aligned(packed, 16)) return GQ_ERR_INVALID_ARG;
  const int blocks = error_blocks();
  if (ws == nullptr || ws_bytes < (size_t)blocks * sizeof(double) || !aligned(ws, 8)) return GQ_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  double* part = static_cast<double*>(ws);
  quant_error_kernel<<<blocks, kMetricThreads, 0, s>>>(X, n, d, ldx, packed, packed_pitch(d, bits),
                                                       header_offset(d, bits), mask, bits, eps, part);
  GQ_TRY(launch_status());
  const double inv_n = n > 0 ? 1.0 / ((double)n * (double)d) : 0.0;
  sum_parts_kernel<<<1, 32, 0, s>>>(part, blocks, inv_n, err);
  return launch_status();
}

extern "C" int gq_assign_bits(const float* beta, const uint8_t* mask, int64_t n, int d, double lam, double gamma,
                              uint8_t* rbits, gq_stream stream) {
  using namespace gq;
  if (n < 0 || d < 1 || !(lam >= 0.0 && lam <= 1.0) || !(gamma >= 0.0) || gamma > 1e300) return GQ_ERR_INVALID_ARG;
  if (n == 0) return GQ_OK;
  if (beta == nullptr || rbits == nullptr) return GQ_ERR_INVALID_ARG;
  const double tw = (1.0 - lam) * gamma;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  assign_bits_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(beta, mask, n, (double)d, lam, tw, rbits);
  return launch_status();
}

extern "C" size_t gq_bits_for_error_workspace_bytes(void) {
  return (size_t)3 * gq::error_blocks() * sizeof(double);
}

extern "C" int gq_bits_for_error(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* mask, uint64_t seed,
                                 double threshold, float eps, double* err3, int32_t* bits, void* ws, size_t ws_bytes,
                                 gq_stream stream) {
  using namespace gq;
  if (bits == nullptr || n < 0 || d < 1 || ldx < d || !(eps > 0.0f) || !(threshold > 0.0) || threshold > 1e300)
    return GQ_ERR_INVALID_ARG;
  if (n > 0 && X == nullptr) return GQ_ERR_INVALID_ARG;
  const int blocks = error_blocks();
  if (ws == nullptr || ws_bytes < (size_t)3 * blocks * sizeof(double) || !aligned(ws, 8)) return GQ_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  double* part = static_cast<double*>(ws);
  error3_kernel<<<blocks, kMetricThreads, 0, s>>>(X, n, d, ldx, mask, seed_key_host(seed), eps, part);
  GQ_TRY(launch_status());
  const double inv_n = n > 0 ? 1.0 / ((double)n * (double)d) : 0.0;
  error3_finish_kernel<<<1, 32, 0, s>>>(part, blocks, inv_n, threshold, err3, bits);
  return launch_status();
}
