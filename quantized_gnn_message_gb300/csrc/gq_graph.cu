// gq_graph.cu -- graph preparation: CSR validation, degree normalizations
// (Sancus Sec. 2: D~ = D + I, A^ = D~^-1/2 (A+I) D~^-1/2), hub-row lists,
// and the stable transpose (CSC + edge permutation) used by the backward
// aggregation and by the out-edge sums of the GAT backward pass.
//
// The transpose is a stable LSD radix sort of (key = source id, value =
// CSR edge id): after it, each CSC row lists its destinations in
// increasing order, so every later fp32 sum over a CSC row runs in a fixed
// order and results are identical run to run.
#include <string.h>

#include <algorithm>
#include <vector>

#include "gq_common.cuh"

namespace gq {
namespace {

constexpr int kDefaultHub = 256;
constexpr int kDefaultSplit = 4096;
constexpr int kMinHub = 32;
constexpr int kMinSplit = 256;
constexpr int kLightEdges = 256;  // edge budget of one light-row run
constexpr int kScanThreads = 512;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;  // 4096
constexpr int kSortWarps = 8;
constexpr int kSortItems = 16;                        // per lane
constexpr int kSortTile = kSortWarps * 32 * kSortItems;  // 4096
constexpr int kRadix = 256;

// Error bits written by the validation kernels.
constexpr int kErrRowptr = 1;
constexpr int kErrCol = 2;

struct Counters {
  int32_t err;
  int32_t n_hub;
  int32_t tr_n_hub;
  int32_t max_deg;
  int32_t tr_max_deg;
  int32_t pad[3];
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// ---------------------------------------------------------------- scan ---
// Exclusive scan of int32 values within tiles of kScanTile; tile totals go
// to `sums` (if non-null).  In-place safe.
__global__ void __launch_bounds__(kScanThreads) scan_tiles_kernel(const int32_t* in, int32_t* out, int64_t n,
                                                                 int32_t* sums) {
  __shared__ int32_t warp_tot[kScanThreads / 32];
  const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
  int32_t v[kScanItems];
  int32_t run = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    v[i] = (base + i < n) ? in[base + i] : 0;
    const int32_t t = v[i];
    v[i] = run;
    run += t;
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int32_t incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int32_t t = lane < kScanThreads / 32 ? warp_tot[lane] : 0;
    int32_t s = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(FULL, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kScanThreads / 32) warp_tot[lane] = s - t;
    if (lane == kScanThreads / 32 - 1 && sums != nullptr) sums[blockIdx.x] = s;
  }
  __syncthreads();
  const int32_t off = warp_tot[w] + incl - run;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i)
    if (base + i < n) out[base + i] = v[i] + off;
}

__global__ void scan_add_kernel(int32_t* out, int64_t n, const int32_t* sums) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] += sums[i / kScanTile];
}

int64_t scan_scratch_elems(int64_t n) {
  int64_t total = 0;
  while (n > kScanTile) {
    n = (n + kScanTile - 1) / kScanTile;
    total += n + 64;
  }
  return total;
}

// Exclusive scan of n int32 values (in may equal out).
int scan_exclusive(const int32_t* in, int32_t* out, int64_t n, int32_t* scratch, cudaStream_t s) {
  const int64_t tiles = (n + kScanTile - 1) / kScanTile;
  if (tiles <= 1) {
    scan_tiles_kernel<<<1, kScanThreads, 0, s>>>(in, out, n, nullptr);
    return launch_status();
  }
  int32_t* sums = scratch;
  scan_tiles_kernel<<<(unsigned)tiles, kScanThreads, 0, s>>>(in, out, n, sums);
  GQ_TRY(launch_status());
  GQ_TRY(scan_exclusive(sums, sums, tiles, scratch + tiles + 64, s));
  scan_add_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(out, n, sums);
  return launch_status();
}

// -------------------------------------------------------- degree kernels ---
__global__ void rows_kernel(int64_t n, int64_t nnz, const int32_t* __restrict__ rowptr, float* dinv_in, float* inv_in,
                            int32_t* hubs, int64_t max_hubs, int hub_threshold, Counters* cnt) {
  const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= n) return;
  const int32_t a = rowptr[v], b = rowptr[v + 1];
  if (v == 0 && a != 0) atomicOr(&cnt->err, kErrRowptr);
  if (v == n - 1 && (int64_t)b != nnz) atomicOr(&cnt->err, kErrRowptr);
  if (b < a || a < 0 || (int64_t)b > nnz) atomicOr(&cnt->err, kErrRowptr);
  const int32_t deg = b - a;
  dinv_in[v] = deg > 0 ? __double2float_rn(1.0 / sqrt((double)deg)) : 0.0f;
  inv_in[v] = deg > 0 ? __double2float_rn(1.0 / (double)deg) : 0.0f;
  if (deg > hub_threshold) {
    const int i = atomicAdd(&cnt->n_hub, 1);
    if (i < max_hubs) {
      hubs[3 * i] = (int32_t)v;
      hubs[3 * i + 1] = a;
      hubs[3 * i + 2] = deg;
    }
  }
  atomicMax(&cnt->max_deg, deg);
}

__global__ void count_cols_kernel(int64_t nnz, int64_t n, const int32_t* __restrict__ col, int32_t* counts,
                                  Counters* cnt) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= nnz) return;
  const int32_t c = col[e];
  if (c < 0 || (int64_t)c >= n) {
    atomicOr(&cnt->err, kErrCol);
    return;
  }
  atomicAdd(&counts[c], 1);
}

__global__ void out_rows_kernel(int64_t n, const int32_t* __restrict__ tr_rowptr, float* dinv_out, int32_t* hubs,
                                int64_t max_hubs, int hub_threshold, Counters* cnt) {
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= n) return;
  const int32_t a = tr_rowptr[u];
  const int32_t deg = tr_rowptr[u + 1] - a;
  dinv_out[u] = deg > 0 ? __double2float_rn(1.0 / sqrt((double)deg)) : 0.0f;
  if (deg > hub_threshold) {
    const int i = atomicAdd(&cnt->tr_n_hub, 1);
    if (i < max_hubs) {
      hubs[3 * i] = (int32_t)u;
      hubs[3 * i + 1] = a;
      hubs[3 * i + 2] = deg;
    }
  }
  atomicMax(&cnt->tr_max_deg, deg);
}

// edge_row[e] = v for e in row v (warp per row; ranges clamped to [0, nnz)
// so a malformed rowptr cannot write out of bounds).
__global__ void expand_rows_kernel(int64_t n, int64_t nnz, const int32_t* __restrict__ rowptr, int32_t* edge_row) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t v = warp; v < n; v += nwarps) {
    int64_t a = rowptr[v], b = rowptr[v + 1];
    a = a < 0 ? 0 : (a > nnz ? nnz : a);
    b = b < a ? a : (b > nnz ? nnz : b);
    for (int64_t e = a + lane; e < b; e += 32) edge_row[e] = (int32_t)v;
  }
}

// ---------------------------------------------------------- radix sort ---
// Digit of a key; invalid keys (already flagged) sort into bucket 0.
__device__ __forceinline__ int digit_of(int32_t key, int shift) { return ((uint32_t)key >> shift) & (kRadix - 1); }

// Per-tile digit histogram, stored digit-major: hist[d * tiles + tile].
__global__ void __launch_bounds__(kSortWarps * 32) radix_hist_kernel(const int32_t* __restrict__ keys, int64_t nnz,
                                                                    int shift, int32_t* hist, int64_t tiles) {
  __shared__ int32_t h[kRadix];
  for (int i = threadIdx.x; i < kRadix; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kSortTile;
  for (int i = threadIdx.x; i < kSortTile; i += blockDim.x) {
    const int64_t e = base + i;
    if (e < nnz) atomicAdd(&h[digit_of(keys[e], shift)], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kRadix; i += blockDim.x) hist[(int64_t)i * tiles + blockIdx.x] = h[i];
}

// Stable scatter.  Warp w of a tile takes items [w*512, (w+1)*512) of the
// tile in 16 rounds of 32 consecutive items; the rank of an item among the
// tile's items with the same digit counts (a) earlier warps, (b) earlier
// rounds of the same warp and (c) lower lanes of the same round.
// keys_in == nullptr means "keys are col[] and values are the identity".
__global__ void __launch_bounds__(kSortWarps * 32) radix_scatter_kernel(
    const int32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in, int64_t nnz, int shift,
    const int32_t* __restrict__ offsets, int64_t tiles, int32_t* __restrict__ keys_out,
    int32_t* __restrict__ vals_out) {
  __shared__ int32_t wcount[kSortWarps][kRadix];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kSortWarps * kRadix; i += blockDim.x) (&wcount[0][0])[i] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kSortTile + (int64_t)w * (32 * kSortItems);
  int32_t key[kSortItems], val[kSortItems], rank[kSortItems];
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < kSortItems; ++r) {
    const int64_t e = base + r * 32 + lane;
    const bool ok = e < nnz;
    key[r] = ok ? keys_in[e] : 0;
    val[r] = ok ? (vals_in ? vals_in[e] : (int32_t)e) : 0;
    const int dg = ok ? digit_of(key[r], shift) : kRadix;  // kRadix: padding, never matched with real
    const unsigned peers = __match_any_sync(FULL, dg);
    const int before = ok ? wcount[w][dg] : 0;
    __syncwarp();
    if (ok && (peers & lt) == 0) wcount[w][dg] = before + __popc(peers);
    __syncwarp();
    rank[r] = before + __popc(peers & lt);
  }
  __syncthreads();
  // exclusive scan over warps, per digit
  for (int dg = threadIdx.x; dg < kRadix; dg += blockDim.x) {
    int32_t run = 0;
#pragma unroll
    for (int ww = 0; ww < kSortWarps; ++ww) {
      const int32_t t = wcount[ww][dg];
      wcount[ww][dg] = run;
      run += t;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kSortItems; ++r) {
    const int64_t e = base + r * 32 + lane;
    if (e < nnz) {
      const int dg = digit_of(key[r], shift);
      const int64_t pos = (int64_t)offsets[(int64_t)dg * tiles + blockIdx.x] + wcount[w][dg] + rank[r];
      if (keys_out) keys_out[pos] = key[r];
      vals_out[pos] = val[r];
    }
  }
}

__global__ void gather_rows_kernel(int64_t nnz, const int32_t* __restrict__ perm, const int32_t* __restrict__ edge_row,
                                   int32_t* __restrict__ tr_col) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < nnz) tr_col[i] = edge_row[perm[i]];
}

int64_t max_tasks(int64_t nnz) { return nnz / kMinHub + nnz / kMinSplit + 2; }
int64_t max_groups(int64_t nnz) { return nnz / kMinSplit + 1; }
int64_t max_hubs(int64_t nnz) { return nnz / kMinHub + 1; }
// runs end at a budget (each run but the last of a stretch holds more than
// half a budget of edges) or at a heavy row
int64_t max_light(int64_t n, int64_t nnz) {
  const int64_t b = 2 * nnz / kLightEdges + max_hubs(nnz) + 2;
  return b < n + 1 ? b : n + 1;
}

struct StorageLayout {
  size_t tr_rowptr, tr_col, tr_perm, dinv_in, dinv_out, inv_in, tasks, groups, tr_tasks, tr_groups, light, tr_light,
      status, total;
};

StorageLayout storage_layout(int64_t n, int64_t nnz) {
  StorageLayout L;
  size_t o = 0;
  L.tr_rowptr = o; o += align256(sizeof(int32_t) * (n + 1));
  L.tr_col = o;    o += align256(sizeof(int32_t) * (nnz > 0 ? nnz : 1));
  L.tr_perm = o;   o += align256(sizeof(int32_t) * (nnz > 0 ? nnz : 1));
  L.dinv_in = o;   o += align256(sizeof(float) * n);
  L.dinv_out = o;  o += align256(sizeof(float) * n);
  L.inv_in = o;    o += align256(sizeof(float) * n);
  L.tasks = o;     o += align256(sizeof(int32_t) * 4 * max_tasks(nnz));
  L.groups = o;    o += align256(sizeof(int32_t) * 4 * max_groups(nnz));
  L.tr_tasks = o;  o += align256(sizeof(int32_t) * 4 * max_tasks(nnz));
  L.tr_groups = o; o += align256(sizeof(int32_t) * 4 * max_groups(nnz));
  L.light = o;     o += align256(sizeof(int32_t) * 2 * max_light(n, nnz));
  L.tr_light = o;  o += align256(sizeof(int32_t) * 2 * max_light(n, nnz));
  L.status = o;    o += align256(sizeof(int32_t));
  L.total = o;
  return L;
}

struct WsLayout {
  size_t counters, counts, keys_a, keys_b, vals_a, vals_b, hist, scan, hubs, tr_hubs, total;
  int64_t tiles;
};

WsLayout ws_layout(int64_t n, int64_t nnz) {
  WsLayout L;
  const int64_t m = nnz > 0 ? nnz : 1;
  L.tiles = (m + kSortTile - 1) / kSortTile;
  const int64_t hist_elems = L.tiles * kRadix;
  const int64_t scan_n = (n + 1) > hist_elems ? (n + 1) : hist_elems;
  size_t o = 0;
  L.counters = o; o += align256(sizeof(Counters));
  L.counts = o;   o += align256(sizeof(int32_t) * (n + 1));
  L.keys_a = o;   o += align256(sizeof(int32_t) * m);
  L.keys_b = o;   o += align256(sizeof(int32_t) * m);
  L.vals_a = o;   o += align256(sizeof(int32_t) * m);
  L.vals_b = o;   o += align256(sizeof(int32_t) * m);  // also edge_row at the end
  L.hist = o;     o += align256(sizeof(int32_t) * hist_elems);
  L.scan = o;     o += align256(sizeof(int32_t) * (scan_scratch_elems(scan_n) + 64));
  L.hubs = o;     o += align256(sizeof(int32_t) * 3 * max_hubs(nnz));
  L.tr_hubs = o;  o += align256(sizeof(int32_t) * 3 * max_hubs(nnz));
  L.total = o;
  return L;
}

unsigned blocks_for(int64_t n, int t) { return (unsigned)((n + t - 1) / t); }

// Runs of consecutive light rows (degree <= threshold) with at most
// kLightEdges edges each (a run holds at least one row); heavy rows end a
// run and belong to none.
int build_light(const std::vector<int32_t>& ptr, int64_t n, int thr, int32_t* d_light, gq_sched* out,
                std::vector<int32_t>& runs, int64_t cap, cudaStream_t s) {
  runs.clear();
  int64_t start = -1, edges = 0;
  for (int64_t r = 0; r < n; ++r) {
    const int64_t deg = (int64_t)ptr[r + 1] - ptr[r];
    if (deg > thr) {
      if (start >= 0) runs.insert(runs.end(), {(int32_t)start, (int32_t)r});
      start = -1;
      edges = 0;
      continue;
    }
    if (start >= 0 && edges + deg > kLightEdges) {
      runs.insert(runs.end(), {(int32_t)start, (int32_t)r});
      start = -1;
      edges = 0;
    }
    if (start < 0) start = r;
    edges += deg;
  }
  if (start >= 0) runs.insert(runs.end(), {(int32_t)start, (int32_t)n});
  if ((int64_t)(runs.size() / 2) > cap) return GQ_ERR_BAD_GRAPH;
  out->light = d_light;
  out->n_light = (int64_t)(runs.size() / 2);
  if (!runs.empty())
    GQ_TRY_CUDA(cudaMemcpyAsync(d_light, runs.data(), runs.size() * 4, cudaMemcpyHostToDevice, s));
  return GQ_OK;
}

// Cut the heavy rows {row, e_begin, deg} into block tasks, heaviest first.
int build_sched(const std::vector<int32_t>& hubs, int split, int32_t* d_tasks, int32_t* d_groups, gq_sched* out,
                std::vector<int32_t>& tasks, std::vector<int32_t>& groups, cudaStream_t s) {
  const size_t nh = hubs.size() / 3;
  std::vector<size_t> order(nh);
  for (size_t i = 0; i < nh; ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](size_t x, size_t y) {
    if (hubs[3 * x + 2] != hubs[3 * y + 2]) return hubs[3 * x + 2] > hubs[3 * y + 2];
    return hubs[3 * x] < hubs[3 * y];
  });
  tasks.clear();
  groups.clear();
  int32_t slots = 0;
  for (size_t k = 0; k < nh; ++k) {
    const int32_t row = hubs[3 * order[k]], e0 = hubs[3 * order[k] + 1], deg = hubs[3 * order[k] + 2];
    const int32_t nch = (deg + split - 1) / split;
    int32_t grp = -1;
    if (nch > 1) {
      grp = (int32_t)(groups.size() / 4);
      groups.insert(groups.end(), {row, (int32_t)(tasks.size() / 4), nch, slots});
      slots += nch;
    }
    for (int32_t c = 0; c < nch; ++c) {
      const int32_t b = e0 + c * split;
      const int32_t e = (c == nch - 1) ? e0 + deg : b + split;
      tasks.insert(tasks.end(), {row, b, e, grp});
    }
  }
  out->tasks = d_tasks;
  out->groups = d_groups;
  out->n_tasks = (int64_t)(tasks.size() / 4);
  out->n_groups = (int64_t)(groups.size() / 4);
  out->n_slots = slots;
  if (!tasks.empty())
    GQ_TRY_CUDA(cudaMemcpyAsync(d_tasks, tasks.data(), tasks.size() * 4, cudaMemcpyHostToDevice, s));
  if (!groups.empty())
    GQ_TRY_CUDA(cudaMemcpyAsync(d_groups, groups.data(), groups.size() * 4, cudaMemcpyHostToDevice, s));
  return GQ_OK;
}

}  // namespace
}  // namespace gq

extern "C" size_t gq_graph_storage_bytes(int64_t n, int64_t nnz) {
  if (n < 1 || nnz < 0) return 0;
  return gq::storage_layout(n, nnz).total;
}

extern "C" size_t gq_graph_prepare_workspace_bytes(int64_t n, int64_t nnz) {
  if (n < 1 || nnz < 0) return 0;
  return gq::ws_layout(n, nnz).total;
}

extern "C" int gq_graph_prepare(int64_t n, int64_t nnz, const int32_t* rowptr, const int32_t* col, int hub_threshold,
                                int split_edges, void* storage, size_t storage_bytes, void* ws, size_t ws_bytes,
                                gq_graph* g, gq_stream stream) {
  using namespace gq;
  if (g == nullptr || rowptr == nullptr || storage == nullptr || ws == nullptr) return GQ_ERR_INVALID_ARG;
  if (n < 1 || nnz < 0 || nnz >= (int64_t)0x7fffffff || n >= (int64_t)0x7fffffff) return GQ_ERR_INVALID_ARG;
  if (nnz > 0 && col == nullptr) return GQ_ERR_INVALID_ARG;
  if (!aligned(storage, 256) || !aligned(ws, 256)) return GQ_ERR_INVALID_ARG;
  const StorageLayout SL = storage_layout(n, nnz);
  const WsLayout WL = ws_layout(n, nnz);
  if (storage_bytes < SL.total || ws_bytes < WL.total) return GQ_ERR_WORKSPACE;
  if (hub_threshold <= 0) hub_threshold = kDefaultHub;
  if (split_edges <= 0) split_edges = kDefaultSplit;
  if (hub_threshold < kMinHub || split_edges < kMinSplit) return GQ_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;

  char* st = static_cast<char*>(storage);
  char* wb = static_cast<char*>(ws);
  gq_graph G;
  memset(&G, 0, sizeof(G));
  G.n = n;
  G.nnz = nnz;
  G.rowptr = rowptr;
  G.col = col;
  G.tr_rowptr = reinterpret_cast<int32_t*>(st + SL.tr_rowptr);
  G.tr_col = reinterpret_cast<int32_t*>(st + SL.tr_col);
  G.tr_perm = reinterpret_cast<int32_t*>(st + SL.tr_perm);
  G.dinv_in = reinterpret_cast<float*>(st + SL.dinv_in);
  G.dinv_out = reinterpret_cast<float*>(st + SL.dinv_out);
  G.inv_in = reinterpret_cast<float*>(st + SL.inv_in);
  G.hub_threshold = hub_threshold;
  G.split_edges = split_edges;
  G.status = reinterpret_cast<int32_t*>(st + SL.status);
  GQ_TRY_CUDA(cudaMemsetAsync(G.status, 0, sizeof(int32_t), s));
  int32_t* hubs = reinterpret_cast<int32_t*>(wb + WL.hubs);
  int32_t* tr_hubs = reinterpret_cast<int32_t*>(wb + WL.tr_hubs);

  Counters* cnt = reinterpret_cast<Counters*>(wb + WL.counters);
  int32_t* counts = reinterpret_cast<int32_t*>(wb + WL.counts);
  int32_t* keys_a = reinterpret_cast<int32_t*>(wb + WL.keys_a);
  int32_t* keys_b = reinterpret_cast<int32_t*>(wb + WL.keys_b);
  int32_t* vals_a = reinterpret_cast<int32_t*>(wb + WL.vals_a);
  int32_t* vals_b = reinterpret_cast<int32_t*>(wb + WL.vals_b);
  int32_t* hist = reinterpret_cast<int32_t*>(wb + WL.hist);
  int32_t* scan = reinterpret_cast<int32_t*>(wb + WL.scan);

  GQ_TRY_CUDA(cudaMemsetAsync(cnt, 0, sizeof(Counters), s));
  GQ_TRY_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * (n + 1), s));
  rows_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, nnz, rowptr, G.dinv_in, G.inv_in, hubs, max_hubs(nnz),
                                                  hub_threshold, cnt);
  GQ_TRY(launch_status());
  if (nnz > 0) {
    count_cols_kernel<<<blocks_for(nnz, 256), 256, 0, s>>>(nnz, n, col, counts, cnt);
    GQ_TRY(launch_status());
  }
  GQ_TRY(scan_exclusive(counts, G.tr_rowptr, n + 1, scan, s));
  out_rows_kernel<<<blocks_for(n, 256), 256, 0, s>>>(n, G.tr_rowptr, G.dinv_out, tr_hubs, max_hubs(nnz),
                                                      hub_threshold, cnt);
  GQ_TRY(launch_status());

  if (nnz > 0) {
    // stable LSD radix sort of (col[e], e) by col
    int key_bits = 1;
    while (key_bits < 31 && ((int64_t)1 << key_bits) < n) ++key_bits;
    const int passes = (key_bits + 7) / 8;
    const int64_t tiles = WL.tiles;
    const int32_t* kin = col;
    const int32_t* vin = nullptr;
    for (int p = 0; p < passes; ++p) {
      const int shift = 8 * p;
      const bool last = (p == passes - 1);
      int32_t* kout = (p % 2 == 0) ? keys_a : keys_b;
      int32_t* vout = last ? G.tr_perm : ((p % 2 == 0) ? vals_a : vals_b);
      radix_hist_kernel<<<(unsigned)tiles, kSortWarps * 32, 0, s>>>(kin, nnz, shift, hist, tiles);
      GQ_TRY(launch_status());
      GQ_TRY(scan_exclusive(hist, hist, tiles * kRadix, scan, s));
      radix_scatter_kernel<<<(unsigned)tiles, kSortWarps * 32, 0, s>>>(kin, vin, nnz, shift, hist, tiles,
                                                                        last ? nullptr : kout, vout);
      GQ_TRY(launch_status());
      kin = kout;
      vin = vout;
    }
    // destination of each CSC entry (keys_b is free once the sort is done)
    int32_t* edge_row = keys_b;
    expand_rows_kernel<<<gq::sm_count() * 8, 256, 0, s>>>(n, nnz, rowptr, edge_row);
    GQ_TRY(launch_status());
    gather_rows_kernel<<<blocks_for(nnz, 256), 256, 0, s>>>(nnz, G.tr_perm, edge_row, G.tr_col);
    GQ_TRY(launch_status());
  }

  Counters h;
  GQ_TRY_CUDA(cudaMemcpyAsync(&h, cnt, sizeof(Counters), cudaMemcpyDeviceToHost, s));
  GQ_TRY_CUDA(cudaStreamSynchronize(s));
  if (h.err != 0) return GQ_ERR_BAD_GRAPH;
  if (h.n_hub > max_hubs(nnz) || h.tr_n_hub > max_hubs(nnz)) return GQ_ERR_BAD_GRAPH;
  std::vector<int32_t> hv((size_t)h.n_hub * 3), thv((size_t)h.tr_n_hub * 3), tasks, groups, tr_tasks, tr_groups;
  if (h.n_hub > 0) GQ_TRY_CUDA(cudaMemcpyAsync(hv.data(), hubs, hv.size() * 4, cudaMemcpyDeviceToHost, s));
  if (h.tr_n_hub > 0) GQ_TRY_CUDA(cudaMemcpyAsync(thv.data(), tr_hubs, thv.size() * 4, cudaMemcpyDeviceToHost, s));
  GQ_TRY_CUDA(cudaStreamSynchronize(s));
  GQ_TRY(build_sched(hv, split_edges, reinterpret_cast<int32_t*>(st + SL.tasks),
                     reinterpret_cast<int32_t*>(st + SL.groups), &G.sched, tasks, groups, s));
  GQ_TRY(build_sched(thv, split_edges, reinterpret_cast<int32_t*>(st + SL.tr_tasks),
                     reinterpret_cast<int32_t*>(st + SL.tr_groups), &G.tr_sched, tr_tasks, tr_groups, s));
  // light-row runs of both directions (row pointers read back once)
  std::vector<int32_t> hptr((size_t)n + 1), htr((size_t)n + 1), runs, tr_runs;
  GQ_TRY_CUDA(cudaMemcpyAsync(hptr.data(), rowptr, (n + 1) * 4, cudaMemcpyDeviceToHost, s));
  GQ_TRY_CUDA(cudaMemcpyAsync(htr.data(), G.tr_rowptr, (n + 1) * 4, cudaMemcpyDeviceToHost, s));
  GQ_TRY_CUDA(cudaStreamSynchronize(s));
  GQ_TRY(build_light(hptr, n, hub_threshold, reinterpret_cast<int32_t*>(st + SL.light), &G.sched, runs,
                     max_light(n, nnz), s));
  GQ_TRY(build_light(htr, n, hub_threshold, reinterpret_cast<int32_t*>(st + SL.tr_light), &G.tr_sched, tr_runs,
                     max_light(n, nnz), s));
  GQ_TRY_CUDA(cudaStreamSynchronize(s));  // host task vectors must outlive the copies
  G.max_deg = h.max_deg;
  G.tr_max_deg = h.tr_max_deg;
  *g = G;
  return GQ_OK;
}
