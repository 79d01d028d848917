// gq_quant.cu -- per-row stochastic integer quantization with bit-packing,
// and the matching de-quantization (AdaQP Sec. 2.3, Eqn 4 and Eqn 5).
//
// A group of G lanes per message row (G = 32 for d > 128, fewer for
// narrower rows, so a warp quantizes 32 / G rows at once).  Lane l of the
// group owns the 8-column chunks c = l + G i of the row, so each lane packs
// its 8 codes into one b-byte word and the group writes the payload with
// contiguous 2/4/8-byte stores.  Row min/max are shuffle reductions within
// the group; the noise is a counter hash of (seed, row, column), so the
// packed bytes do not depend on the launch shape.
#include "gq_common.cuh"
#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr int kQuantThreads = 256;

// Load the 8 values of chunk c (columns 8c .. 8c+7) of row x; columns >= d
// read as `fill`.
__device__ __forceinline__ void load_chunk(const float* __restrict__ x, int c, int d, bool vec,
                                           float fill, float (&v)[8]) {
  const int j0 = c * 8;
  if (vec && j0 + 8 <= d) {
    const float4 a = ldg_f4(x + j0);
    const float4 b = ldg_f4(x + j0 + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = (j0 + i < d) ? __ldg(x + j0 + i) : fill;
  }
}

// Codes of one chunk, packed LSB-first into BITS bytes.
template <int BITS>
__device__ __forceinline__ uint64_t quantize_chunk(const float (&v)[8], int j0, int d, float mn,
                                                   float inv, bool constant, uint32_t kr) {
  constexpr uint32_t L = (1u << BITS) - 1u;
  uint64_t word = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t q = 0;
    if (!constant && j0 + i < d) {
      const float t = __fmul_rn(__fsub_rn(v[i], mn), inv);
      const float s = __fadd_rn(t, noise_u(kr, (uint32_t)(j0 + i)));
      // floor(s) for s in [0, 2^23): add 2^23 rounding down, read the mantissa
      q = __float_as_uint(__fadd_rd(s, 8388608.0f)) - 0x4B000000u;
      q = min(q, L);
    }
    word |= (uint64_t)q << (i * BITS);
  }
  return word;
}

template <int BITS>
__device__ __forceinline__ void store_word(uint8_t* p, uint64_t w) {
  if (BITS == 8) {
    *reinterpret_cast<uint2*>(p) = make_uint2((uint32_t)w, (uint32_t)(w >> 32));
  } else if (BITS == 4) {
    *reinterpret_cast<uint32_t*>(p) = (uint32_t)w;
  } else {
    *reinterpret_cast<uint16_t*>(p) = (uint16_t)w;
  }
}

// A row is the job of a group of G lanes (G <= 32, a power of two); a warp
// takes 32 / G consecutive rows per iteration.  CPL > 0: the row stays in
// registers (d <= 8 G CPL).  CPL == 0 (G = 32): two passes over global
// memory (the second hits L1/L2), any d.
// Mixed bit-widths (MIX): `mask` holds each row's bit-width
// and the kernel quantizes the rows whose width is BITS, row r at byte
// roff[r] of `packed`.
template <int BITS, int CPL, int G, bool MIX>
__global__ void __launch_bounds__(kQuantThreads) quantize_pack_kernel(
    const float* __restrict__ X, int64_t n, int d, int64_t ldx, const uint8_t* __restrict__ mask,
    uint32_t seed_key, uint8_t* __restrict__ packed, int64_t pitch, int hoff, bool vec,
    const int64_t* __restrict__ roff) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr int NGR = 32 / G;
  const int lane = threadIdx.x & 31;
  const int gl = lane % G;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nchunks = (d + 7) >> 3;
  const int p8 = nchunks * BITS;  // bytes the chunk stores cover

  for (int64_t r0 = warp * NGR; r0 < n; r0 += nwarps * NGR) {  // warp-uniform
    const int64_t r = r0 + lane / G;
    const bool act = r < n && (MIX ? mask[r] == BITS : (mask == nullptr || mask[r] != 0));  // group-uniform
    const float* x = X + (act ? r : 0) * ldx;
    uint8_t* row = packed + (MIX ? (act ? roff[r] : 0) : r * pitch);

    float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
    float v[CPL > 0 ? CPL : 1][8];
    if (CPL > 0) {
#pragma unroll
      for (int i = 0; i < (CPL > 0 ? CPL : 1); ++i) {
        const int c = gl + G * i;
        if (act && c < nchunks) {
          load_chunk(x, c, d, vec, x[0], v[i]);
#pragma unroll
          for (int k = 0; k < 8; ++k) { mn = fminf(mn, v[i][k]); mx = fmaxf(mx, v[i][k]); }
        }
      }
    } else if (act) {
      for (int c = gl; c < nchunks; c += G) {
        float w[8];
        load_chunk(x, c, d, vec, x[0], w);
#pragma unroll
        for (int k = 0; k < 8; ++k) { mn = fminf(mn, w[k]); mx = fmaxf(mx, w[k]); }
      }
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(FULL, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
    }
    if (!act) continue;
    // Eqn 4: Z = min, S = (max - min) / (2^b - 1)
    const float S = __fdiv_rn(__fsub_rn(mx, mn), L);
    const bool constant = !(S >= 1.17549435e-38f);  // S below FLT_MIN: code as constant
    const float inv = constant ? 0.0f : __frcp_rn(S);
    const uint32_t kr = row_key(seed_key, (uint32_t)r);

    if (CPL > 0) {
#pragma unroll
      for (int i = 0; i < (CPL > 0 ? CPL : 1); ++i) {
        const int c = gl + G * i;
        if (c < nchunks) store_word<BITS>(row + (int64_t)c * BITS, quantize_chunk<BITS>(v[i], c * 8, d, mn, inv, constant, kr));
      }
    } else {
      for (int c = gl; c < nchunks; c += G) {
        float w[8];
        load_chunk(x, c, d, vec, x[0], w);
        store_word<BITS>(row + (int64_t)c * BITS, quantize_chunk<BITS>(w, c * 8, d, mn, inv, constant, kr));
      }
    }
    if (gl == 0) *reinterpret_cast<float2*>(row + hoff) = make_float2(S, mn);
    for (int b = p8 + gl; b < hoff; b += G) row[b] = 0;
    for (int b = hoff + 8 + gl; b < pitch; b += G) row[b] = 0;
  }
}

// The same quantization, rows of d <= 8 G (one chunk per lane), one mask
// (or none): a warp takes the rows in blocks of 32, reads the block's mask
// bytes at once (one per lane), lists its marginal rows in shared memory and
// quantizes them 32 / G at a time, loading the next step's rows before the
// current ones are reduced and packed.  Central rows cost nothing but their
// mask byte.  The packed bytes are those of quantize_pack_kernel.
template <int BITS, int G>
__global__ void __launch_bounds__(kQuantThreads) quantize_rows_kernel(
    const float* __restrict__ X, int64_t n, int d, int64_t ldx, const uint8_t* __restrict__ mask,
    uint32_t seed_key, uint8_t* __restrict__ packed, int64_t pitch, int hoff, bool vec) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr int NGR = 32 / G;
  __shared__ uint8_t list_all[kQuantThreads / 32][32];
  const int lane = threadIdx.x & 31;
  const int gl = lane % G, k = lane / G;
  uint8_t* list = list_all[threadIdx.x >> 5];
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nchunks = (d + 7) >> 3;
  const int p8 = nchunks * BITS;
  const bool live = gl < nchunks;
  const float nan = __int_as_float(0x7fc00000);  // fill of columns >= d: ignored by fminf / fmaxf
  for (int64_t rb = warp * 32; rb < n; rb += nwarps * 32) {  // warp-uniform
    const bool on = rb + lane < n && (mask == nullptr || mask[rb + lane] != 0);
    const unsigned act = __ballot_sync(FULL, on);
    const int na = __popc(act);
    if (on) list[__popc(act & ((1u << lane) - 1u))] = (uint8_t)lane;
    __syncwarp();
    int64_t r = k < na ? rb + list[k] : -1;
    float v[8];
    if (r >= 0 && live) load_chunk(X + r * ldx, gl, d, vec, nan, v);
    for (int s0 = 0; s0 < na; s0 += NGR) {
      const int jn = s0 + NGR + k;
      const int64_t rn = jn < na ? rb + list[jn] : -1;
      float vn[8];
      if (rn >= 0 && live) load_chunk(X + rn * ldx, gl, d, vec, nan, vn);
      float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
      if (r >= 0 && live) {
#pragma unroll
        for (int i = 0; i < 8; ++i) { mn = fminf(mn, v[i]); mx = fmaxf(mx, v[i]); }
      }
#pragma unroll
      for (int o = G / 2; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(FULL, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
      }
      if (r >= 0) {
        // Eqn 4: Z = min, S = (max - min) / (2^b - 1)
        const float S = __fdiv_rn(__fsub_rn(mx, mn), L);
        const bool constant = !(S >= 1.17549435e-38f);  // S below FLT_MIN: code as constant
        const float inv = constant ? 0.0f : __frcp_rn(S);
        const uint32_t kr = row_key(seed_key, (uint32_t)r);
        uint8_t* row = packed + r * pitch;
        if (live) store_word<BITS>(row + (int64_t)gl * BITS, quantize_chunk<BITS>(v, gl * 8, d, mn, inv, constant, kr));
        if (gl == 0) *reinterpret_cast<float2*>(row + hoff) = make_float2(S, mn);
        for (int b = p8 + gl; b < hoff; b += G) row[b] = 0;
        for (int b = hoff + 8 + gl; b < pitch; b += G) row[b] = 0;
      }
      r = rn;
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = vn[i];
    }
    __syncwarp();  // the list is rewritten by the next block
  }
}

template <int BITS>
__global__ void __launch_bounds__(kQuantThreads) dequant_unpack_kernel(
    const uint8_t* __restrict__ packed, int64_t n, int d, int64_t pitch, int hoff,
    const uint8_t* __restrict__ mask, float* __restrict__ Y, int64_t ldy) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nchunks = (d + 7) >> 3;
  for (int64_t r = warp; r < n; r += nwarps) {
    if (mask != nullptr && mask[r] == 0) continue;
    const uint8_t* row = packed + r * pitch;
    const float2 h = *reinterpret_cast<const float2*>(row + hoff);
    for (int c = lane; c < nchunks; c += 32) {
      uint64_t w;
      if (BITS == 8) {
        const uint2 t = *reinterpret_cast<const uint2*>(row + (int64_t)c * 8);
        w = (uint64_t)t.x | ((uint64_t)t.y << 32);
      } else if (BITS == 4) {
        w = *reinterpret_cast<const uint32_t*>(row + (int64_t)c * 4);
      } else {
        w = *reinterpret_cast<const uint16_t*>(row + (int64_t)c * 2);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = c * 8 + i;
        if (j < d) {
          const uint32_t q = (uint32_t)(w >> (i * BITS)) & ((1u << BITS) - 1u);
          Y[r * ldy + j] = __fmaf_rn(code_to_float(q), h.x, h.y);
        }
      }
    }
  }
}

int grid_for_rows(int64_t n) {
  const int64_t rows_per_block = kQuantThreads / 32;
  int64_t g = (n + rows_per_block - 1) / rows_per_block;
  const int64_t cap = (int64_t)sm_count() * 8 * 4;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

template <int BITS, bool MIX>
int launch_quantize_t(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* mask, uint64_t seed,
                      uint8_t* packed, cudaStream_t s, const int64_t* roff) {
  const int64_t pitch = packed_pitch(d, BITS);
  const int hoff = (int)header_offset(d, BITS);
  const bool vec = aligned(X, 16) && (ldx % 4 == 0);
  const uint32_t h = seed_key_host(seed);
  // lanes per row: enough 8-column chunks for one each, up to a warp
  const int nch = (d + 7) / 8;
  const int G = nch <= 1 ? 1 : nch <= 2 ? 2 : nch <= 4 ? 4 : nch <= 8 ? 8 : nch <= 16 ? 16 : 32;
  const int grid = grid_for_rows((n + 32 / G - 1) / (32 / G));
  if (!MIX && d <= 8 * G) {  // one chunk per lane: the block-listing kernel
    const int gridb = grid_for_rows((n + 31) / 32);
    switch (G) {
      case 1: quantize_rows_kernel<BITS, 1><<<gridb, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec); break;
      case 2: quantize_rows_kernel<BITS, 2><<<gridb, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec); break;
      case 4: quantize_rows_kernel<BITS, 4><<<gridb, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec); break;
      case 8: quantize_rows_kernel<BITS, 8><<<gridb, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec); break;
      case 16: quantize_rows_kernel<BITS, 16><<<gridb, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec); break;
      default: quantize_rows_kernel<BITS, 32><<<gridb, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec); break;
    }
    return launch_status();
  }
  switch (G) {
    case 1: quantize_pack_kernel<BITS, 1, 1, MIX><<<grid, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec, roff); break;
    case 2: quantize_pack_kernel<BITS, 1, 2, MIX><<<grid, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec, roff); break;
    case 4: quantize_pack_kernel<BITS, 1, 4, MIX><<<grid, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec, roff); break;
    case 8: quantize_pack_kernel<BITS, 1, 8, MIX><<<grid, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec, roff); break;
    case 16: quantize_pack_kernel<BITS, 1, 16, MIX><<<grid, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec, roff); break;
    default:
      if (d <= 256)
        quantize_pack_kernel<BITS, 1, 32, MIX><<<grid, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec, roff);
      else if (d <= 512)
        quantize_pack_kernel<BITS, 2, 32, MIX><<<grid, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec, roff);
      else if (d <= 1024)
        quantize_pack_kernel<BITS, 4, 32, MIX><<<grid, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec, roff);
      else
        quantize_pack_kernel<BITS, 0, 32, MIX><<<grid, kQuantThreads, 0, s>>>(X, n, d, ldx, mask, h, packed, pitch, hoff, vec, roff);
  }
  return launch_status();
}

template <int BITS>
int launch_quantize(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* mask, uint64_t seed,
                    uint8_t* packed, cudaStream_t s, const int64_t* roff = nullptr) {
  return roff != nullptr ? launch_quantize_t<BITS, true>(X, n, d, ldx, mask, seed, packed, s, roff)
                         : launch_quantize_t<BITS, false>(X, n, d, ldx, mask, seed, packed, s, roff);
}

template <int BITS>
int launch_dequant(const uint8_t* packed, int64_t n, int d, const uint8_t* mask, float* Y, int64_t ldy,
                   cudaStream_t s) {
  dequant_unpack_kernel<BITS><<<grid_for_rows(n), kQuantThreads, 0, s>>>(
      packed, n, d, packed_pitch(d, BITS), (int)header_offset(d, BITS), mask, Y, ldy);
  return launch_status();
}

// Row offsets of a mixed packed buffer: rows of 4096 per block; each block
// adds up the sizes of the blocks before it, scans its own rows and writes
// roff[r] (and roff[n], the buffer size).
constexpr int kScanRows = 4096;
constexpr int kScanThr = 1024;

__device__ __forceinline__ int64_t row_bytes(uint8_t b, int d) {
  return (b == 2 || b == 4 || b == 8) ? packed_pitch(d, b) : 0;
}

__global__ void __launch_bounds__(kScanThr) offsets_tile_kernel(const uint8_t* __restrict__ rbits, int64_t n, int d,
                                                               int64_t* __restrict__ tile_sum) {
  __shared__ int64_t red[kScanThr / 32];
  const int64_t base = (int64_t)blockIdx.x * kScanRows;
  int64_t t = 0;
  for (int i = threadIdx.x; i < kScanRows; i += kScanThr)
    if (base + i < n) t += row_bytes(rbits[base + i], d);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(FULL, t, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t s = 0;
    for (int i = 0; i < kScanThr / 32; ++i) s += red[i];
    tile_sum[blockIdx.x] = s;
  }
}

__global__ void __launch_bounds__(kScanThr) offsets_scan_kernel(const uint8_t* __restrict__ rbits, int64_t n, int d,
                                                               const int64_t* __restrict__ tile_sum,
                                                               int64_t* __restrict__ roff) {
  __shared__ int64_t wsum[kScanThr / 32];
  __shared__ int64_t tile_base;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // the sizes of all earlier tiles, summed in tile order by warp 0
  if (w == 0) {
    int64_t t = 0;
    for (int64_t i = lane; i < (int64_t)blockIdx.x; i += 32) t += tile_sum[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(FULL, t, o);
    if (lane == 0) tile_base = t;
  }
  // each thread scans 4 consecutive rows of the tile
  constexpr int PER = kScanRows / kScanThr;
  const int64_t r0 = (int64_t)blockIdx.x * kScanRows + (int64_t)threadIdx.x * PER;
  int64_t sz[PER], own = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    sz[i] = r0 + i < n ? row_bytes(rbits[r0 + i], d) : 0;
    own += sz[i];
  }
  int64_t incl = own;  // inclusive scan over the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  int64_t before = tile_base;
  for (int i = 0; i < w; ++i) before += wsum[i];
  before += incl - own;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    if (r0 + i < n) roff[r0 + i] = before;
    before += sz[i];
  }
  if (r0 + PER >= n && r0 < n) roff[n] = before;  // the thread holding the last row
}

}  // namespace

int64_t offsets_tiles(int64_t n) { return (n + kScanRows - 1) / kScanRows; }

int packed_row_offsets(const uint8_t* rbits, int64_t n, int d, int64_t* roff, void* ws, size_t ws_bytes,
                       cudaStream_t s) {
  if (n < 0 || d < 1 || roff == nullptr || (n > 0 && rbits == nullptr)) return GQ_ERR_INVALID_ARG;
  if (n == 0) {
    GQ_TRY_CUDA(cudaMemsetAsync(roff, 0, sizeof(int64_t), s));
    return GQ_OK;
  }
  const int64_t tiles = offsets_tiles(n);
  if (tiles > 0x7fffffff) return GQ_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < (size_t)tiles * sizeof(int64_t) || !aligned(ws, 8)) return GQ_ERR_WORKSPACE;
  int64_t* tile_sum = static_cast<int64_t*>(ws);
  offsets_tile_kernel<<<(unsigned)tiles, kScanThr, 0, s>>>(rbits, n, d, tile_sum);
  GQ_TRY(launch_status());
  offsets_scan_kernel<<<(unsigned)tiles, kScanThr, 0, s>>>(rbits, n, d, tile_sum, roff);
  return launch_status();
}

int quantize_pack_mixed(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* rbits, const int64_t* roff,
                        uint64_t seed, uint8_t* packed, cudaStream_t s) {
  if (n < 0 || d < 1 || ldx < d) return GQ_ERR_INVALID_ARG;
  if (n > 0 && (X == nullptr || packed == nullptr || rbits == nullptr || roff == nullptr)) return GQ_ERR_INVALID_ARG;
  if (!aligned(packed, 16)) return GQ_ERR_INVALID_ARG;
  if (d > 16384) return GQ_ERR_UNSUPPORTED;
  if (n == 0) return GQ_OK;
  GQ_TRY(launch_quantize<2>(X, n, d, ldx, rbits, seed, packed, s, roff));
  GQ_TRY(launch_quantize<4>(X, n, d, ldx, rbits, seed, packed, s, roff));
  return launch_quantize<8>(X, n, d, ldx, rbits, seed, packed, s, roff);
}

int quantize_pack(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* mask, int bits, uint64_t seed,
                  uint8_t* packed, cudaStream_t s) {
  if (n < 0 || d < 1 || ldx < d || !valid_bits(bits)) return GQ_ERR_INVALID_ARG;
  if (n > 0 && (X == nullptr || packed == nullptr)) return GQ_ERR_INVALID_ARG;
  if (!aligned(packed, 16)) return GQ_ERR_INVALID_ARG;
  if (d > 16384) return GQ_ERR_UNSUPPORTED;
  if (n == 0) return GQ_OK;
  switch (bits) {
    case 2: return launch_quantize<2>(X, n, d, ldx, mask, seed, packed, s);
    case 4: return launch_quantize<4>(X, n, d, ldx, mask, seed, packed, s);
    default: return launch_quantize<8>(X, n, d, ldx, mask, seed, packed, s);
  }
}

}  // namespace gq

extern "C" int gq_quantize_pack(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* mask, int bits,
                                uint64_t seed, uint8_t* packed, gq_stream stream) {
  return gq::quantize_pack(X, n, d, ldx, mask, bits, seed, packed, (cudaStream_t)stream);
}

extern "C" int gq_dequant_unpack(const uint8_t* packed, int64_t n, int d, int bits, const uint8_t* mask, float* Y,
                                 int64_t ldy, gq_stream stream) {
  if (n < 0 || d < 1 || ldy < d || !gq::valid_bits(bits)) return GQ_ERR_INVALID_ARG;
  if (n > 0 && (packed == nullptr || Y == nullptr)) return GQ_ERR_INVALID_ARG;
  if (!gq::aligned(packed, 16)) return GQ_ERR_INVALID_ARG;
  if (n == 0) return GQ_OK;
  cudaStream_t s = (cudaStream_t)stream;
  switch (bits) {
    case 2: return gq::launch_dequant<2>(packed, n, d, mask, Y, ldy, s);
    case 4: return gq::launch_dequant<4>(packed, n, d, mask, Y, ldy, s);
    default: return gq::launch_dequant<8>(packed, n, d, mask, Y, ldy, s);
  }
}

extern "C" size_t gq_packed_row_offsets_workspace_bytes(int64_t n) {
  return n > 0 ? (size_t)gq::offsets_tiles(n) * sizeof(int64_t) : 0;
}

extern "C" int gq_packed_row_offsets(const uint8_t* rbits, int64_t n, int d, int64_t* roff, void* ws,
                                     size_t ws_bytes, gq_stream stream) {
  return gq::packed_row_offsets(rbits, n, d, roff, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int gq_quantize_pack_mixed(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* rbits,
                                      const int64_t* roff, uint64_t seed, uint8_t* packed, gq_stream stream) {
  return gq::quantize_pack_mixed(X, n, d, ldx, rbits, roff, seed, packed, (cudaStream_t)stream);
}
