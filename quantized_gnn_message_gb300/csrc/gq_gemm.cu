// gq_gemm.cu -- dense update GEMMs of the layer on 5th-generation tensor
// cores (tcgen05, kind::f16 with bf16 inputs and fp32 accumulation in TMEM).
//
//   row GEMM     C[M x N] = act(A[M x K] B[N x K]^T)      (Z = A W, dA = dZ W^T,
//                                                          H' = H W)
//   weight GEMM  C[K1 x N1] = X[R x K1]^T Y[R x N1]        (dW = A^T dZ)
//
// (AdaQP Sec. 2.1: the update h_v = sigma(W h_N(v)); Tango Sec. 2.1 step 1
// H' = H W and its backward dW = H^T dH', dH = dH' W^T.)
//
// Row GEMM: persistent, one CTA per SM, warp-specialized.
//   warp 0  one thread issues TMA: all of B once (K-major, 128-byte swizzle,
//           resident in shared memory), then 128 x 64 tiles of A into a ring
//           of stages;
//   warp 1  allocates TMEM; one thread issues tcgen05.mma (M=128, N<=256,
//           K=16 per instruction) into one of two TMEM accumulators and
//           commits stage releases / accumulator-ready to mbarriers;
//   warps 2-9  epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (thread =
//           row) over one half of the columns, 64 columns per wait,
//           activation, optional GAT head projections (the head vectors in
//           shared memory), fp32 rows staged in shared memory and written
//           by TMA stores, 32 rows x 16 columns each, two in flight per
//           warp; then release the accumulator, so the next tile's MMAs
//           overlap it.
// Weight GEMM: grid (M tiles of K1) x (row splits); both operands MN-major
// (their rows are the contraction), one TMEM accumulator per CTA, fp32
// partials to a workspace, then a fixed-order reduction over splits.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>

#include "gq_common.cuh"
#include "gq_internal.cuh"
#include "gq_sm100.cuh"

namespace gq {
namespace {

constexpr int kRgThreads = 320;  // TMA warp, MMA warp, 8 epilogue warps
constexpr int kRgEpiWarps = 8;
constexpr int kTileM = 128;
constexpr int kChunkK = 64;                       // bf16 elements per 128-byte swizzle row
constexpr int kATileBytes = kTileM * kChunkK * 2;  // 16 KB
constexpr int kSmemBudget = 225 * 1024;
// epilogue staging, 4 KB per epilogue warp: two 32-row x 16-column fp32
// boxes for TMA stores (64-byte rows, 64-byte swizzle: conflict-free 16-byte
// writes by row), or one 32 x 16 block at a row pitch of 20 floats for
// plain stores
constexpr int kStgPitch = 20;
constexpr int kStgWarpBytes = 4096;
constexpr int kStgBytes = kRgEpiWarps * kStgWarpBytes;
constexpr int kVecBytes = 2 * 256 * 4;  // a_src | a_dst of the GAT head projections

// ---------------------------------------------------------------- host ---
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D bf16 tensor [outer][inner] with row pitch ld (elements); box of
// box_inner x box_outer, 128-byte swizzle, zero fill out of bounds.
// 2-D fp32 tensor [outer][inner] with row pitch ld (elements); box of
// 16 x 32, 64-byte swizzle: the output boxes of the row GEMM's TMA stores.
int make_tmap_f32_out(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t ld) {
  auto fn = encode_fn();
  if (fn == nullptr) return GQ_ERR_CUDA;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 4};
  const cuuint32_t box[2] = {16, 32};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GQ_OK : GQ_ERR_INVALID_ARG;
}

int make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
              uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return GQ_ERR_CUDA;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GQ_OK : GQ_ERR_INVALID_ARG;
}

uint32_t pow2_at_least(uint32_t x) {
  uint32_t p = 32;
  while (p < x) p <<= 1;
  return p;
}

// ------------------------------------------------------------- row GEMM ---
struct RowGemmArgs {
  int64_t M;
  int N, Npad, K, kch, stages;
  uint32_t tmem_cols, acc_stride;
  float* C;
  int64_t ldc;
  int act;
  int vec;
  int tma;              // C written by TMA stores (tmC)
  int half;             // columns [0, half) to epilogue warps 2-5, [half, Npad) to warps 6-9
  uint32_t* rbits;      // optional [C > 0] bits: bit c % 32 of rbits[r * ldrb + c / 32]
  int64_t ldrb;
  const float* a_src;   // optional GAT head projections
  const float* a_dst;
  float* S;
  float* D;
  int heads, fshift;
  int* err;
};

__global__ void __launch_bounds__(kRgThreads, 1)
    row_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const RowGemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sB = smem;
  uint8_t* sA = sB + (size_t)p.kch * p.Npad * 128;
  float* stg_all = reinterpret_cast<float*>(sA + (size_t)p.stages * kATileBytes);  // 1024-byte aligned
  float* svec = stg_all + kStgBytes / 4;                                              // [2][Npad]
  uint64_t* full = reinterpret_cast<uint64_t*>(svec + kVecBytes / 4);
  uint64_t* empty = full + p.stages;
  uint64_t* bfull = empty + p.stages;
  uint64_t* tfull = bfull + 1;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(bfull, 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kRgEpiWarps);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  if (p.S != nullptr)
    for (int j = threadIdx.x; j < p.Npad; j += kRgThreads) {
      svec[j] = j < p.N ? __ldg(p.a_src + j) : 0.0f;
      svec[p.Npad + j] = j < p.N ? __ldg(p.a_dst + j) : 0.0f;
    }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int64_t ntiles = (p.M + kTileM - 1) / kTileM;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      if (p.tma) prefetch_tmap(&tmC);
      mbar_expect_tx(bfull, (uint32_t)(p.kch * p.Npad * 128));
      for (int kc = 0; kc < p.kch; ++kc) tma_load_2d(sB + (size_t)kc * p.Npad * 128, &tmB, kc * kChunkK, 0, bfull);
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        bool ok = true;
        for (int kc = 0; kc < p.kch && ok; ++kc) {
          ok = mbar_wait(&empty[stage], phase ^ 1, abort, p.err, 1);
          if (!ok) break;
          mbar_expect_tx(&full[stage], kATileBytes);
          tma_load_2d(sA + (size_t)stage * kATileBytes, &tmA, kc * kChunkK, (int)(t * kTileM), &full[stage]);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, p.Npad, 0, 0);
      bool ok = mbar_wait(bfull, 0, abort, p.err, 2);
      int stage = 0;
      uint32_t phase = 0;
      int i = 0;
      for (int64_t t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++i) {
        const int a = i & 1;
        const uint32_t use = (uint32_t)(i >> 1);
        if (!(ok = mbar_wait(&tempty[a], (use & 1) ^ 1, abort, p.err, 3))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + a * p.acc_stride;
        for (int kc = 0; kc < p.kch; ++kc) {
          if (!(ok = mbar_wait(&full[stage], phase, abort, p.err, 4))) break;
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + (size_t)stage * kATileBytes);
          const uint32_t b_base = smem_u32(sB + (size_t)kc * p.Npad * 128);
#pragma unroll
          for (int k = 0; k < kChunkK / 16; ++k) {
            umma_f16(d_tmem, smem_desc_sw128(a_base + 32 * k, 16, 1024), smem_desc_sw128(b_base + 32 * k, 16, 1024),
                     idesc, (kc | k) != 0);
          }
          umma_commit(&empty[stage]);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[a]);
      }
    }
  } else {
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    const int h = (warp - 2) >> 2;
    const int cb = h ? p.half : 0, ce = h ? p.Npad : p.half;
    float* stg = stg_all + (warp - 2) * (kStgWarpBytes / 4);
    int nbox = 0;  // boxes this warp has stored
    int i = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int a = i & 1;
      const uint32_t use = (uint32_t)(i >> 1);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[a], use & 1, abort, p.err, 5);
      ok = __shfl_sync(FULL, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int64_t row = t * kTileM + row_in_tile;
      const bool live = row < p.M;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + a * p.acc_stride;
      float* crow = p.C + row * p.ldc;
      float hs = 0.0f, hd = 0.0f;
      for (int c1 = cb; c1 < ce; c1 += 64) {
        const int nc = min(4, (ce - c1) >> 4);  // 16-column chunks this round
        uint64_t rb = 0;                         // [value > 0] of the round's columns
        uint32_t r[4][16];
        tmem_ld16(taddr + c1, r[0]);
        if (nc > 1) tmem_ld16(taddr + c1 + 16, r[1]);
        if (nc > 2) tmem_ld16(taddr + c1 + 32, r[2]);
        if (nc > 3) tmem_ld16(taddr + c1 + 48, r[3]);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (u >= nc) break;
          const int c0 = c1 + 16 * u;
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            v[j] = __uint_as_float(r[u][j]);
            if (p.act == GQ_ACT_RELU) v[j] = fmaxf(v[j], 0.0f);
            rb |= (uint64_t)(v[j] > 0.0f ? 1u : 0u) << (16 * u + j);
          }
          if (p.tma && c0 < p.N) {
            // row `lane` of the box; 16-byte piece j at piece j ^ ((lane >> 1) & 3)
            float* box = stg + (nbox & 1) * 512;
            if (lane == 0) bulk_wait_read<1>();  // the store of two boxes ago has read this buffer
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<float4*>(box + lane * 16 + 4 * (j ^ ((lane >> 1) & 3))) =
                  make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            const int64_t y = t * kTileM + q * 32;
            if (lane == 0) {
              if (y < p.M) tma_store_2d(&tmC, box, c0, (int)y);
              bulk_commit();
            }
            ++nbox;
          } else if (p.vec && c0 + 16 <= p.N) {
            // through shared memory, so that each store instruction writes 8
            // rows x 64 contiguous bytes instead of 32 rows x 16 bytes
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<float4*>(stg + lane * kStgPitch + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int rr = 8 * k + (lane >> 2), cg = 4 * (lane & 3);
              const int64_t grow = t * kTileM + q * 32 + rr;
              const float4 o = *reinterpret_cast<const float4*>(stg + rr * kStgPitch + cg);
              if (grow < p.M) *reinterpret_cast<float4*>(p.C + grow * p.ldc + c0 + cg) = o;
            }
            __syncwarp();
          } else if (live) {
            for (int j = 0; j < 16 && c0 + j < p.N; ++j) crow[c0 + j] = v[j];
          }
          if (live && p.S != nullptr && c0 < p.N) {
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const float4 as = *reinterpret_cast<const float4*>(svec + c0 + j);
              const float4 ad = *reinterpret_cast<const float4*>(svec + p.Npad + c0 + j);
              hs = __fmaf_rn(v[j], as.x, hs);
              hs = __fmaf_rn(v[j + 1], as.y, hs);
              hs = __fmaf_rn(v[j + 2], as.z, hs);
              hs = __fmaf_rn(v[j + 3], as.w, hs);
              hd = __fmaf_rn(v[j], ad.x, hd);
              hd = __fmaf_rn(v[j + 1], ad.y, hd);
              hd = __fmaf_rn(v[j + 2], ad.z, hd);
              hd = __fmaf_rn(v[j + 3], ad.w, hd);
            }
            if (((c0 + 16) >> p.fshift) != (c0 >> p.fshift) || c0 + 16 >= p.N) {
              const int head = c0 >> p.fshift;
              p.S[row * p.heads + head] = hs;
              p.D[row * p.heads + head] = hd;
              hs = hd = 0.0f;
            }
          }
        }
        if (p.rbits != nullptr && live) {
          if (c1 < p.N) p.rbits[row * p.ldrb + (c1 >> 5)] = (uint32_t)rb;
          if (nc > 2 && c1 + 32 < p.N) p.rbits[row * p.ldrb + (c1 >> 5) + 1] = (uint32_t)(rb >> 32);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
    }
    if (lane == 0) bulk_wait<0>();  // every TMA store of this warp done
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ---------------------------------------------------------- weight GEMM ---
constexpr int kWgThreads = 192;
constexpr int kWgRows = 64;  // contraction rows per stage

struct WgradArgs {
  int64_t R;
  int K1, N1, Npad, nb;   // nb = 64-wide blocks of N1
  int stages;
  int64_t rows_per_split;
  uint32_t tmem_cols;
  float* partial;         // [split][mtile][128][Npad]
  int mtiles;
  int* err;
};

__global__ void __launch_bounds__(kWgThreads, 1)
    wgrad_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                      const WgradArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int a_bytes = 2 * kWgRows * 128;           // two 64-wide blocks of K1
  const int b_bytes = p.nb * kWgRows * 128;
  const int stage_bytes = a_bytes + b_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * stage_bytes);
  uint64_t* empty = full + p.stages;
  uint64_t* tfull = empty + p.stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x;
  const int64_t r0 = (int64_t)blockIdx.y * p.rows_per_split;
  int64_t r1 = r0 + p.rows_per_split;
  if (r1 > p.R) r1 = p.R;
  const int nsteps = r1 > r0 ? (int)((r1 - r0 + kWgRows - 1) / kWgRows) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmY);
      int stage = 0;
      uint32_t phase = 0;
      for (int s = 0; s < nsteps; ++s) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort, p.err, 11)) break;
        uint8_t* st = smem + (size_t)stage * stage_bytes;
        const int row = (int)(r0 + (int64_t)s * kWgRows);
        mbar_expect_tx(&full[stage], (uint32_t)stage_bytes);
        tma_load_2d(st, &tmX, mt * 128, row, &full[stage]);
        tma_load_2d(st + kWgRows * 128, &tmX, mt * 128 + 64, row, &full[stage]);
        for (int b = 0; b < p.nb; ++b) tma_load_2d(st + a_bytes + b * kWgRows * 128, &tmY, b * 64, row, &full[stage]);
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.Npad, 1, 1);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int s = 0; s < nsteps; ++s) {
        if (!(ok = mbar_wait(&full[stage], phase, abort, p.err, 12))) break;
        tc_fence_after();
        const uint32_t base = smem_u32(smem + (size_t)stage * stage_bytes);
#pragma unroll
        for (int k = 0; k < kWgRows / 16; ++k) {
          // 16 contraction rows = two 8-row swizzle atoms (SBO apart)
          const uint64_t ad = smem_desc_sw128(base + 2048 * k, kWgRows * 128, 1024);
          const uint64_t bd = smem_desc_sw128(base + a_bytes + 2048 * k, kWgRows * 128, 1024);
          umma_f16(tmem, ad, bd, idesc, (s | k) != 0);
        }
        umma_commit(&empty[stage]);
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (ok) umma_commit(tfull);
    }
  } else {
    const int q = warp & 3;
    const int row = q * 32 + lane;  // row of the 128 x Npad tile (a K1 index)
    float* out = p.partial + (((int64_t)blockIdx.y * p.mtiles + mt) * 128 + row) * p.Npad;
    if (nsteps == 0) {
      for (int c = 0; c < p.Npad; ++c) out[c] = 0.0f;
    } else {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(tfull, 0, abort, p.err, 13);
      ok = __shfl_sync(FULL, ok, 0);
      if (ok) {
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
        for (int c0 = 0; c0 < p.Npad; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(taddr + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            st_f4(out + c0 + j, __uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                  __uint_as_float(r[j + 3]));
        }
        tc_fence_before();
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// C[i][j] = sum over splits, in split order.
__global__ void wgrad_reduce_kernel(const float* __restrict__ partial, int splits, int mtiles, int K1, int N1,
                                    int Npad, float* C, int64_t ldc, int accumulate) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)K1 * N1) return;
  const int i = (int)(idx / N1), j = (int)(idx % N1);
  const int mt = i >> 7, r = i & 127;
  float s = 0.0f;
  for (int sp = 0; sp < splits; ++sp) s += partial[(((int64_t)sp * mtiles + mt) * 128 + r) * Npad + j];
  C[(int64_t)i * ldc + j] = accumulate ? C[(int64_t)i * ldc + j] + s : s;
}

// -------------------------------------------------------- conversions ---
// dst[r][c] = bf16(src[r][c]) for c < cols, 0 for cols <= c < dcols, and
// 0 also where gate[r][c] <= 0 (ReLU' taken from the layer output).  A
// block covers rpb rows, tpr threads a row, each thread 4 columns at a time
// (VEC: one 16-byte load per operand and one 8-byte store).
template <bool VEC>
__global__ void to_bf16_kernel(const float* __restrict__ src, int64_t rows, int cols, int64_t lds,
                               __nv_bfloat16* __restrict__ dst, int64_t ldd, int dcols,
                               const float* __restrict__ gate, int64_t ldg, int tpr, int rpb) {
  const int local = (int)threadIdx.x / tpr;
  const int64_t r = (int64_t)blockIdx.x * rpb + local;
  if (local >= rpb || r >= rows) return;
  for (int c = ((int)threadIdx.x - local * tpr) * 4; c < dcols; c += 4 * tpr) {
  float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (VEC && c + 4 <= cols) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(src + r * lds + c));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    if (gate != nullptr) {
      const float4 gv = __ldg(reinterpret_cast<const float4*>(gate + r * ldg + c));
      if (!(gv.x > 0.0f)) v[0] = 0.0f;
      if (!(gv.y > 0.0f)) v[1] = 0.0f;
      if (!(gv.z > 0.0f)) v[2] = 0.0f;
      if (!(gv.w > 0.0f)) v[3] = 0.0f;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (c + k < cols) {
        v[k] = src[r * lds + c + k];
        if (gate != nullptr && !(gate[r * ldg + c + k] > 0.0f)) v[k] = 0.0f;
      }
    }
  }
  __nv_bfloat16* d = dst + r * ldd + c;
  if (VEC && c + 4 <= dcols) {
    *reinterpret_cast<uint2*>(d) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (c + k < dcols) d[k] = __float2bfloat16_rn(v[k]);
  }
  }
}

// dst[n][k] = bf16(W[k][n]) (transpose), zero for k >= K.
__global__ void transpose_bf16_kernel(const float* __restrict__ W, int K, int N, int64_t ldw,
                                      __nv_bfloat16* __restrict__ dst, int64_t ldd, int kpad) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)N * kpad) return;
  const int n = (int)(idx / kpad), k = (int)(idx % kpad);
  dst[(int64_t)n * ldd + k] = __float2bfloat16_rn(k < K ? W[(int64_t)k * ldw + n] : 0.0f);
}

}  // namespace

// ------------------------------------------------------------------ API ---
int row_gemm(const void* A, int64_t M, int K, int64_t lda, const void* B, int N, int64_t ldb, int act, float* C,
             int64_t ldc, const float* a_src, const float* a_dst, float* S, float* D, int heads, int* err,
             cudaStream_t s, uint32_t* rbits, int64_t ldrb) {
  if (A == nullptr || B == nullptr || C == nullptr || M < 0 || K < 1 || N < 1) return GQ_ERR_INVALID_ARG;
  if (K > 256 || N > 256) return GQ_ERR_UNSUPPORTED;
  if (lda < K || ldb < K || ldc < N || lda % 8 || ldb % 8 || !aligned(A, 16) || !aligned(B, 16))
    return GQ_ERR_INVALID_ARG;
  if (act != GQ_ACT_NONE && act != GQ_ACT_RELU) return GQ_ERR_INVALID_ARG;
  int fshift = 0;
  if (S != nullptr) {
    if (D == nullptr || a_src == nullptr || a_dst == nullptr || heads < 1 || N % heads) return GQ_ERR_INVALID_ARG;
    const int F = N / heads;
    while ((1 << fshift) < F) ++fshift;
    if ((1 << fshift) != F || F < 16) return GQ_ERR_UNSUPPORTED;
  }
  if (M == 0) return GQ_OK;
  RowGemmArgs p{};
  p.M = M;
  p.N = N;
  p.Npad = (N + 15) / 16 * 16;
  p.K = K;
  p.kch = (K + kChunkK - 1) / kChunkK;
  const int b_bytes = p.kch * p.Npad * 128;
  p.stages = (kSmemBudget - 2048 - b_bytes - kStgBytes - kVecBytes) / kATileBytes;
  if (p.stages > 8) p.stages = 8;
  if (p.stages < 2) return GQ_ERR_UNSUPPORTED;
  p.tmem_cols = pow2_at_least(2 * (uint32_t)p.Npad);
  p.acc_stride = p.tmem_cols / 2;
  p.C = C;
  p.ldc = ldc;
  p.act = act;
  p.vec = (ldc % 4 == 0) && aligned(C, 16);
  p.tma = p.vec && M <= INT32_MAX - kTileM;
  // the two epilogue column halves, 16-aligned; with head projections a
  // half holds whole heads, else every column goes to the first half
  p.half = (p.Npad / 2 + 15) / 16 * 16;
  if (S != nullptr && p.half % (1 << fshift) != 0) p.half = p.Npad;
  if (rbits != nullptr) {  // a word of bits is one 32-column round of one half
    if (ldrb < (N + 31) / 32 || !aligned(rbits, 4)) return GQ_ERR_INVALID_ARG;
    p.half = min((p.Npad / 2 + 31) / 32 * 32, p.Npad);
    if (S != nullptr && p.half % (1 << fshift) != 0) p.half = p.Npad;
  }
  p.rbits = rbits;
  p.ldrb = ldrb;
  p.a_src = a_src;
  p.a_dst = a_dst;
  p.S = S;
  p.D = D;
  p.heads = heads;
  p.fshift = fshift;
  p.err = err;
  CUtensorMap tmA, tmB, tmC;
  GQ_TRY(make_tmap(&tmA, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, kChunkK, kTileM));
  GQ_TRY(make_tmap(&tmB, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, kChunkK, (uint32_t)p.Npad));
  memset(&tmC, 0, sizeof(tmC));
  if (p.tma) GQ_TRY(make_tmap_f32_out(&tmC, C, (uint64_t)N, (uint64_t)M, (uint64_t)ldc));
  const size_t smem = 1024 + (size_t)b_bytes + (size_t)p.stages * kATileBytes + kStgBytes + kVecBytes + 256;
  GQ_TRY_CUDA(cudaFuncSetAttribute(row_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  const int64_t ntiles = (M + kTileM - 1) / kTileM;
  const int grid = (int)(ntiles < sm_count() ? ntiles : sm_count());
  row_gemm_kernel<<<grid, kRgThreads, smem, s>>>(tmA, tmB, tmC, p);
  return launch_status();
}

static void wgrad_plan(int64_t R, int K1, int N1, int* mtiles, int* splits, int* npad) {
  *mtiles = (K1 + 127) / 128;
  *npad = (N1 + 15) / 16 * 16;
  int64_t steps = (R + kWgRows - 1) / kWgRows;
  int64_t sp = sm_count() / *mtiles;
  if (sp < 1) sp = 1;
  if (sp > steps) sp = steps > 0 ? steps : 1;
  *splits = (int)sp;
}

size_t wgrad_workspace(int64_t R, int K1, int N1) {
  int mt, sp, np;
  wgrad_plan(R, K1, N1, &mt, &sp, &np);
  return (size_t)sp * mt * 128 * np * sizeof(float) + 256;
}

int wgrad_gemm(const void* X, int64_t R, int K1, int64_t ldx, const void* Y, int N1, int64_t ldy, float* C,
               int64_t ldc, int accumulate, void* ws, size_t ws_bytes, int* err, cudaStream_t s) {
  if (C == nullptr || R < 0 || K1 < 1 || N1 < 1 || ldc < N1) return GQ_ERR_INVALID_ARG;
  if (K1 > 256 || N1 > 256) return GQ_ERR_UNSUPPORTED;
  if (R == 0) {  // empty contraction: C = 0, or C unchanged when accumulating
    if (accumulate) return GQ_OK;
    GQ_TRY_CUDA(cudaMemset2DAsync(C, (size_t)ldc * sizeof(float), 0, (size_t)N1 * sizeof(float), (size_t)K1, s));
    return GQ_OK;
  }
  if (X == nullptr || Y == nullptr) return GQ_ERR_INVALID_ARG;
  if (ldx < K1 || ldy < N1 || ldx % 8 || ldy % 8 || !aligned(X, 16) || !aligned(Y, 16)) return GQ_ERR_INVALID_ARG;
  WgradArgs p{};
  int splits;
  wgrad_plan(R, K1, N1, &p.mtiles, &splits, &p.Npad);
  if (ws == nullptr || ws_bytes < wgrad_workspace(R, K1, N1) || !aligned(ws, 16)) return GQ_ERR_WORKSPACE;
  p.R = R;
  p.K1 = K1;
  p.N1 = N1;
  p.nb = (N1 + 63) / 64;
  const int stage_bytes = (2 + p.nb) * kWgRows * 128;
  p.stages = (kSmemBudget - 2048) / stage_bytes;
  if (p.stages > 6) p.stages = 6;
  if (p.stages < 2) return GQ_ERR_UNSUPPORTED;
  const int64_t steps = (R + kWgRows - 1) / kWgRows;
  p.rows_per_split = ((steps + splits - 1) / splits) * kWgRows;
  p.tmem_cols = pow2_at_least((uint32_t)p.Npad);
  p.partial = static_cast<float*>(ws);
  p.err = err;
  CUtensorMap tmX, tmY;
  const uint64_t rows = R > 0 ? (uint64_t)R : 1;
  GQ_TRY(make_tmap(&tmX, X, (uint64_t)K1, rows, (uint64_t)ldx, 64, kWgRows));
  GQ_TRY(make_tmap(&tmY, Y, (uint64_t)N1, rows, (uint64_t)ldy, 64, kWgRows));
  const size_t smem = 1024 + (size_t)p.stages * stage_bytes + 256;
  GQ_TRY_CUDA(cudaFuncSetAttribute(wgrad_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  dim3 grid(p.mtiles, splits);
  wgrad_gemm_kernel<<<grid, kWgThreads, smem, s>>>(tmX, tmY, p);
  GQ_TRY(launch_status());
  const int64_t total = (int64_t)K1 * N1;
  wgrad_reduce_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(p.partial, splits, p.mtiles, K1, N1, p.Npad, C,
                                                                      ldc, accumulate);
  return launch_status();
}

int to_bf16(const float* src, int64_t rows, int cols, int64_t lds, void* dst, int64_t ldd, int dcols,
            const float* gate, int64_t ldg, cudaStream_t s) {
  if (rows == 0 || dcols == 0) return GQ_OK;
  const int tpr = min((dcols + 3) / 4, 256);  // threads a row; wider rows loop
  const int rpb = 256 / tpr;
  const int64_t blocks = (rows + rpb - 1) / rpb;
  if (blocks > 0x7fffffff) return GQ_ERR_UNSUPPORTED;
  auto* d = static_cast<__nv_bfloat16*>(dst);
  const bool vec = lds % 4 == 0 && ldd % 4 == 0 && aligned(src, 16) && aligned(dst, 8) &&
                   (gate == nullptr || (ldg % 4 == 0 && aligned(gate, 16)));
  if (vec)
    to_bf16_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(src, rows, cols, lds, d, ldd, dcols, gate, ldg, tpr, rpb);
  else
    to_bf16_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(src, rows, cols, lds, d, ldd, dcols, gate, ldg, tpr, rpb);
  return launch_status();
}

int transpose_bf16(const float* W, int K, int N, int64_t ldw, void* dst, int64_t ldd, int kpad, cudaStream_t s) {
  const int64_t total = (int64_t)N * kpad;
  transpose_bf16_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(W, K, N, ldw,
                                                                         static_cast<__nv_bfloat16*>(dst), ldd, kpad);
  return launch_status();
}

}  // namespace gq

extern "C" int gq_gemm_bf16_nt(const uint16_t* A, int64_t M, int K, int64_t lda, const uint16_t* B, int N,
                               int64_t ldb, int act, float* C, int64_t ldc, int* dev_err, gq_stream stream) {
  return gq::row_gemm(A, M, K, lda, B, N, ldb, act, C, ldc, nullptr, nullptr, nullptr, nullptr, 0, dev_err,
                      (cudaStream_t)stream);
}

extern "C" size_t gq_gemm_bf16_tn_workspace_bytes(int64_t R, int K1, int N1) {
  if (R < 0 || K1 < 1 || N1 < 1) return 0;
  return gq::wgrad_workspace(R, K1, N1);
}

extern "C" int gq_gemm_bf16_tn(const uint16_t* X, int64_t R, int K1, int64_t ldx, const uint16_t* Y, int N1,
                               int64_t ldy, float* C, int64_t ldc, int accumulate, void* ws, size_t ws_bytes,
                               int* dev_err, gq_stream stream) {
  return gq::wgrad_gemm(X, R, K1, ldx, Y, N1, ldy, C, ldc, accumulate, ws, ws_bytes, dev_err, (cudaStream_t)stream);
}

extern "C" int gq_to_bf16(const float* src, int64_t rows, int cols, int64_t lds, uint16_t* dst, int64_t ldd,
                          int dcols, gq_stream stream) {
  if (src == nullptr || dst == nullptr || rows < 0 || cols < 1 || dcols < cols || lds < cols || ldd < dcols)
    return GQ_ERR_INVALID_ARG;
  return gq::to_bf16(src, rows, cols, lds, dst, ldd, dcols, nullptr, 0, (cudaStream_t)stream);
}
