// gq_internal.cuh -- library-internal entry points shared between the
// translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gq.h"

namespace gq {

int quantize_pack(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* mask, int bits, uint64_t seed,
                  uint8_t* packed, cudaStream_t s);

// Aggregation; Yb != nullptr writes the output in bf16 (leading dim ldy);
// gate != nullptr zeroes every output element (r, c) whose bit c % 32 of
// gate[r * ldg + c / 32] is clear.
size_t spmm_workspace(const gq_graph* g, int transpose, int d);
int spmm_check(const gq_graph* g, const float* X, int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d,
               int bits, const float* Y, int64_t ldy, const void* Yb);
int dequant_spmm(const gq_graph* g, int transpose, int coef, const float* X, int64_t ldx, const uint8_t* packed,
                 const uint8_t* mask, int d, int bits, float* Y, int64_t ldy, void* ws, size_t ws_bytes,
                 cudaStream_t s, void* Yb, const uint32_t* gate = nullptr, int64_t ldg = 0);
int edge_spmm(const gq_graph* g, int transpose, const float* alpha, int heads, const float* X, int64_t ldx,
              const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y, int64_t ldy, void* ws,
              size_t ws_bytes, cudaStream_t s);
int edge_spmm_alpha8(const gq_graph* g, const uint8_t* acode, const float* ahdr, int heads, const float* X,
                     int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y,
                     int64_t ldy, void* ws, size_t ws_bytes, cudaStream_t s);

// rbits != nullptr: bit c % 32 of rbits[r * ldrb + c / 32] = [C[r][c] > 0]
int row_gemm(const void* A, int64_t M, int K, int64_t lda, const void* B, int N, int64_t ldb, int act, float* C,
             int64_t ldc, const float* a_src, const float* a_dst, float* S, float* D, int heads, int* err,
             cudaStream_t s, uint32_t* rbits = nullptr, int64_t ldrb = 0);
size_t wgrad_workspace(int64_t R, int K1, int N1);
int wgrad_gemm(const void* X, int64_t R, int K1, int64_t ldx, const void* Y, int N1, int64_t ldy, float* C,
               int64_t ldc, int accumulate, void* ws, size_t ws_bytes, int* err, cudaStream_t s);
// dst = bf16(src), columns [cols, dcols) zero; with gate, elements whose
// gate value is not > 0 become 0 (ReLU derivative taken from the output).
int to_bf16(const float* src, int64_t rows, int cols, int64_t lds, void* dst, int64_t ldd, int dcols,
            const float* gate, int64_t ldg, cudaStream_t s);
// dst[n][k] = bf16(W[k][n]) for k < K, 0 for K <= k < kpad.
int transpose_bf16(const float* W, int K, int N, int64_t ldw, void* dst, int64_t ldd, int kpad, cudaStream_t s);

// Bump allocator over a caller workspace (256-byte aligned pieces).
struct Carve {
  char* base;
  size_t cap, used = 0;
  Carve(void* b, size_t c) : base(static_cast<char*>(b)), cap(c) {}
  void* take(size_t bytes) {
    const size_t off = (used + 255) & ~(size_t)255;
    used = off + bytes;
    return (base == nullptr || used > cap) ? nullptr : base + off;
  }
  bool ok() const { return base != nullptr && used <= cap; }
};

inline int64_t round8(int64_t x) { return (x + 7) / 8 * 8; }

}  // namespace gq

namespace gq {

// GAT edge kernels (gq_gat.cu)
size_t edge_softmax_workspace(const gq_graph* g, int heads);
size_t edge_bwd_workspace(const gq_graph* g, int heads);
size_t node_bwd_workspace(const gq_graph* g, int heads, int d);
int edge_softmax(const gq_graph* g, const float* S, const float* D, int heads, float slope, float* Epre,
                 float* alpha, void* ws, size_t ws_bytes, cudaStream_t s);
size_t edge_quant_workspace(const gq_graph* g, int heads);
int quantize_edge_values(const gq_graph* g, const float* alpha, int heads, uint64_t seed, uint8_t* codes, float* hdr,
                         void* ws, size_t ws_bytes, cudaStream_t s);
int dequant_edge_values(const gq_graph* g, const uint8_t* codes, const float* hdr, int heads, float* out,
                        cudaStream_t s);
int gat_edge_bwd(const gq_graph* g, const float* dOut, const float* Hp, const uint8_t* packed, const uint8_t* mask,
                 int bits, const float* alpha, const float* S, const float* D, int heads, int d, float slope,
                 float* dEpre, float* dD, void* ws, size_t ws_bytes, cudaStream_t s);
int gat_node_bwd(const gq_graph* g, const float* dEpre, const float* dD, const float* dM, const float* Hp,
                 const float* a_src, const float* a_dst, int heads, int d, void* dHp_bf16, int64_t ldb, float* dHp32,
                 float* dS, float* da_src, float* da_dst, void* ws, size_t ws_bytes, cudaStream_t s);

}  // namespace gq
