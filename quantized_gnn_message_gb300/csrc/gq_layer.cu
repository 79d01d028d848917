// gq_layer.cu -- one GCN / GraphSAGE-mean layer, forward and backward,
// composed from the library's kernels on one stream.
//
// Forward (AdaQP Sec. 2.1 weighted-sum form, Sec. 3.1 mixed messages;
// Sancus Sec. 2 H' = sigma(A^ H W)):
//   1. quantize_pack(H_in rows of marginal nodes)            (Eqn 4)
//   2. A = sum_u a_uv m_u, de-quantization fused (Eqn 5)     -> A_save (bf16)
//   3. H_out = act(A W) on tcgen05, activation in the epilogue
// Backward (the same layer read in reverse; AdaQP Sec. 2.3 and Sec. 3:
// embedding gradients are the messages that travel quantized backward):
//   1. dZ = dH_out * act'(.)  (ReLU' read from H_out > 0)    -> bf16
//   2. dW = A^T dZ            (split over rows, fixed-order reduction)
//   3. dA = dZ W^T            (tcgen05)                       -> fp32
//   4. quantize_pack(dA rows of marginal nodes)
//   5. dH_in = A^T-aggregation of the mixed messages (transposed CSR)
// The quantizer is treated as the identity in backward (straight-through):
// its codes are constants of the forward pass.
#include <cuda_bf16.h>

#include "gq_common.cuh"
#include "gq_internal.cuh"

namespace gq {
namespace {

// Optional stage tracing: events[2k] is recorded before stage k and
// events[2k+1] after it, on the call's stream.
struct Trace {
  void* const* ev;
  cudaStream_t s;
  int begin(int k) const { return ev ? (cudaEventRecord((cudaEvent_t)ev[2 * k], s) == cudaSuccess ? GQ_OK : GQ_ERR_CUDA) : GQ_OK; }
  int end(int k) const { return ev ? (cudaEventRecord((cudaEvent_t)ev[2 * k + 1], s) == cudaSuccess ? GQ_OK : GQ_ERR_CUDA) : GQ_OK; }
};

struct GcnWs {
  uint8_t* packed;
  void* wt;        // fwd: W^T bf16 [d_out][round8(d_in)]; bwd: W bf16 [d_in][round8(d_out)]
  void* dz;        // bwd: dZ bf16 [n][round8(d_out)]
  float* dA;       // bwd: dA fp32 [n][d_in]
  void* wg;        // bwd: weight-GEMM partials
  size_t wg_bytes;
  void* sp;        // aggregation scratch (split heavy rows)
  size_t sp_bytes;
};

// Carves the layer workspace; with ws == nullptr it only measures (c.used).
Carve carve_gcn(const gq_graph* g, void* ws, size_t ws_bytes, int d_in, int d_out, int bits, GcnWs& w) {
  const int64_t n = g->n;
  Carve c(ws, ws_bytes);
  w.packed = bits < 32 ? static_cast<uint8_t*>(c.take((size_t)n * packed_pitch(d_in, bits))) : nullptr;
  const int64_t wt_elems = (int64_t)d_out * round8(d_in) > (int64_t)d_in * round8(d_out)
                               ? (int64_t)d_out * round8(d_in)
                               : (int64_t)d_in * round8(d_out);
  w.wt = c.take((size_t)wt_elems * 2);
  w.dz = c.take((size_t)n * round8(d_out) * 2);
  w.dA = static_cast<float*>(c.take((size_t)n * d_in * sizeof(float)));
  w.wg_bytes = wgrad_workspace(n, d_in, d_out);
  w.wg = c.take(w.wg_bytes);
  const size_t a = spmm_workspace(g, 0, d_in), b = spmm_workspace(g, 1, d_in);
  w.sp_bytes = a > b ? a : b;
  w.sp = w.sp_bytes ? c.take(w.sp_bytes) : nullptr;
  return c;
}

}  // namespace
}  // namespace gq

extern "C" size_t gq_gcn_layer_workspace_bytes(const gq_graph* g, int d_in, int d_out, int bits) {
  if (g == nullptr || d_in < 1 || d_out < 1) return 0;
  gq::GcnWs w;
  return gq::carve_gcn(g, nullptr, 0, d_in, d_out, bits, w).used + 256;
}

extern "C" int gq_gcn_layer_fwd(const gq_graph* g, int coef, const float* H_in, int64_t ldh, int d_in,
                                const float* W, int d_out, const uint8_t* mask, int bits, uint64_t seed, int act,
                                uint16_t* A_save, int64_t lda, float* H_out, int64_t ldo, void* ws,
                                size_t ws_bytes, int* dev_err, void* const* stage_events, gq_stream stream) {
  using namespace gq;
  cudaStream_t s = (cudaStream_t)stream;
  if (g == nullptr || H_in == nullptr || W == nullptr || A_save == nullptr || H_out == nullptr)
    return GQ_ERR_INVALID_ARG;
  if (d_in < 1 || d_out < 1 || d_in % 4 || lda < d_in || lda % 8 || ldo < d_out || ldh < d_in)
    return GQ_ERR_INVALID_ARG;
  if (!(bits == 32 || valid_bits(bits))) return GQ_ERR_INVALID_ARG;
  if (d_in > 256 || d_out > 256) return GQ_ERR_UNSUPPORTED;
  GcnWs w;
  if (ws == nullptr || !carve_gcn(g, ws, ws_bytes, d_in, d_out, bits, w).ok()) return GQ_ERR_WORKSPACE;
  const Trace tr{stage_events, s};
  GQ_TRY(tr.begin(0));
  if (bits < 32) GQ_TRY(quantize_pack(H_in, g->n, d_in, ldh, mask, bits, seed, w.packed, s));
  GQ_TRY(tr.end(0));
  GQ_TRY(tr.begin(1));
  GQ_TRY(dequant_spmm(g, 0, coef, H_in, ldh, w.packed, mask, d_in, bits, nullptr, lda, w.sp, w.sp_bytes, s, A_save));
  GQ_TRY(tr.end(1));
  GQ_TRY(tr.begin(2));
  GQ_TRY(transpose_bf16(W, d_in, d_out, d_out, w.wt, round8(d_in), (int)round8(d_in), s));
  GQ_TRY(row_gemm(A_save, g->n, d_in, lda, w.wt, d_out, round8(d_in), act, H_out, ldo, nullptr, nullptr, nullptr,
                  nullptr, 0, dev_err, s));
  return tr.end(2);
}

extern "C" int gq_gcn_layer_bwd(const gq_graph* g, int coef, const float* dH_out, int64_t ldd,
                                const uint16_t* A_save, int64_t lda, const float* H_out, int64_t ldo,
                                const float* W, int d_in, int d_out, const uint8_t* mask, int bits, uint64_t seed,
                                int act, int need_dinput, float* dW, float* dH_in, int64_t ldi, float* dA_save,
                                void* ws, size_t ws_bytes, int* dev_err, void* const* stage_events,
                                gq_stream stream) {
  using namespace gq;
  cudaStream_t s = (cudaStream_t)stream;
  if (g == nullptr || dH_out == nullptr || A_save == nullptr || W == nullptr || dW == nullptr)
    return GQ_ERR_INVALID_ARG;
  if (act == GQ_ACT_RELU && H_out == nullptr) return GQ_ERR_INVALID_ARG;
  if (d_in < 1 || d_out < 1 || d_in % 4 || lda < d_in || lda % 8 || ldd < d_out) return GQ_ERR_INVALID_ARG;
  if (need_dinput && (dH_in == nullptr || ldi < d_in)) return GQ_ERR_INVALID_ARG;
  if (!(bits == 32 || valid_bits(bits))) return GQ_ERR_INVALID_ARG;
  if (d_in > 256 || d_out > 256) return GQ_ERR_UNSUPPORTED;
  GcnWs w;
  if (ws == nullptr || !carve_gcn(g, ws, ws_bytes, d_in, d_out, bits, w).ok()) return GQ_ERR_WORKSPACE;
  const Trace tr{stage_events, s};
  const int64_t ldz = round8(d_out);
  // 1. dZ = dH_out * relu'(Z), with relu'(Z) = [H_out > 0]
  GQ_TRY(tr.begin(0));
  GQ_TRY(to_bf16(dH_out, g->n, d_out, ldd, w.dz, ldz, (int)ldz, act == GQ_ACT_RELU ? H_out : nullptr, ldo, s));
  GQ_TRY(tr.end(0));
  // 2. dW = A^T dZ
  GQ_TRY(tr.begin(1));
  GQ_TRY(wgrad_gemm(A_save, g->n, d_in, lda, w.dz, d_out, ldz, dW, d_out, 0, w.wg, w.wg_bytes, dev_err, s));
  GQ_TRY(tr.end(1));
  if (!need_dinput) return GQ_OK;
  // 3. dA = dZ W^T : B operand is W itself, [d_in][d_out] in bf16
  float* dA = dA_save != nullptr ? dA_save : w.dA;
  GQ_TRY(tr.begin(2));
  GQ_TRY(to_bf16(W, d_in, d_out, d_out, w.wt, ldz, (int)ldz, nullptr, 0, s));
  GQ_TRY(row_gemm(w.dz, g->n, d_out, ldz, w.wt, d_in, ldz, GQ_ACT_NONE, dA, d_in, nullptr, nullptr, nullptr,
                  nullptr, 0, dev_err, s));
  GQ_TRY(tr.end(2));
  // 4-5. quantize the marginal rows of dA, aggregate over the transpose
  GQ_TRY(tr.begin(3));
  if (bits < 32) GQ_TRY(quantize_pack(dA, g->n, d_in, d_in, mask, bits, seed, w.packed, s));
  GQ_TRY(tr.end(3));
  GQ_TRY(tr.begin(4));
  GQ_TRY(dequant_spmm(g, 1, coef, dA, d_in, w.packed, mask, d_in, bits, dH_in, ldi, w.sp, w.sp_bytes, s, nullptr));
  return tr.end(4);
}
