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
//
// The GAT layer (Tango Sec. 2.1, Fig. 1a / 1b) composes the GEMM with head
// projections, the edge softmax, the optional 8-bit attention values (Tango
// Sec. 3.3) and the multi-head SpMM forward; backward, the edge pass, the
// transposed multi-head SpMM on the forward's weights, the node pass and
// the two GEMMs.
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
                                uint16_t* A_save, int64_t lda, float* H_out, int64_t ldo, uint32_t* relu_bits,
                                int64_t ldrb, void* ws, size_t ws_bytes, int* dev_err, void* const* stage_events,
                                gq_stream stream) {
  using namespace gq;
  cudaStream_t s = (cudaStream_t)stream;
  if (g == nullptr || H_in == nullptr || W == nullptr || A_save == nullptr || H_out == nullptr)
    return GQ_ERR_INVALID_ARG;
  if (relu_bits != nullptr && ldrb < (d_out + 31) / 32) return GQ_ERR_INVALID_ARG;
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
                  nullptr, 0, dev_err, s, relu_bits, ldrb));
  return tr.end(2);
}

extern "C" int gq_gcn_layer_bwd(const gq_graph* g, int coef, const float* dH_out, int64_t ldd,
                                const uint16_t* dZ_in, int64_t ldzi, const uint16_t* A_save, int64_t lda,
                                const float* H_out, int64_t ldo, const float* W, int d_in, int d_out,
                                const uint8_t* mask, int bits, uint64_t seed, int act, int need_dinput, float* dW,
                                float* dH_in, int64_t ldi, const uint32_t* gate_in, int64_t ldgi, uint16_t* dZ_prev,
                                int64_t ldzp, float* dA_save, void* ws, size_t ws_bytes, int* dev_err,
                                void* const* stage_events, gq_stream stream) {
  using namespace gq;
  cudaStream_t s = (cudaStream_t)stream;
  if (g == nullptr || A_save == nullptr || W == nullptr || dW == nullptr) return GQ_ERR_INVALID_ARG;
  if (dZ_in == nullptr) {
    if (dH_out == nullptr || ldd < d_out) return GQ_ERR_INVALID_ARG;
    if (act == GQ_ACT_RELU && H_out == nullptr) return GQ_ERR_INVALID_ARG;
  } else if (ldzi < d_out || ldzi % 8 || !aligned(dZ_in, 16)) {
    return GQ_ERR_INVALID_ARG;
  }
  if (d_in < 1 || d_out < 1 || d_in % 4 || lda < d_in || lda % 8) return GQ_ERR_INVALID_ARG;
  if (need_dinput) {
    if (dZ_prev != nullptr) {
      if (ldzp < d_in || ldzp % 8 || !aligned(dZ_prev, 16)) return GQ_ERR_INVALID_ARG;
      if (gate_in != nullptr && (ldgi < (d_in + 31) / 32 || !aligned(gate_in, 4))) return GQ_ERR_INVALID_ARG;
    } else if (dH_in == nullptr || ldi < d_in) {
      return GQ_ERR_INVALID_ARG;
    }
  }
  if (!(bits == 32 || valid_bits(bits))) return GQ_ERR_INVALID_ARG;
  if (d_in > 256 || d_out > 256) return GQ_ERR_UNSUPPORTED;
  GcnWs w;
  if (ws == nullptr || !carve_gcn(g, ws, ws_bytes, d_in, d_out, bits, w).ok()) return GQ_ERR_WORKSPACE;
  const Trace tr{stage_events, s};
  // 1. dZ = dH_out * relu'(Z), with relu'(Z) = [H_out > 0]  (given by the caller as dZ_in, or made here)
  const void* dz = dZ_in != nullptr ? static_cast<const void*>(dZ_in) : w.dz;
  const int64_t ldz = dZ_in != nullptr ? ldzi : round8(d_out);
  GQ_TRY(tr.begin(0));
  if (dZ_in == nullptr)
    GQ_TRY(to_bf16(dH_out, g->n, d_out, ldd, w.dz, ldz, (int)ldz, act == GQ_ACT_RELU ? H_out : nullptr, ldo, s));
  GQ_TRY(tr.end(0));
  // 2. dW = A^T dZ
  GQ_TRY(tr.begin(1));
  GQ_TRY(wgrad_gemm(A_save, g->n, d_in, lda, dz, d_out, ldz, dW, d_out, 0, w.wg, w.wg_bytes, dev_err, s));
  GQ_TRY(tr.end(1));
  if (!need_dinput) return GQ_OK;
  // 3. dA = dZ W^T : B operand is W itself, [d_in][d_out] in bf16
  float* dA = dA_save != nullptr ? dA_save : w.dA;
  const int64_t ldw = round8(d_out);
  GQ_TRY(tr.begin(2));
  GQ_TRY(to_bf16(W, d_in, d_out, d_out, w.wt, ldw, (int)ldw, nullptr, 0, s));
  GQ_TRY(row_gemm(dz, g->n, d_out, ldz, w.wt, d_in, ldw, GQ_ACT_NONE, dA, d_in, nullptr, nullptr, nullptr, nullptr,
                  0, dev_err, s));
  GQ_TRY(tr.end(2));
  // 4-5. quantize the marginal rows of dA, aggregate over the transpose: fp32
  // dH_in, or the previous layer's dZ = bf16(dH_in * relu'), relu' as the gate_in bits
  GQ_TRY(tr.begin(3));
  if (bits < 32) GQ_TRY(quantize_pack(dA, g->n, d_in, d_in, mask, bits, seed, w.packed, s));
  GQ_TRY(tr.end(3));
  GQ_TRY(tr.begin(4));
  if (dZ_prev != nullptr)
    GQ_TRY(dequant_spmm(g, 1, coef, dA, d_in, w.packed, mask, d_in, bits, nullptr, ldzp, w.sp, w.sp_bytes, s,
                        dZ_prev, gate_in, ldgi));
  else
    GQ_TRY(dequant_spmm(g, 1, coef, dA, d_in, w.packed, mask, d_in, bits, dH_in, ldi, w.sp, w.sp_bytes, s, nullptr));
  return tr.end(4);
}

// ---------------------------------------------------------------------------
// GAT layer (Tango Sec. 2.1, Fig. 1a forward, Fig. 1b backward)
// ---------------------------------------------------------------------------
namespace gq {
namespace {

struct GatWs {
  void* hb;          // H in bf16 [n][round8(d_in)]
  void* wb;          // W^T (fwd) or W (bwd) in bf16
  uint8_t* packed;   // quantized H' (fwd, if the caller keeps none) / quantized dOut (bwd)
  void* sx;          // softmax / edge-backward split scratch
  size_t sx_bytes;
  void* sp;          // edge SpMM scratch
  size_t sp_bytes;
  float* dEpre;      // E x heads
  float* dD;         // n x heads
  float* dM;         // n x d
  void* dhb;         // dH' bf16 [n][d]
  void* nb;          // node-kernel partials
  size_t nb_bytes;
  void* wg;          // weight-GEMM partials
  size_t wg_bytes;
  uint8_t* acode;    // 8-bit attention codes E x heads (fwd, if the caller keeps none)
  float* ahdr;       // their {S, Z} per row and head
  float* ahat;       // de-quantized attention values E x heads (bwd)
};

Carve carve_gat(const gq_graph* g, void* ws, size_t ws_bytes, int d_in, int heads, int d, int bits, int alpha_bits,
                GatWs& w) {
  const int64_t n = g->n;
  Carve c(ws, ws_bytes);
  w.hb = c.take((size_t)n * round8(d_in) * 2);
  const int64_t a = (int64_t)d * round8(d_in), b = (int64_t)d_in * round8(d);
  w.wb = c.take((size_t)(a > b ? a : b) * 2);
  w.packed = bits < 32 ? static_cast<uint8_t*>(c.take((size_t)n * packed_pitch(d, bits))) : nullptr;
  const size_t s1 = edge_softmax_workspace(g, heads), s2 = edge_bwd_workspace(g, heads);
  w.sx_bytes = s1 > s2 ? s1 : s2;
  w.sx = w.sx_bytes ? c.take(w.sx_bytes) : nullptr;
  const size_t p0 = spmm_workspace(g, 0, d), p1 = spmm_workspace(g, 1, d);
  w.sp_bytes = p0 > p1 ? p0 : p1;
  w.sp = w.sp_bytes ? c.take(w.sp_bytes) : nullptr;
  w.dEpre = static_cast<float*>(c.take((size_t)g->nnz * heads * sizeof(float)));
  w.dD = static_cast<float*>(c.take((size_t)n * heads * sizeof(float)));
  w.dM = static_cast<float*>(c.take((size_t)n * d * sizeof(float)));
  w.dhb = c.take((size_t)n * d * 2);
  w.nb_bytes = node_bwd_workspace(g, heads, d);
  w.nb = c.take(w.nb_bytes);
  w.wg_bytes = wgrad_workspace(n, d_in, d);
  w.wg = c.take(w.wg_bytes);
  if (alpha_bits == 8) {  // after every other buffer: the rest of the carve is the same either way
    w.acode = static_cast<uint8_t*>(c.take((size_t)g->nnz * heads));
    w.ahdr = static_cast<float*>(c.take((size_t)n * heads * 2 * sizeof(float)));
    w.ahat = static_cast<float*>(c.take((size_t)g->nnz * heads * sizeof(float)));
    // the quantizer's scratch (one pair per head and task) is the softmax's, in sx
  } else {
    w.acode = nullptr;
    w.ahdr = nullptr;
    w.ahat = nullptr;
  }
  return c;
}

int gat_check(const gq_graph* g, int d_in, int heads, int f, int bits) {
  if (g == nullptr || d_in < 1 || heads < 1 || f < 1) return GQ_ERR_INVALID_ARG;
  if (!(bits == 32 || valid_bits(bits))) return GQ_ERR_INVALID_ARG;
  const int d = heads * f;
  if (d_in > 256 || d > 256 || d % 8 || !(heads == 1 || heads == 2 || heads == 4 || heads == 8) || f < 16 ||
      (f & (f - 1)))
    return GQ_ERR_UNSUPPORTED;
  return GQ_OK;
}

}  // namespace
}  // namespace gq

extern "C" size_t gq_gat_layer_workspace_bytes(const gq_graph* g, int d_in, int heads, int f, int bits,
                                               int alpha_bits) {
  if (g == nullptr || d_in < 1 || heads < 1 || f < 1) return 0;
  gq::GatWs w;
  return gq::carve_gat(g, nullptr, 0, d_in, heads, heads * f, bits, alpha_bits, w).used + 256;
}

extern "C" int gq_gat_layer_fwd(const gq_graph* g, const float* H, int64_t ldh, int d_in, const float* W,
                                const float* a_src, const float* a_dst, int heads, int f, float slope,
                                const uint8_t* mask, int bits, uint64_t seed, int alpha_bits, float* Hp_save,
                                float* S_save, float* D_save, float* alpha_save, uint8_t* packed_save,
                                uint8_t* acode_save, float* ahdr_save, float* out, void* ws, size_t ws_bytes,
                                int* dev_err, gq_stream stream) {
  using namespace gq;
  GQ_TRY(gat_check(g, d_in, heads, f, bits));
  if (H == nullptr || W == nullptr || a_src == nullptr || a_dst == nullptr || Hp_save == nullptr ||
      S_save == nullptr || D_save == nullptr || (alpha_save == nullptr && g->nnz > 0) || out == nullptr ||
      ldh < d_in)
    return GQ_ERR_INVALID_ARG;
  // attention codes are kept in both buffers or in neither; with no edges the codes are empty (may be NULL)
  if (!(alpha_bits == 32 || alpha_bits == 8) || (acode_save != nullptr && ahdr_save == nullptr) ||
      (ahdr_save != nullptr && acode_save == nullptr && g->nnz > 0))
    return GQ_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int d = heads * f;
  GatWs w;
  if (ws == nullptr || !carve_gat(g, ws, ws_bytes, d_in, heads, d, bits, alpha_bits, w).ok())
    return GQ_ERR_WORKSPACE;
  const int64_t ldhb = round8(d_in);
  // step 1: H' = H W ; step 2: S = H' a_src, D = H' a_dst (GEMM epilogue)
  GQ_TRY(to_bf16(H, g->n, d_in, ldh, w.hb, ldhb, (int)ldhb, nullptr, 0, s));
  GQ_TRY(transpose_bf16(W, d_in, d, d, w.wb, ldhb, (int)ldhb, s));
  GQ_TRY(row_gemm(w.hb, g->n, d_in, ldhb, w.wb, d, ldhb, GQ_ACT_NONE, Hp_save, d, a_src, a_dst, S_save, D_save,
                  heads, dev_err, s));
  // optional quantization of the messages H' of marginal nodes
  uint8_t* packed = nullptr;
  if (bits < 32) {
    packed = packed_save != nullptr ? packed_save : w.packed;
    GQ_TRY(quantize_pack(Hp_save, g->n, d, d, mask, bits, seed, packed, s));
  }
  // steps 3-4: SDDMM add + LeakyReLU + edge softmax ; step 5: SpMM
  GQ_TRY(edge_softmax(g, S_save, D_save, heads, slope, nullptr, alpha_save, w.sx, w.sx_bytes, s));
  if (alpha_bits == 8) {
    // the SpMM reads the attention values as 8-bit codes (Tango Sec. 3.3)
    uint8_t* acode = acode_save != nullptr ? acode_save : w.acode;
    float* ahdr = ahdr_save != nullptr ? ahdr_save : w.ahdr;
    GQ_TRY(quantize_edge_values(g, alpha_save, heads, seed ^ GQ_ALPHA_SEED_TAG, acode, ahdr, w.sx, w.sx_bytes, s));
    return edge_spmm_alpha8(g, acode, ahdr, heads, Hp_save, d, packed, mask, d, bits, out, d, w.sp, w.sp_bytes, s);
  }
  return edge_spmm(g, 0, alpha_save, heads, Hp_save, d, packed, mask, d, bits, out, d, w.sp, w.sp_bytes, s);
}

extern "C" int gq_gat_layer_bwd(const gq_graph* g, const float* dOut, const float* H, int64_t ldh,
                                const float* Hp_save, const float* S_save, const float* D_save,
                                const float* alpha_save, const uint8_t* packed_save, const uint8_t* acode_save,
                                const float* ahdr_save, const float* W, const float* a_src, const float* a_dst,
                                int d_in, int heads, int f, float slope, const uint8_t* mask, int bits,
                                uint64_t seed, float* dW, float* da_src, float* da_dst, float* dH,
                                float* dEpre_save, float* dHp_save, void* ws, size_t ws_bytes, int* dev_err,
                                gq_stream stream) {
  using namespace gq;
  GQ_TRY(gat_check(g, d_in, heads, f, bits));
  if (dOut == nullptr || H == nullptr || Hp_save == nullptr || S_save == nullptr || D_save == nullptr ||
      (alpha_save == nullptr && g->nnz > 0) || W == nullptr || a_src == nullptr || a_dst == nullptr || dW == nullptr ||
      da_src == nullptr || da_dst == nullptr || dH == nullptr || ldh < d_in)
    return GQ_ERR_INVALID_ARG;
  if (bits < 32 && packed_save == nullptr) return GQ_ERR_INVALID_ARG;
  if ((acode_save != nullptr && ahdr_save == nullptr) || (ahdr_save != nullptr && acode_save == nullptr && g->nnz > 0))
    return GQ_ERR_INVALID_ARG;
  const int alpha_bits = ahdr_save != nullptr ? 8 : 32;
  cudaStream_t s = (cudaStream_t)stream;
  const int d = heads * f;
  GatWs w;
  if (ws == nullptr || !carve_gat(g, ws, ws_bytes, d_in, heads, d, bits, alpha_bits, w).ok())
    return GQ_ERR_WORKSPACE;
  float* dEpre = dEpre_save != nullptr ? dEpre_save : w.dEpre;
  // SDDMM dot -> dalpha; softmax derivative; LeakyReLU'; dD = in-edge sums
  GQ_TRY(gat_edge_bwd(g, dOut, Hp_save, packed_save, mask, bits, alpha_save, S_save, D_save, heads, d, slope, dEpre,
                      w.dD, w.sx, w.sx_bytes, s));
  // dM = transposed multi-head SpMM of dOut (marginal rows travel quantized)
  // with 8-bit attention codes the forward multiplied by their values, so
  // the transposed SpMM does too
  if (bits < 32) GQ_TRY(quantize_pack(dOut, g->n, d, d, mask, bits, seed, w.packed, s));
  const float* aT = alpha_save;
  if (alpha_bits == 8) {
    GQ_TRY(dequant_edge_values(g, acode_save, ahdr_save, heads, w.ahat, s));
    aT = w.ahat;
  }
  GQ_TRY(edge_spmm(g, 1, aT, heads, dOut, d, w.packed, mask, d, bits, w.dM, d, w.sp, w.sp_bytes, s));
  // dS = out-edge sums; dH' = dM + dS a_src + dD a_dst; da_src, da_dst
  GQ_TRY(gat_node_bwd(g, dEpre, w.dD, w.dM, Hp_save, a_src, a_dst, heads, d, w.dhb, d, dHp_save, nullptr, da_src,
                      da_dst, w.nb, w.nb_bytes, s));
  // dW = H^T dH' ; dH = dH' W^T
  const int64_t ldhb = round8(d_in);
  GQ_TRY(to_bf16(H, g->n, d_in, ldh, w.hb, ldhb, (int)ldhb, nullptr, 0, s));
  GQ_TRY(wgrad_gemm(w.hb, g->n, d_in, ldhb, w.dhb, d, d, dW, d, 0, w.wg, w.wg_bytes, dev_err, s));
  GQ_TRY(to_bf16(W, d_in, d, d, w.wb, round8(d), (int)round8(d), nullptr, 0, s));
  return row_gemm(w.dhb, g->n, d, d, w.wb, d_in, round8(d), GQ_ACT_NONE, dH, d_in, nullptr, nullptr, nullptr,
                  nullptr, 0, dev_err, s);
}
