/*
 * gq.h -- C ABI of libgq: quantized message passing for full-graph GNN
 * training on one NVIDIA GB300 (sm_103a).
 *
 * What the library computes (each entry point cites its passage):
 *   AdaQP, "Adaptive Message Quantization and Parallelization for Distributed
 *   Full-graph GNN Training" (arXiv 2306.01381):
 *     Sec. 2.1  a layer is aggregation then update, written as a weighted sum
 *               h_v = sigma(W * sum_{u in {v} U N(v)} a_{u,v} h_u)
 *     Sec. 2.3  Eqn 4: b-bit stochastic integer quantization of a message row,
 *               Z = min(h), S = (max(h) - min(h)) / (2^b - 1),
 *               q = round_st((h - Z) / S), b in {2, 4, 8};
 *               Eqn 5: de-quantization h^ = q * S + Z
 *     Sec. 3.1  only the messages of "marginal" nodes travel quantized; the
 *               others are aggregated in full precision
 *   Sancus (IJCAI 2023, extended abstract), Sec. 2 Preliminaries:
 *               A^ = D~^{-1/2} (A + I) D~^{-1/2},  H' = sigma(A^ H W)
 *     Sec. 3.2 / 4.2  a bit-width per message; Problem 11's per-message
 *               variance weight beta_k
 *   Tango, "Rethinking quantization for graph neural network training on
 *   GPUs" (arXiv 2308.00890), Sec. 2.1, Fig. 1: GAT forward as GEMM, head
 *   projections, SDDMM add, LeakyReLU, edge softmax, SpMM; and its backward.
 *     Sec. 3.2  Eq. 4: relative quantization error Error_X and the bit rule
 *     Sec. 3.3  the SPMM reads quantized node and edge features
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers owned by the caller unless a parameter
 *     says "host".  The library allocates no device memory: scratch comes
 *     from a caller buffer sized by the matching *_workspace_bytes query.
 *     The one exception is gq_dequant_spmm_noalloc, whose scratch is a
 *     fixed array compiled into the library (see there).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and performs no host<->device copy and no
 *     synchronization, except gq_graph_prepare, which synchronizes `stream`
 *     once (documented there).
 *   - Matrices are row-major with a leading dimension (row pitch) counted in
 *     elements.  fp32 matrices read or written with vector accesses must be
 *     16-byte aligned with a leading dimension that is a multiple of 4.
 *   - Graphs are CSR by DESTINATION: row v lists the sources u of the edges
 *     u -> v, in ascending order, int32.  Every node should carry its own
 *     self-loop (the "+ I" of A + I); the library does not add one.  On a
 *     graph without edges, per-edge buffers (col, alpha, E_pre, attention
 *     codes) are empty and may be NULL.
 *   - Errors: every call returns a gq_status.  Arguments are checked on the
 *     host before any launch; a failed check launches nothing.  A CUDA launch
 *     error is reported as GQ_ERR_CUDA.  No kernel traps or asserts.
 *   - Thread safety: no global mutable host state; calls on different
 *     streams may run concurrently if their buffers do not overlap, except
 *     gq_dequant_spmm_noalloc, whose calls share one device array and must
 *     not overlap on the GPU.
 */
#ifndef GQ_H
#define GQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GQ_API __attribute__((visibility("default")))
#else
#define GQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gq_stream; /* == cudaStream_t */

typedef enum {
  GQ_OK = 0,
  GQ_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bits, alignment      */
  GQ_ERR_UNSUPPORTED = 2,  /* valid but not supported (e.g. width too big) */
  GQ_ERR_BAD_GRAPH = 3,    /* CSR fails validation in gq_graph_prepare     */
  GQ_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
  GQ_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up           */
  GQ_ERR_WORKSPACE = 6,    /* workspace or storage buffer too small        */
  GQ_ERR_SCRATCH_LIMIT = 7 /* request exceeds the fixed scratch of
                              gq_dequant_spmm_noalloc                      */
} gq_status;

/* Aggregation coefficient a_{u,v} of an edge u -> v. */
typedef enum {
  GQ_COEF_GCN = 0,  /* 1/sqrt(deg_in(v) * deg_out(u)), degrees incl. self-loop
                       (Sancus Sec. 2; for a symmetric graph this is exactly
                       D~^{-1/2}(A+I)D~^{-1/2})                               */
  GQ_COEF_SAGE = 1, /* 1/deg_in(v): mean over {v} U N(v) (AdaQP Sec. 2.1)    */
  GQ_COEF_ONE = 2   /* 1: plain sum                                          */
} gq_coef;

typedef enum { GQ_ACT_NONE = 0, GQ_ACT_RELU = 1 } gq_act;

/* Human-readable text of a status code (static storage, never NULL). */
GQ_API const char* gq_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
GQ_API int gq_version(void);

/* sizeof(gq_graph) as compiled into the library (lets bindings that mirror
 * the struct check their layout). */
GQ_API size_t gq_graph_struct_bytes(void);

/* ------------------------------------------------------------------------
 * Packed message rows (AdaQP Sec. 2.3, Eqn 4).  One row of the packed
 * buffer holds one quantized message vector of width d at b bits:
 *   bytes [0, ceil(d*b/8))  codes q_j, LSB-first: code j occupies bits
 *                           [(j*b) mod 8, +b) of byte floor(j*b/8)
 *   bytes up to H           zero, H = gq_packed_header_offset(d, b)
 *                           (payload rounded up to a multiple of 8)
 *   bytes [H, H+4)          S, the scale, little-endian fp32
 *   bytes [H+4, H+8)        Z = min of the row, little-endian fp32
 *   bytes up to the pitch   zero; pitch = gq_packed_pitch(d, b), a multiple
 *                           of 16, so every row starts 16-byte aligned.
 * Row r of the buffer belongs to node r.  Returns -1 for invalid d / bits.
 * ---------------------------------------------------------------------- */
GQ_API int64_t gq_packed_pitch(int d, int bits);
GQ_API int64_t gq_packed_header_offset(int d, int bits);

/* ------------------------------------------------------------------------
 * gq_quantize_pack -- AdaQP Sec. 2.3, Eqn 4, for every row r with
 * mask[r] != 0 (every row when mask == NULL):
 *   Z = min_j X[r,j];  S = (max_j X[r,j] - Z) / (2^b - 1)   (fp32 division)
 *   u = (fmix32(fmix32(r ^ fmix32(s)) + j * 0x9E3779B9) >> 9) * 2^-23, with
 *       s = low32(seed) ^ high32(seed) and fmix32 MurmurHash3's finalizer
 *   q = min(floor((X[r,j] - Z) * (1/S) + u), 2^b - 1)  (fp32, each op
 *       rounded to nearest, no fused multiply-add); q = 0 for every
 *       element when S is below the smallest normal fp32 (a constant row).
 * Rows must be finite with max - min finite; other rows give unspecified
 * codes (no fault).
 * The result is bit-for-bit reproducible.  Rows with mask[r] == 0 are not
 * written.
 *   X       n x d fp32, leading dimension ldx >= d
 *   mask    n bytes or NULL
 *   bits    2, 4 or 8
 *   packed  n x gq_packed_pitch(d, bits) bytes, 16-byte aligned
 * Errors: GQ_ERR_INVALID_ARG for null X/packed, n < 0, d < 1, ldx < d,
 * bits not in {2,4,8}, a misaligned packed buffer; GQ_ERR_UNSUPPORTED for
 * d > 16384.
 * ---------------------------------------------------------------------- */
GQ_API int gq_quantize_pack(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* mask, int bits,
                     uint64_t seed, uint8_t* packed, gq_stream stream);

/* gq_dequant_unpack -- AdaQP Sec. 2.3, Eqn 5: Y[r,j] = fmaf(q_j, S, Z) for
 * every row with mask[r] != 0 (all rows when mask == NULL); other rows of Y
 * are not written.  Y is n x d fp32 with leading dimension ldy >= d.       */
GQ_API int gq_dequant_unpack(const uint8_t* packed, int64_t n, int d, int bits, const uint8_t* mask,
                      float* Y, int64_t ldy, gq_stream stream);

/* ------------------------------------------------------------------------
 * Prepared graph.  gq_graph_prepare derives from the caller's CSR the
 * transposed CSR (CSC: row u lists the destinations v of the edges u -> v,
 * ascending, with tr_perm giving each entry's edge id in the CSR), the
 * degree normalizations, and, for each direction, a static schedule of the
 * "heavy" rows (degree > hub_threshold): each is one thread-block task, or
 * several tasks of at most split_edges edges whose partial rows are summed
 * in task order (a split group).  Light rows are one warp each.
 * All arrays live in the caller's `storage` buffer.
 * ---------------------------------------------------------------------- */
typedef struct gq_sched {
  const int32_t* tasks;     /* n_tasks x {row, e_begin, e_end, group}; group
                               = index into groups, or -1 (unsplit row)   */
  const int32_t* groups;    /* n_groups x {row, first_task, n_tasks,
                               first_slot}: the group's tasks write their
                               partial rows to workspace slots
                               first_slot .. first_slot + n_tasks - 1    */
  int64_t n_tasks;
  int64_t n_groups;
  int64_t n_slots;          /* partial-row slots over all groups          */
  const int32_t* light;     /* n_light x {row_begin, row_end}: runs of
                               consecutive light rows with at most 256
                               edges in all, or one light row (heavy rows
                               never inside), covering every light row
                               once                                       */
  int64_t n_light;
} gq_sched;

typedef struct gq_graph {
  int64_t n;                /* nodes                                      */
  int64_t nnz;              /* edges, self-loops included                 */
  const int32_t* rowptr;    /* n+1, caller's CSR (destinations)           */
  const int32_t* col;       /* nnz                                        */
  int32_t* tr_rowptr;       /* n+1, CSC (sources)                         */
  int32_t* tr_col;          /* nnz: destination of each CSC entry         */
  int32_t* tr_perm;         /* nnz: CSR edge id of each CSC entry         */
  float* dinv_in;           /* n: 1/sqrt(deg_in)  (0 if deg 0)            */
  float* dinv_out;          /* n: 1/sqrt(deg_out)                         */
  float* inv_in;            /* n: 1/deg_in                                */
  gq_sched sched;           /* heavy rows of the CSR                      */
  gq_sched tr_sched;        /* heavy rows of the CSC                      */
  int32_t hub_threshold;    /* rows with more edges are heavy             */
  int32_t split_edges;      /* heavy rows are cut into tasks of this size */
  int32_t max_deg;          /* largest in-degree                          */
  int32_t tr_max_deg;       /* largest out-degree                         */
  int32_t* status;          /* device int in `storage`, zeroed by
                               gq_graph_prepare: an aggregation kernel on
                               this graph whose bounded wait for its own
                               row copies gave up writes a non-zero code
                               here (first writer wins; it stays set);
                               the attention-value kernels write 0x4551
                               for a row or task whose edge range lies
                               outside the graph (and skip it).
                               Read it after synchronizing the stream.  */
} gq_graph;

/* Bytes of `storage` gq_graph_prepare needs for a graph of n nodes and nnz
 * edges (all derived arrays, 256-byte aligned sub-buffers).               */
GQ_API size_t gq_graph_storage_bytes(int64_t n, int64_t nnz);
/* Bytes of scratch gq_graph_prepare needs (free again when it returns).   */
GQ_API size_t gq_graph_prepare_workspace_bytes(int64_t n, int64_t nnz);

/* gq_graph_prepare -- validates the CSR (rowptr[0] == 0, non-decreasing,
 * rowptr[n] == nnz, 0 <= col < n) and fills *g (a HOST struct) with device
 * pointers into `storage`.  Degrees count every CSR entry, so with the
 * self-loops present they are the D~ = D + I of Sancus Sec. 2.  The norms
 * are (float)(1.0 / sqrt((double)deg)) and (float)(1.0 / (double)deg),
 * each rounded once.  The CSC is the stable transpose: entries of a CSC
 * row are in increasing destination order.
 * hub_threshold (>= 32; <= 0 selects 256) and split_edges (>= 256; <= 0
 * selects 4096) shape the heavy-row schedule; heavier tasks come first.
 * Synchronizes `stream` and copies the (small) heavy-row lists through
 * host memory once per direction.
 * Errors: GQ_ERR_INVALID_ARG (null pointers, n < 1, nnz < 0 or nnz >= 2^31,
 * hub_threshold or split_edges out of range), GQ_ERR_WORKSPACE (storage or
 * ws too small), GQ_ERR_BAD_GRAPH, GQ_ERR_CUDA.                           */
GQ_API int gq_graph_prepare(int64_t n, int64_t nnz, const int32_t* rowptr, const int32_t* col,
                     int hub_threshold, int split_edges, void* storage, size_t storage_bytes,
                     void* ws, size_t ws_bytes, gq_graph* g, gq_stream stream);

/* ------------------------------------------------------------------------
 * gq_dequant_spmm -- the aggregation of AdaQP Sec. 2.1 / Sancus Sec. 2 with
 * de-quantization (AdaQP Eqn 5) fused into the gather, mixing quantized and
 * full-precision rows as AdaQP Sec. 3.1 does:
 *   transpose == 0:  Y[v,:] = sum_{e = (u -> v)} a_{u,v} m_u
 *   transpose == 1:  Y[u,:] = sum_{e = (u -> v)} a_{u,v} m_v     (= A^T M)
 * where the message row m_x = deq(packed row x) if bits < 32 and
 * (mask == NULL or mask[x] != 0), and m_x = X[x,:] otherwise.
 *   coef        gq_coef
 *   X           n x d fp32 (ldx), may be NULL only when every row is read
 *               from `packed` (bits < 32 and mask == NULL)
 *   packed      n x gq_packed_pitch(d, bits) bytes (ignored for bits == 32)
 *   bits        2, 4, 8, or 32 (no quantization)
 *   Y           n x d fp32 (ldy); every row is written
 *   ws          gq_spmm_workspace_bytes(g, transpose, d) bytes of scratch
 *               (partial rows of split heavy rows); may be NULL when that
 *               size is 0.  Calls sharing one workspace must not overlap.
 * Sums run in fp32 in a fixed order (deterministic run to run).
 * Errors: GQ_ERR_INVALID_ARG (null or misaligned pointers, d % 4 != 0 for
 * an fp32 operand, bad bits/coef); GQ_ERR_UNSUPPORTED for d > 1024;
 * GQ_ERR_WORKSPACE.                                                       */
GQ_API size_t gq_spmm_workspace_bytes(const gq_graph* g, int transpose, int d);
GQ_API int gq_dequant_spmm(const gq_graph* g, int transpose, int coef, const float* X, int64_t ldx,
                    const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y,
                    int64_t ldy, void* ws, size_t ws_bytes, gq_stream stream);

/* ------------------------------------------------------------------------
 * Mixed bit-widths per row -- AdaQP Sec. 3.2 / 4.2 assign a bit-width to
 * every message (or group of messages); the uniform-sampling ablation
 * (Sec. 5.3) draws it per message from {2, 4, 8}.  A mixed packed buffer
 * holds row r at byte roff[r], in the packed-row layout of its own width
 * rbits[r] (pitch gq_packed_pitch(d, rbits[r])); rows whose width is not 2,
 * 4 or 8 (e.g. 0) are full-precision rows and take no bytes.
 *
 * gq_packed_row_offsets -- roff[0..n] (n+1 int64, device) from rbits (n
 * uint8, device): roff[r] = sum_{i<r} size of row i; roff[n] is the buffer
 * size.  ws: gq_packed_row_offsets_workspace_bytes(n) bytes, 8-byte aligned.
 * gq_quantize_pack_mixed -- AdaQP Eqn 4 on every row with width 2, 4 or 8,
 * each at its own width; row r's bytes equal gq_quantize_pack's row r at
 * that width and seed.  packed: roff[n] bytes, 16-byte aligned.
 * gq_dequant_spmm_mixed -- gq_dequant_spmm over such a buffer (each packed
 * row de-quantized at its own width, other rows read from X); d <= 256
 * (GQ_ERR_UNSUPPORTED otherwise), d % 4 == 0.  Workspace:
 * gq_spmm_workspace_bytes.
 * Errors: as gq_quantize_pack / gq_dequant_spmm.
 * ---------------------------------------------------------------------- */
GQ_API size_t gq_packed_row_offsets_workspace_bytes(int64_t n);
GQ_API int gq_packed_row_offsets(const uint8_t* rbits, int64_t n, int d, int64_t* roff, void* ws,
                                 size_t ws_bytes, gq_stream stream);
GQ_API int gq_quantize_pack_mixed(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* rbits,
                                  const int64_t* roff, uint64_t seed, uint8_t* packed, gq_stream stream);
GQ_API int gq_dequant_spmm_mixed(const gq_graph* g, int transpose, int coef, const float* X, int64_t ldx,
                                 const uint8_t* packed, const int64_t* roff, const uint8_t* rbits, int d,
                                 float* Y, int64_t ldy, void* ws, size_t ws_bytes, gq_stream stream);

/* ------------------------------------------------------------------------
 * gq_edge_spmm -- multi-head attention aggregation (Tango Sec. 2.1, Fig. 1a
 * step 5, H^(l) = (G (.) alpha) H'), all heads in one pass, with the same
 * quantized / full-precision message mix as gq_dequant_spmm:
 *   transpose == 0:  Y[v, kF+f] = sum_{e=(u->v)} alpha[e,k] m_u[kF+f]
 *   transpose == 1:  Y[u, kF+f] = sum_{e=(u->v)} alpha[e,k] m_v[kF+f]
 *                    (the backward pass of step 5, Fig. 1b)
 * with F = d / heads; edge e is the CSR edge id (alpha is E x heads fp32,
 * row-major, indexed by CSR edge id in both directions).
 * Errors: as gq_dequant_spmm, plus GQ_ERR_INVALID_ARG when heads does not
 * divide d and GQ_ERR_UNSUPPORTED unless F is a power of two >= 16.
 * Workspace: as gq_dequant_spmm.                                          */
GQ_API int gq_edge_spmm(const gq_graph* g, int transpose, const float* alpha, int heads, const float* X,
                 int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d, int bits,
                 float* Y, int64_t ldy, void* ws, size_t ws_bytes, gq_stream stream);


/* ------------------------------------------------------------------------
 * 8-bit attention values for the multi-head SpMM (Tango Sec. 3.3: the SpMM
 * reads quantized node and edge features, produced by a separate sequential
 * quantization pass).  Each (destination v, head k) segment of alpha, i.e.
 * alpha[e,k] for the CSR edges e = rowptr[v] .. rowptr[v+1]-1, is one
 * vector quantized as in gq_quantize_pack with b = 8 (its own Z = min and
 * S = (max - Z)/255, the same fp32 steps), except that u is hashed from
 * (seed, e, k) in place of (seed, row, column):
 *   codes  E x heads uint8, by CSR edge id (16-byte aligned)
 *   hdr    n x heads x {S, Z} fp32 (16-byte aligned); {0, 0} for a row
 *          without edges.
 * Values must be finite.  Bit-for-bit reproducible.  Each row and task
 * range is checked against the graph before use; an invalid one is skipped
 * and recorded in the graph's status word (0x4551).
 *
 * gq_quantize_edge_values: alpha (E x heads fp32, 16-byte aligned) ->
 *   codes, hdr.  heads in {1, 2, 4, 8} (GQ_ERR_UNSUPPORTED otherwise).
 *   Workspace: gq_quantize_edge_values_workspace_bytes (split heavy rows
 *   only; may be 0; 256-byte aligned).
 * gq_dequant_edge_values: out[e,k] = fmaf(codes[e,k], S[v,k], Z[v,k])
 *   (AdaQP Eqn 5), E x heads fp32, 16-byte aligned.
 * gq_edge_spmm_alpha8: gq_edge_spmm with transpose == 0 whose weights are
 *   the de-quantized codes (each computed as in gq_dequant_edge_values);
 *   d <= 256 (GQ_ERR_UNSUPPORTED otherwise); other arguments, errors and
 *   workspace as gq_edge_spmm.
 * GQ_ALPHA_SEED_TAG: the GAT layer quantizes its attention values with
 *   seed ^ GQ_ALPHA_SEED_TAG, so their noise is independent of the
 *   messages' noise drawn with the same seed.
 * ---------------------------------------------------------------------- */
#define GQ_ALPHA_SEED_TAG 0x5851F42D4C957F2DULL
GQ_API size_t gq_quantize_edge_values_workspace_bytes(const gq_graph* g, int heads);
GQ_API int gq_quantize_edge_values(const gq_graph* g, const float* alpha, int heads, uint64_t seed,
                                   uint8_t* codes, float* hdr, void* ws, size_t ws_bytes, gq_stream stream);
GQ_API int gq_dequant_edge_values(const gq_graph* g, const uint8_t* codes, const float* hdr, int heads,
                                  float* out, gq_stream stream);
GQ_API int gq_edge_spmm_alpha8(const gq_graph* g, const uint8_t* codes, const float* hdr, int heads,
                               const float* X, int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d,
                               int bits, float* Y, int64_t ldy, void* ws, size_t ws_bytes, gq_stream stream);

/* ------------------------------------------------------------------------
 * Dense update GEMMs on the tcgen05 tensor cores (bf16 inputs, fp32
 * accumulation in tensor memory).  AdaQP Sec. 2.1 (update W h), Tango
 * Sec. 2.1 step 1 (H' = H W) and their backward products.
 * bf16 matrices are read with TMA: 16-byte aligned base, leading dimension a
 * multiple of 8 elements.  `dev_err` (nullable) is a device int that a
 * kernel sets to a non-zero code if a bounded internal wait gave up; read
 * it after synchronizing (0 = fine).
 *
 * gq_gemm_bf16_nt: C[M x N] = act(A[M x K] * B[N x K]^T), i.e. C = A W with
 *   B = W^T stored row-major.  K <= 256, N <= 256 (whole B stays in shared
 *   memory).  C fp32 with leading dimension ldc >= N.
 * ---------------------------------------------------------------------- */
GQ_API int gq_gemm_bf16_nt(const uint16_t* A, int64_t M, int K, int64_t lda, const uint16_t* B, int N,
                    int64_t ldb, int act, float* C, int64_t ldc, int* dev_err, gq_stream stream);

/* gq_gemm_bf16_tn: C[K1 x N1] = X[R x K1]^T * Y[R x N1] (+ C if accumulate;
 *   R == 0 gives C = 0, X and Y may then be NULL),
 *   the weight gradient dW = A^T dZ.  K1, N1 <= 256.  Rows are split across
 *   thread blocks; fp32 partials go to `ws` (size from the query, which
 *   depends on the current device's SM count) and are summed in a fixed
 *   order, so the result is deterministic.                                */
GQ_API size_t gq_gemm_bf16_tn_workspace_bytes(int64_t R, int K1, int N1);
GQ_API int gq_gemm_bf16_tn(const uint16_t* X, int64_t R, int K1, int64_t ldx, const uint16_t* Y, int N1,
                    int64_t ldy, float* C, int64_t ldc, int accumulate, void* ws, size_t ws_bytes,
                    int* dev_err, gq_stream stream);

/* gq_to_bf16: dst[r][c] = bf16(src[r][c]) (round to nearest even) for
 *   c < cols, and 0 for cols <= c < dcols (padding for TMA strides).       */
GQ_API int gq_to_bf16(const float* src, int64_t rows, int cols, int64_t lds, uint16_t* dst, int64_t ldd,
               int dcols, gq_stream stream);

/* ------------------------------------------------------------------------
 * GCN / GraphSAGE-mean layer (AdaQP Sec. 2.1 weighted sum, Sec. 3.1 mixed
 * quantized/full-precision messages; Sancus Sec. 2 H' = sigma(A^ H W)).
 *
 * gq_gcn_layer_fwd:
 *   packed = quantize_pack(H_in rows with mask != 0, bits, seed)   (bits<32)
 *   A      = sum_{u->v} a_{u,v} m_u   -> A_save, bf16, n x d_in (lda)
 *   H_out  = act(A W)                 -> fp32, n x d_out (ldo)
 *   relu_bits (nullable): the derivative of act as bits, bit c % 32 of
 *           word relu_bits[r * ldrb + c / 32] = [H_out[r][c] > 0]
 *           (ldrb >= ceil(d_out / 32); words 4-byte aligned) -- the gate
 *           the layer above's backward applies to this layer's dZ.
 *   W is d_in x d_out fp32 row-major.  d_in % 4 == 0, lda % 8 == 0,
 *   d_in, d_out <= 256.  A_save is what the backward pass needs.
 *
 * gq_gcn_layer_bwd (same arguments read in reverse; the quantizer is the
 * identity in backward):
 *   dZ    = dH_out * [H_out > 0]  (act = RELU; dH_out for act = NONE), in
 *           bf16; or dZ_in when non-NULL (bf16, n x d_out, ldzi >= d_out,
 *           ldzi % 8 == 0), already made by the layer above, and then
 *           dH_out and H_out are not read (may be NULL)
 *   dW    = A^T dZ                -> fp32 d_in x d_out (ld d_out)
 *   if need_dinput:
 *     dA    = dZ W^T              -> dA_save if non-NULL (n x d_in, ld d_in)
 *     packed= quantize_pack(dA rows with mask != 0, bits, seed)
 *     dH_in = A^T-aggregation of the mixed messages -> n x d_in (ldi)
 *     or, when dZ_prev is non-NULL, the layer below's dZ in its place:
 *     dZ_prev = bf16(dH_in * g) -> n x d_in (ldzp >= d_in, ldzp % 8 == 0;
 *     columns d_in .. ldzp are not written), with g[r][c] = bit c % 32 of
 *     gate_in[r * ldgi + c / 32]: the relu_bits the layer below's forward
 *     wrote for its output, this layer's input (ldgi >= ceil(d_in / 32);
 *     NULL: no gate) -- the row flush of the aggregation applies the gate
 *     and the rounding, so no fp32 dH_in is written.
 * Both take a workspace of gq_gcn_layer_workspace_bytes(g, d_in, d_out,
 * bits) bytes (256-byte aligned) and a nullable device error word (see
 * the GEMMs).  Errors: GQ_ERR_INVALID_ARG, GQ_ERR_UNSUPPORTED,
 * GQ_ERR_WORKSPACE, GQ_ERR_CUDA.
 * Tracing: stage_events (nullable) is an array of cudaEvent_t handles,
 * 2 per stage; events[2k] is recorded on `stream` before stage k and
 * events[2k+1] after it.  Forward stages: 0 quantize, 1 aggregate,
 * 2 update GEMM.  Backward stages: 0 dZ, 1 dW, 2 dA, 3 quantize,
 * 4 transposed aggregate (stages 2-4 only when need_dinput).
 * ---------------------------------------------------------------------- */
GQ_API size_t gq_gcn_layer_workspace_bytes(const gq_graph* g, int d_in, int d_out, int bits);
GQ_API int gq_gcn_layer_fwd(const gq_graph* g, int coef, const float* H_in, int64_t ldh, int d_in,
                     const float* W, int d_out, const uint8_t* mask, int bits, uint64_t seed, int act,
                     uint16_t* A_save, int64_t lda, float* H_out, int64_t ldo, uint32_t* relu_bits,
                     int64_t ldrb, void* ws, size_t ws_bytes, int* dev_err, void* const* stage_events,
                     gq_stream stream);
GQ_API int gq_gcn_layer_bwd(const gq_graph* g, int coef, const float* dH_out, int64_t ldd,
                     const uint16_t* dZ_in, int64_t ldzi, const uint16_t* A_save, int64_t lda,
                     const float* H_out, int64_t ldo, const float* W, int d_in, int d_out,
                     const uint8_t* mask, int bits, uint64_t seed, int act, int need_dinput, float* dW,
                     float* dH_in, int64_t ldi, const uint32_t* gate_in, int64_t ldgi, uint16_t* dZ_prev,
                     int64_t ldzp, float* dA_save, void* ws, size_t ws_bytes, int* dev_err,
                     void* const* stage_events, gq_stream stream);

/* ------------------------------------------------------------------------
 * gq_sddmm_edge_softmax -- Tango Sec. 2.1, Fig. 1a steps 3-4, per
 * destination v and head k (heads contiguous, S and D n x heads fp32):
 *   E_pre[e,k] = S[u,k] + D[v,k]                  (SDDMM add, e = u -> v)
 *   E[e,k]     = E_pre if E_pre > 0, else slope * E_pre      (LeakyReLU)
 *   alpha[e,k] = exp(E[e,k]) / sum_{e' in in(v)} exp(E[e',k])
 * computed with the per-(v,k) maximum subtracted (same value), in fp32
 * (Tango Sec. 3.2 keeps the layer before softmax in full precision).
 * alpha and E_pre (nullable) are E x heads, indexed by CSR edge id.
 * heads in {1, 2, 4, 8}; S, D, alpha and E_pre 16-byte aligned
 * (GQ_ERR_INVALID_ARG otherwise).  Workspace:
 * gq_edge_softmax_workspace_bytes (split heavy rows only; may be 0).
 * ---------------------------------------------------------------------- */
GQ_API size_t gq_edge_softmax_workspace_bytes(const gq_graph* g, int heads);
GQ_API int gq_sddmm_edge_softmax(const gq_graph* g, const float* S, const float* D, int heads, float slope,
                          float* E_pre, float* alpha, void* ws, size_t ws_bytes, gq_stream stream);

/* ------------------------------------------------------------------------
 * GAT layer (Tango Sec. 2.1, Fig. 1a / 1b), F = f features per head,
 * d = heads * f, W is d_in x d fp32, a_src / a_dst are heads x f fp32.
 *
 * gq_gat_layer_fwd:
 *   H'    = H W          (tcgen05 bf16 GEMM)                 -> Hp_save n x d
 *   S, D  = H' a_src, H' a_dst per head (GEMM epilogue)      -> n x heads
 *   [bits < 32: the H' rows of marginal nodes are quantized  -> packed_save]
 *   alpha = edge softmax of LeakyReLU(S[u] + D[v])           -> E x heads
 *   [alpha_bits == 8: alpha quantized per destination and head with
 *    seed ^ GQ_ALPHA_SEED_TAG (gq_quantize_edge_values) -> acode_save,
 *    ahdr_save, and a^ = its de-quantized values; alpha_bits == 32: a^ =
 *    alpha.  Other values: GQ_ERR_INVALID_ARG]
 *   out   = sum_{u->v} a^[e,k] m_u[kF+f]                     -> n x d
 *   packed_save (n x gq_packed_pitch(d, bits), nullable) keeps the
 *   forward's quantized messages for the backward pass (required there
 *   when bits < 32); acode_save / ahdr_save (both or neither; nullable;
 *   acode_save may be NULL on a graph without edges) keep the attention
 *   codes, which the backward needs to use a^.
 * gq_gat_layer_bwd (the quantizer is the identity in backward):
 *   dalpha = SDDMM dot of dOut[v] with the forward messages m_u;
 *   dE_pre = alpha (dalpha - P) LeakyReLU'; dD = in-edge sums, dS =
 *   out-edge sums; dM = transposed multi-head SpMM of dOut (rows of
 *   marginal nodes quantized when bits < 32, seed) weighted by a^
 *   (the forward's codes acode_save / ahdr_save when ahdr_save is given,
 *   else alpha);
 *   dH' = dM + dS a_src + dD a_dst; da_src = sum_u dS[u] H'[u],
 *   da_dst likewise; dW = H^T dH'; dH = dH' W^T.
 *   dEpre_save (E x heads) and dHp_save (n x d fp32) are optional copies.
 * Limits: heads in {1,2,4,8}, f a power of two >= 16, d_in, d <= 256.
 * Workspace: gq_gat_layer_workspace_bytes(g, d_in, heads, f, bits,
 * alpha_bits), with alpha_bits = 8 for a backward given attention codes.
 * ---------------------------------------------------------------------- */
GQ_API size_t gq_gat_layer_workspace_bytes(const gq_graph* g, int d_in, int heads, int f, int bits,
                                           int alpha_bits);
GQ_API int gq_gat_layer_fwd(const gq_graph* g, const float* H, int64_t ldh, int d_in, const float* W,
                     const float* a_src, const float* a_dst, int heads, int f, float slope,
                     const uint8_t* mask, int bits, uint64_t seed, int alpha_bits, float* Hp_save,
                     float* S_save, float* D_save, float* alpha_save, uint8_t* packed_save,
                     uint8_t* acode_save, float* ahdr_save, float* out, void* ws, size_t ws_bytes,
                     int* dev_err, gq_stream stream);
GQ_API int gq_gat_layer_bwd(const gq_graph* g, const float* dOut, const float* H, int64_t ldh,
                     const float* Hp_save, const float* S_save, const float* D_save,
                     const float* alpha_save, const uint8_t* packed_save, const uint8_t* acode_save,
                     const float* ahdr_save, const float* W, const float* a_src, const float* a_dst,
                     int d_in, int heads, int f, float slope, const uint8_t* mask, int bits, uint64_t seed,
                     float* dW, float* da_src, float* da_dst, float* dH, float* dEpre_save,
                     float* dHp_save, void* ws, size_t ws_bytes, int* dev_err, gq_stream stream);

/* ------------------------------------------------------------------------
 * gq_dequant_spmm_noalloc -- no counterpart on the pages: a convenience of
 * this library.  Same arguments and result as gq_dequant_spmm, minus the
 * workspace, for callers that may not allocate device memory where they
 * aggregate (a memory-pool hook, a plug-in that is only lent its input and
 * output buffers, a path that must not block on or fail in an allocator).
 * Its scratch is one fixed array of gq_noalloc_scratch_bytes() bytes (8 MiB)
 * compiled into the library, held on every GPU that loads the library until
 * the process exits.  The call allocates nothing.
 *   - Each call looks up the array's address on the current device (a
 *     host-side lookup).  Under CUDA's lazy module loading the first call on
 *     a device may load the library's module and reserve the array there
 *     (and can fail for lack of device memory, as any module load can);
 *     make that first call before any stream capture.
 *   - All calls on a device share the array and find the previous call's
 *     contents in it; each call clears what must start at zero.  Calls that
 *     overlap on the GPU race on the array.
 *   - The arguments are checked as gq_dequant_spmm checks them; then a
 *     graph and width whose scratch need (gq_spmm_workspace_bytes) exceeds
 *     the array return GQ_ERR_SCRATCH_LIMIT.  Nothing is launched on error.
 * ---------------------------------------------------------------------- */
GQ_API size_t gq_noalloc_scratch_bytes(void);
GQ_API int gq_dequant_spmm_noalloc(const gq_graph* g, int transpose, int coef, const float* X,
                                   int64_t ldx, const uint8_t* packed, const uint8_t* mask, int d,
                                   int bits, float* Y, int64_t ldy, gq_stream stream);

/* ------------------------------------------------------------------------
 * gq_message_variance_weights -- AdaQP Sec. 4.2, the weight of message k in
 * the gradient-variance objective (Problem 11):
 *   beta[k] = sum_{v in N_T(k)} a_{k,v}^2 * d * (max X[k,:] - min X[k,:])^2 / 6
 * with N_T(k) every destination v of an edge k -> v (on one GPU all of
 * them live on the "target device") and a_{k,v} the coefficient `coef`
 * (gq_coef) the aggregation applies; the aggregated error of message k
 * quantized at b bits has variance beta[k] / (2^b - 1)^2.  X: n x d fp32
 * (ldx), the message rows before quantization; beta: n fp32.  ws:
 * gq_message_variance_weights_workspace_bytes(g) bytes (partial sums of
 * the nodes with more out-edges than the hub threshold; may be NULL when 0).
 * Sums in fp32 in a fixed order.  Errors: GQ_ERR_INVALID_ARG,
 * GQ_ERR_WORKSPACE, GQ_ERR_CUDA.
 * ---------------------------------------------------------------------- */
GQ_API size_t gq_message_variance_weights_workspace_bytes(const gq_graph* g);
GQ_API int gq_message_variance_weights(const gq_graph* g, int coef, const float* X, int64_t ldx, int d,
                                       float* beta, void* ws, size_t ws_bytes, gq_stream stream);

/* ------------------------------------------------------------------------
 * gq_assign_bits -- AdaQP Sec. 4.2, the bit-width choice (Problems 10-12)
 * on one device.  With a single device pair the time objective is
 * theta + gamma * sum_k d * b_k (theta a constant), and the weighted sum
 * lam * sum_k beta_k / (2^b_k - 1)^2 + (1 - lam) * time separates per
 * message, so each row k takes
 *   rbits[k] = argmin_{b in {2,4,8}} lam*(beta[k]/(L*L)) + tw*(d*b),
 *   L = 2^b - 1, tw = (1 - lam) * gamma,
 * each operation an fp64 round-to-nearest in that order, ties to the fewer
 * bits; rbits[k] = 0 (a full-precision row) where mask[k] == 0.  beta: n
 * fp32 (gq_message_variance_weights); mask: n bytes or NULL (every row);
 * rbits: n bytes, the per-row widths of gq_quantize_pack_mixed.  lam in
 * [0, 1], gamma >= 0 (seconds per transferred bit in the pages' cost model;
 * any consistent unit).  Errors: GQ_ERR_INVALID_ARG, GQ_ERR_CUDA.
 * ---------------------------------------------------------------------- */
GQ_API int gq_assign_bits(const float* beta, const uint8_t* mask, int64_t n, int d, double lam, double gamma,
                          uint8_t* rbits, gq_stream stream);

/* ------------------------------------------------------------------------
 * gq_quant_error -- Tango Sec. 3.2, Eq. 4, the relative quantization error
 * of a tensor:
 *   *err = (1/(n d)) sum_{r, j} |X[r,j] - Xq[r,j]| / (|X[r,j]| + |Xq[r,j]| + eps)
 * with Xq[r,j] = fmaf(q, S, Z) from the packed row r (bits 2, 4, 8) where
 * mask[r] != 0 (mask NULL: every row), and Xq = X (a zero term) otherwise.
 * The absolute values read the page's denominator X + Xq, written for a
 * symmetric quantizer whose two values share one sign; the metric lies in
 * [0, 1].  Tango takes eps = 0.0005 and keeps the fewest bits with an error
 * below 0.3.  err: one device double.  ws: gq_quant_error_workspace_bytes()
 * bytes (8-byte aligned).  fp32 per row, fp64 across rows, fixed order.
 * Errors: GQ_ERR_INVALID_ARG (bad bits, eps <= 0, null or misaligned
 * pointers), GQ_ERR_WORKSPACE, GQ_ERR_CUDA.
 * ---------------------------------------------------------------------- */
GQ_API size_t gq_quant_error_workspace_bytes(void);
GQ_API int gq_quant_error(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* packed,
                          const uint8_t* mask, int bits, float eps, double* err, void* ws, size_t ws_bytes,
                          gq_stream stream);

/* ------------------------------------------------------------------------
 * gq_bits_for_error -- Tango Sec. 3.2, Eq. 4 and the rule built on it: the
 * fewest bits whose relative quantization error Error_X stays below a
 * threshold (Tango: 0.3, eps = 0.0005), chosen from 2, 4 and 8 (8 when none
 * does).  One pass over X: for every row with mask[r] != 0 (mask NULL:
 * every row) the codes gq_quantize_pack writes at each width with this seed
 * (same fp32 operations, same noise), de-quantized by fmaf(q, S, Z), enter
 * the three sums of gq_quant_error; nothing is written but the results.
 * err3: NULL or three device doubles, Error_X at 2, 4 and 8 bits.  bits: one
 * device int32, the chosen width.  ws: gq_bits_for_error_workspace_bytes()
 * bytes (8-byte aligned).  Asynchronous; the caller reads *bits after a
 * synchronization.  Errors: GQ_ERR_INVALID_ARG (null bits or X, d < 1,
 * ldx < d, eps <= 0, threshold <= 0), GQ_ERR_WORKSPACE, GQ_ERR_CUDA.
 * ---------------------------------------------------------------------- */
GQ_API size_t gq_bits_for_error_workspace_bytes(void);
GQ_API int gq_bits_for_error(const float* X, int64_t n, int d, int64_t ldx, const uint8_t* mask, uint64_t seed,
                             double threshold, float eps, double* err3, int32_t* bits, void* ws, size_t ws_bytes,
                             gq_stream stream);

/* ------------------------------------------------------------------------
 * gq_selftest_bounded_wait -- no counterpart on the pages: a check of the
 * failure path of the library's bounded waits, without a GPU fault.  One
 * warp waits for phase 0 of an mbarrier, through the wait helper of the
 * GEMMs (helper 0) or of the aggregation kernels (helper 1), for at most
 * limit_cycles SM cycles (1e3 .. 2e9).  With complete == 0 nothing ever
 * arrives on the barrier: the wait gives up and writes 0x5354 to
 * *dev_status (a device int; only if it still holds 0).  With complete != 0
 * the barrier completes first and *dev_status is left unchanged.  In the
 * library's kernels the same helpers write, on a timeout, the GEMM stage
 * (1 .. 13) to the caller's dev_err word, or 0x5350 to the graph's status
 * word (an aggregation row copy that did not land).
 * Errors: GQ_ERR_INVALID_ARG (null dev_status, helper or limit out of
 * range), GQ_ERR_CUDA.
 * ---------------------------------------------------------------------- */
GQ_API int gq_selftest_bounded_wait(int helper, int complete, long long limit_cycles, int* dev_status,
                                    gq_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* GQ_H */
