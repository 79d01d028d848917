// gq_noalloc.cu -- the aggregation without a caller workspace.
//
// gq_dequant_spmm needs scratch when a heavy row is cut into several block
// tasks: one partial row per task plus an arrival counter per cut row.  The
// regular entry point takes that scratch from a caller buffer.  Some callers
// cannot provide one, because they may not allocate device memory where
// they aggregate: a framework's memory-pool hook, a plug-in whose host only
// lends it the input and output buffers, or code on a path that must never
// block on, or fail in, the allocator.  For them, gq_dequant_spmm_noalloc
// uses a fixed scratch array compiled into this library instead.
//
// Facts a caller must know (also in gq.h):
//   - the array holds kNoallocScratchBytes (8 MiB) on every GPU that loads
//     the library, until the process exits.  With CUDA's lazy module
//     loading the module that holds it may be loaded, and the array
//     reserved, by the first call on a device; make that first call before
//     any stream capture (it can fail for lack of device memory like any
//     module load);
//   - every call looks up the array's device address on the current device
//     (a host-side lookup, no allocation), so the address stays right after
//     a device reset or a new primary context;
//   - every call on a device shares the one array, which keeps whatever the
//     last call left in it.  The arrival counters are cleared at the start
//     of each call; partial rows are written before they are read.  Calls
//     that overlap on the GPU (different streams, no ordering) race on it;
//   - the arguments are checked first (as gq_dequant_spmm checks them); a
//     graph / width whose scratch need exceeds the array is then rejected
//     with GQ_ERR_SCRATCH_LIMIT before anything is launched;
//   - the call allocates nothing: no cudaMalloc, no cudaFree, no allocating
//     library routine.
#include "gq_common.cuh"
#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr size_t kNoallocScratchBytes = (size_t)8 << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name only stands in for the symbol; this address is what a
// kernel can use.
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return GQ_ERR_CUDA;
  *out = p;
  return GQ_OK;
}

}  // namespace
}  // namespace gq

extern "C" size_t gq_noalloc_scratch_bytes(void) { return gq::kNoallocScratchBytes; }

extern "C" int gq_dequant_spmm_noalloc(const gq_graph* g, int transpose, int coef, const float* X, int64_t ldx,
                                       const uint8_t* packed, const uint8_t* mask, int d, int bits, float* Y,
                                       int64_t ldy, gq_stream stream) {
  using namespace gq;
  GQ_TRY(spmm_check(g, X, ldx, packed, mask, d, bits, Y, ldy, nullptr));
  if (spmm_workspace(g, transpose, d) > kNoallocScratchBytes) return GQ_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  GQ_TRY(scratch_address(&scratch));
  return dequant_spmm(g, transpose, coef, X, ldx, packed, mask, d, bits, Y, ldy, scratch, kNoallocScratchBytes,
                      (cudaStream_t)stream, nullptr);
}
