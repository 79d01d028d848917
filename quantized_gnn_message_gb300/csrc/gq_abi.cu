// gq_abi.cu -- small ABI helpers: status text, version, packed-row sizes.
#include "gq_common.cuh"

extern "C" const char* gq_status_string(int status) {
  switch (status) {
    case GQ_OK: return "ok";
    case GQ_ERR_INVALID_ARG: return "invalid argument";
    case GQ_ERR_UNSUPPORTED: return "unsupported shape or option";
    case GQ_ERR_BAD_GRAPH: return "graph fails CSR validation";
    case GQ_ERR_CUDA: return "CUDA runtime error";
    case GQ_ERR_TIMEOUT: return "device-side wait timed out";
    case GQ_ERR_WORKSPACE: return "workspace or storage too small";
    case GQ_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

extern "C" int gq_version(void) { return 200; }

extern "C" size_t gq_graph_struct_bytes(void) { return sizeof(gq_graph); }

extern "C" int64_t gq_packed_pitch(int d, int bits) {
  if (d < 1 || !gq::valid_bits(bits)) return -1;
  return gq::packed_pitch(d, bits);
}

extern "C" int64_t gq_packed_header_offset(int d, int bits) {
  if (d < 1 || !gq::valid_bits(bits)) return -1;
  return gq::header_offset(d, bits);
}
