// wqmm_gemm.cu -- fused dequantize + tcgen05 GEMM for large M (placeholder:
// the GEMV path serves every shape until the tensor-core GEMM lands).
#include "wqmm_device.cuh"

namespace wqmm {

bool gemm_supports(const GemvArgs&) { return false; }

int launch_gemm(const GemvArgs&, cudaStream_t) { return kUnsupported; }

}  // namespace wqmm
