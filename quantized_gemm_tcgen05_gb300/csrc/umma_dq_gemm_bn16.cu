// Instantiation of the scaled-operand tcgen05 GEMM kernel for tile width 16
// (one width per translation unit, so they compile in parallel).
#include "umma_dq_gemm.cuh"

namespace qg {
template cudaError_t launch_dq_bn<16>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int dq_stages_bn<16>();
}  // namespace qg
