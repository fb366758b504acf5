// Instantiations of the scaled-operand tcgen05 GEMM kernel for tile widths 16, 32, 64.
#include "umma_dq_gemm.cuh"

namespace qg {
template cudaError_t launch_dq_bn<16>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int dq_stages_bn<16>();
template cudaError_t launch_dq_bn<32>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int dq_stages_bn<32>();
template cudaError_t launch_dq_bn<64>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int dq_stages_bn<64>();
}  // namespace qg
