// Instantiations of the dense tcgen05 GEMM kernel for tile widths 16, 32, 64
// (separate translation units so they compile in parallel).
#include "umma_gemm.cuh"

namespace qg {
template cudaError_t launch_umma_bn<16>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int umma_stages_bn<16>(int);
template cudaError_t launch_umma_bn<32>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int umma_stages_bn<32>(int);
template cudaError_t launch_umma_bn<64>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int umma_stages_bn<64>(int);
}  // namespace qg
