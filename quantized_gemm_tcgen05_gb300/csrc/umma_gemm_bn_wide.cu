// Instantiations of the dense tcgen05 GEMM kernel for tile widths 224, 256
// (separate translation units so they compile in parallel).
#include "umma_gemm.cuh"

namespace qg {
template cudaError_t launch_umma_bn<224>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int umma_stages_bn<224>(int);
template cudaError_t launch_umma_bn<256>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int umma_stages_bn<256>(int);
}  // namespace qg
