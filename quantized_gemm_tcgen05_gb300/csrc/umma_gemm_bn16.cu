// Instantiation of the dense tcgen05 GEMM kernel for tile width 16 (one
// width per translation unit, so they compile in parallel).
#include "umma_gemm.cuh"

namespace qg {
template cudaError_t launch_umma_bn<16>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int umma_stages_bn<16>(int);
}  // namespace qg
