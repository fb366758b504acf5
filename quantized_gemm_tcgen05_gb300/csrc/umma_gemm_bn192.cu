// Instantiation of the dense tcgen05 GEMM kernel for tile width 192 (one
// width per translation unit, so they compile in parallel).
#include "umma_gemm.cuh"

namespace qg {
template cudaError_t launch_umma_bn<192>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int umma_stages_bn<192>(int);
}  // namespace qg
