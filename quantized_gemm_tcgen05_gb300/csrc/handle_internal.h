// Internal accessors of the opaque gemm handle for other translation units of
// the library.
#pragma once
#include "gemm.h"

namespace qg {
// CUDA device ordinal the handle is bound to, or -1 for a NULL handle.
int handle_device(gemm_handle_t h);
}  // namespace qg
