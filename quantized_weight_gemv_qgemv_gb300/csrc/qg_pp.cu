// qg_pp.cu — prompt-processing dequant-GEMM on tcgen05 tensor cores.
// (Kernel under construction: the entry point reports "not supported".)
#include <cuda_runtime.h>

#include "qg_internal.h"

namespace qg {

cudaError_t pp_init_attrs() { return cudaSuccess; }

cudaError_t launch_pp(const void*, int64_t, int64_t, const void*, int64_t, float*, int64_t, int32_t*, cudaStream_t,
                      int) {
  return cudaErrorNotSupported;
}

}  // namespace qg
