// fmha_sm103.cu -- tensor-core attention forward for sm_103a (placeholder:
// routes to the CUDA-core kernel until the tcgen05 kernel lands).
#include <cuda_runtime.h>

#include "fmha_common.h"

namespace fmha {

__device__ int g_status;   // FMHA_OK, or FMHA_ERR_TIMEOUT after a bounded wait expired

int sm103_read_status(int reset) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    if (reset) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return FMHA_ERR_CUDA;
        }
    }
    return v;
}

int launch_sm103(const Params &p, cudaStream_t stream) { return launch_simt(p, stream); }

}  // namespace fmha
