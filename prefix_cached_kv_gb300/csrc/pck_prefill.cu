// pck_prefill.cu -- batched-Q (M > 1) prefix attention on the tensor cores (tcgen05).
#include "pck_common.cuh"
#include "pck_kernels.h"

namespace pck {

bool prefill_supported(int D) { (void)D; return false; }

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t st, int sms, int D) {
    (void)p; (void)st; (void)sms; (void)D;
    return cudaErrorNotSupported;
}

}  // namespace pck
