// Tensor-core (tcgen05) attention for bf16, d = 128: not built yet.
#include "attend.cuh"

namespace csahca {

bool attend_tc_supported(const AttendArgs& a) {
    (void)a;
    return false;
}

cudaError_t attend_tc_launch(const AttendArgs& a, int S, int kps, float* o_part, float* lse_part, unsigned* err,
                             cudaStream_t st) {
    (void)a; (void)S; (void)kps; (void)o_part; (void)lse_part; (void)err; (void)st;
    return cudaErrorNotSupported;
}

}  // namespace csahca
