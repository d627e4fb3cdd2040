// draft_tc.cu -- tensor-core (tcgen05) V sweep of the drafter.
#include "common.cuh"
#include "kernels.h"

namespace dspark {

bool draft_tc_supported(const DraftArgs& a) {
    (void)a;
    return false;
}
int draft_tc_slices(const DraftArgs& a) {
    (void)a;
    return 1;
}
cudaError_t launch_draft_tc_sweep(DraftArgs& a, int k, cudaStream_t s) {
    (void)a;
    (void)k;
    (void)s;
    return cudaErrorNotSupported;
}

}  // namespace dspark
