// dwc_fgrad_f16.cu -- filter-gradient kernels, f16 inputs (tensor-core and CUDA-core).
#include "dwc_fgrad.cuh"
#include "dwc_mma_fgrad.cuh"

namespace dwc {
cudaError_t launch_filter_grad_f16(const FilterGrad& p) {
    if (p.FH != p.FW) return launch_fgrad_stripe_f16(p);
    // tensor-core kernels where they serve the shape (tcgen05 first, then the warp-level
    // MMA kernel), the CUDA-core kernel otherwise; a family preference picks one of them
    const int pref = family_preference();
    if (tc_fgrad_taken(p)) {
        const cudaError_t err = launch_tc_fgrad_f16(p);
        if (err != cudaErrorNotSupported) return err;
    }
    if (pref == 0 || pref == 4) {
        const cudaError_t err = launch_mma_fgrad<__half>(p);
        if (err != cudaErrorNotSupported) return err;
    }
    return launch_fgrad_dispatch<__half>(p);
}

size_t fgrad_workspace_floats_f16(int N, int OH, int OW, int C, int FH, int FW) {
    return fgrad_workspace_t<__half>(N, OH, OW, C, FH, FW);
}
cudaError_t launch_filter_grad_s2_f16(const FilterGrad& p) { return launch_fgrad_s2_dispatch<__half>(p); }
size_t fgrad_s2_workspace_floats_f16(int N, int OH, int OW, int C, int FH, int FW) {
    return fgrad_s2_workspace_t<__half>(N, OH, OW, C, FH, FW);
}
}  // namespace dwc
