// dwc_fgrad_bf16.cu -- filter-gradient kernels, bf16 inputs (tensor-core and CUDA-core).
#include "dwc_fgrad.cuh"
#include "dwc_mma_fgrad.cuh"

namespace dwc {
cudaError_t launch_filter_grad_bf16(const FilterGrad& p) {
    if (p.FH != p.FW) return launch_fgrad_stripe_bf16(p);
    // tensor-core kernels where they serve the shape (tcgen05 first, then the warp-level
    // MMA kernel), the CUDA-core kernel otherwise; a family preference picks one of them
    const int pref = family_preference();
    if (tc_fgrad_taken(p)) {
        const cudaError_t err = launch_tc_fgrad_bf16(p);
        if (err != cudaErrorNotSupported) return err;
    }
    if (pref == 0 || pref == 4) {
        const cudaError_t err = launch_mma_fgrad<__nv_bfloat16>(p);
        if (err != cudaErrorNotSupported) return err;
    }
    return launch_fgrad_dispatch<__nv_bfloat16>(p);
}

bool tc_fgrad_taken(const FilterGrad& p) {
    if (p.FH != p.FW || (p.dtype != kBF16 && p.dtype != kF16)) return false;
    const int pref = family_preference();
    if (pref != 0 && pref != 2) return false;
    return (pref == 2 || tc_fgrad_wanted(p.FW, p.OW)) && tc_fgrad_fits(p);
}

bool tensor_core_fgrad(int N, int C, int OH, int OW, int FH, int FW) {
    return mma_fgrad_workspace_floats(N, C, OH, OW, FH, FW) > 0;
}

size_t fgrad_workspace_floats_bf16(int N, int OH, int OW, int C, int FH, int FW) {
    return fgrad_workspace_t<__nv_bfloat16>(N, OH, OW, C, FH, FW);
}
cudaError_t launch_filter_grad_s2_bf16(const FilterGrad& p) { return launch_fgrad_s2_dispatch<__nv_bfloat16>(p); }
size_t fgrad_s2_workspace_floats_bf16(int N, int OH, int OW, int C, int FH, int FW) {
    return fgrad_s2_workspace_t<__nv_bfloat16>(N, OH, OW, C, FH, FW);
}
}  // namespace dwc
