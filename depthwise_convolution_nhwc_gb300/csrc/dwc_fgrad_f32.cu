// dwc_fgrad_f32.cu -- filter-gradient kernels, f32 inputs.
#include "dwc_fgrad.cuh"
#include "dwc_mma_fgrad.cuh"

namespace dwc {
size_t cuda_core_fgrad_workspace_floats(int N, int OH, int OW, int C, int FH, int FW, int e);

cudaError_t launch_filter_grad_f32(const FilterGrad& p) { return launch_fgrad_dispatch<float>(p); }

size_t filter_grad_workspace_floats(int N, int OH, int OW, int C, int FH, int FW, int e) {
    if (FH != FW) return 0;
    // 16-bit inputs may run the tensor-core kernel: its slices must fit too
    const size_t mma = e == 2 ? mma_fgrad_workspace_floats(N, C, OH, OW, FH, FW) : 0;
    return std::max(mma, cuda_core_fgrad_workspace_floats(N, OH, OW, C, FH, FW, e));
}

size_t cuda_core_fgrad_workspace_floats(int N, int OH, int OW, int C, int FH, int FW, int e) {
    switch (FH) {
#define DWC_FGRAD_WS(F) \
    case F:             \
        return fgrad_workspace_dispatch<F>(N, OH, OW, C, e);
        DWC_FGRAD_FILTERS(DWC_FGRAD_WS)
#undef DWC_FGRAD_WS
        default:
            return 0;
    }
}

bool filter_grad_supported(int FH, int FW) { return FH == FW && FH >= 3 && FH <= 31 && (FH & 1); }
bool rows_supported(int FH, int FW) { return FH == FW && FH >= 3 && FH <= 31 && (FH & 1); }
}  // namespace dwc
