// dwc_fgrad_f32.cu -- filter-gradient kernels, f32 inputs.
#include "dwc_fgrad.cuh"

namespace dwc {
cudaError_t launch_filter_grad_f32(const FilterGrad& p) { return launch_fgrad_dispatch<float>(p); }

size_t filter_grad_workspace_floats(int N, int OH, int OW, int C, int FH, int FW, int e) {
    if (FH != FW) return 0;
    switch (FH) {
#define DWC_FGRAD_WS(F) \
    case F:             \
        return fgrad_workspace_inst<F, F>(N, OH, OW, C, e);
        DWC_FGRAD_FILTERS(DWC_FGRAD_WS)
#undef DWC_FGRAD_WS
        default:
            return 0;
    }
}

bool filter_grad_supported(int FH, int FW) { return FH == FW && FH >= 3 && FH <= 31 && (FH & 1); }
bool rows_supported(int FH, int FW) { return FH == FW && FH >= 3 && FH <= 31 && (FH & 1); }
}  // namespace dwc
