// dwc_fgrad_f32.cu -- filter-gradient kernels, f32 inputs; workspace query of all dtypes.
#include "dwc_fgrad.cuh"
#include "dwc_mma_fgrad.cuh"

namespace dwc {
cudaError_t launch_filter_grad_f32(const FilterGrad& p) {
    if (p.FH != p.FW) return launch_fgrad_stripe_f32(p);
    return launch_fgrad_dispatch<float>(p);
}

size_t fgrad_workspace_floats_f32(int N, int OH, int OW, int C, int FH, int FW) {
    return fgrad_workspace_t<float>(N, OH, OW, C, FH, FW);
}

size_t filter_grad_workspace_floats(int N, int OH, int OW, int C, int FH, int FW, int dtype) {
    if (FH != FW) {
        switch (dtype) {
            case kF32: return fgrad_stripe_workspace_floats_f32(N, OH, OW, C, FH, FW);
            case kBF16: return fgrad_stripe_workspace_floats_bf16(N, OH, OW, C, FH, FW);
            default: return fgrad_stripe_workspace_floats_f16(N, OH, OW, C, FH, FW);
        }
    }
    if (dtype == kF32) return fgrad_workspace_floats_f32(N, OH, OW, C, FH, FW);
    // 16-bit inputs may run the tensor-core kernel: its slices must fit too
    const size_t mma = mma_fgrad_workspace_floats(N, C, OH, OW, FH, FW);
    const size_t cc = dtype == kBF16 ? fgrad_workspace_floats_bf16(N, OH, OW, C, FH, FW)
                                     : fgrad_workspace_floats_f16(N, OH, OW, C, FH, FW);
    return std::max(mma, cc);
}

bool filter_grad_supported(int FH, int FW) { return FH == FW && FH >= 3 && FH <= 31 && (FH & 1); }
bool rows_supported(int FH, int FW) { return FH == FW && FH >= 3 && FH <= 51 && (FH & 1); }
bool stripe_supported(int FH, int FW) {
    return FH != FW && FH >= 1 && FH <= 255 && FW >= 1 && FW <= 51 && (FW & 1);
}
cudaError_t launch_filter_grad_s2_f32(const FilterGrad& p) { return launch_fgrad_s2_dispatch<float>(p); }

size_t fgrad_s2_workspace_floats_f32(int N, int OH, int OW, int C, int FH, int FW) {
    return fgrad_s2_workspace_t<float>(N, OH, OW, C, FH, FW);
}

size_t filter_grad_s2_workspace_floats(int N, int OH, int OW, int C, int FH, int FW, int dtype) {
    switch (dtype) {
        case kF32: return fgrad_s2_workspace_floats_f32(N, OH, OW, C, FH, FW);
        case kBF16: return fgrad_s2_workspace_floats_bf16(N, OH, OW, C, FH, FW);
        default: return fgrad_s2_workspace_floats_f16(N, OH, OW, C, FH, FW);
    }
}
}  // namespace dwc
