// dwc_rows_bf16.cu -- forward / backward-data kernels, bf16 inputs (tensor-core kernel for
// filters from 15 taps on rows of at least 24 outputs, row-streaming kernel otherwise).
#include "dwc_mma.cuh"
#include "dwc_s2data.cuh"

namespace dwc {
cudaError_t launch_rows_bf16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_rows_o16_bf16(p);
    return launch_rows_or_mma<__nv_bfloat16>(p);
}

bool tensor_core_rows(const RowConv& p) {
    MmaArgs a;
    size_t smem = 0;
    return mma_rows_wanted(p) && mma_plan(p, a, smem);
}
cudaError_t launch_rows_s2_bf16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_rows_s2_o16_bf16(p);
    return launch_rows_s2_dispatch<__nv_bfloat16>(p);
}
cudaError_t launch_s2_bwd_data_bf16(const GeneralConv& p) {
    if (p.out_dtype != kF32) return launch_s2_bwd_data_o16_bf16(p);
    return launch_s2_bwd_data_dispatch<__nv_bfloat16>(p);
}
}  // namespace dwc
