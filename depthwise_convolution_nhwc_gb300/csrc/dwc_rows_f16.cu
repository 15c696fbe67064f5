// dwc_rows_f16.cu -- forward / backward-data kernels, f16 inputs (the tcgen05 kernel where
// tc_rows_wanted says so, the warp-level MMA kernel or the row-streaming kernel otherwise).
#include "dwc_mma.cuh"
#include "dwc_s2data.cuh"

namespace dwc {
cudaError_t launch_rows_f16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_rows_o16_f16(p);
    return launch_rows_or_mma<__half>(p);
}
cudaError_t launch_rows_s2_f16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_rows_s2_o16_f16(p);
    return launch_rows_s2_dispatch<__half>(p);
}
cudaError_t launch_s2_bwd_data_f16(const GeneralConv& p) {
    if (p.out_dtype != kF32) return launch_s2_bwd_data_o16_f16(p);
    return launch_s2_bwd_data_dispatch<__half>(p);
}
}  // namespace dwc
