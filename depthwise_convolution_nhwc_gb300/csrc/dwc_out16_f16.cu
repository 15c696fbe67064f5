// dwc_out16_f16.cu -- forward / backward-data kernels writing f16 outputs (f16 inputs, fp32
// accumulation rounded once at the store).
#include "dwc_mma.cuh"
#include "dwc_s2data.cuh"
#include "dwc_small.cuh"

namespace dwc {
cudaError_t launch_rows_o16_f16(const RowConv& p) { return launch_rows_or_mma<__half, __half>(p); }
cudaError_t launch_rows_s2_o16_f16(const RowConv& p) { return launch_rows_s2_dispatch<__half, __half>(p); }
cudaError_t launch_small_rows_o16_f16(const RowConv& p) { return launch_small_rows_t<__half, __half>(p); }
cudaError_t launch_s2_bwd_data_o16_f16(const GeneralConv& p) {
    return launch_s2_bwd_data_dispatch<__half, __half>(p);
}
}  // namespace dwc
