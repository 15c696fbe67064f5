// dwc_rows_f32.cu -- row-streaming forward / backward-data kernels, f32 inputs.
#include "dwc_rows.cuh"
#include "dwc_s2data.cuh"

namespace dwc {
cudaError_t launch_rows_f32(const RowConv& p) { return launch_rows_dispatch<float>(p); }
cudaError_t launch_rows_s2_f32(const RowConv& p) { return launch_rows_s2_dispatch<float>(p); }
cudaError_t launch_s2_bwd_data_f32(const GeneralConv& p) { return launch_s2_bwd_data_dispatch<float>(p); }
}  // namespace dwc
