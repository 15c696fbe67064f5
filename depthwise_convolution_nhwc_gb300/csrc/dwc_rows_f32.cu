// dwc_rows_f32.cu -- row-streaming forward / backward-data kernels, f32 inputs.
#include "dwc_rows.cuh"

namespace dwc {
cudaError_t launch_rows_f32(const RowConv& p) { return launch_rows_dispatch<float>(p); }
cudaError_t launch_rows_s2_f32(const RowConv& p) { return launch_rows_s2_dispatch<float>(p); }
}  // namespace dwc
