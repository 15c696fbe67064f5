// dwc_rows_bf16.cu -- row-streaming forward / backward-data kernels, bf16 inputs.
#include "dwc_rows.cuh"

namespace dwc {
cudaError_t launch_rows_bf16(const RowConv& p) { return launch_rows_dispatch<__nv_bfloat16>(p); }
}  // namespace dwc
