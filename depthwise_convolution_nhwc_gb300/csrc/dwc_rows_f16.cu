// dwc_rows_f16.cu -- row-streaming forward / backward-data kernels, f16 inputs.
#include "dwc_rows.cuh"

namespace dwc {
cudaError_t launch_rows_f16(const RowConv& p) { return launch_rows_dispatch<__half>(p); }
}  // namespace dwc
