// dwc_stripe_f32.cu -- forward / backward data for stripe (non-square) filters, f32 inputs.
#include "dwc_rows.cuh"

namespace dwc {
cudaError_t launch_rows_stripe_f32(const RowConv& p) { return launch_rows_stripe_dispatch<float>(p); }
}  // namespace dwc
