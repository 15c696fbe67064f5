// dwc_stripe_f16.cu -- forward / backward data for stripe (non-square) filters, f16 inputs.
#include "dwc_rows.cuh"

namespace dwc {
cudaError_t launch_rows_stripe_f16(const RowConv& p) { return launch_rows_stripe_dispatch<__half>(p); }
}  // namespace dwc
