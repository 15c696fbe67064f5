// dwc_stripe_bf16.cu -- forward / backward data for stripe (non-square) filters, bf16 inputs.
#include "dwc_rows.cuh"

namespace dwc {
cudaError_t launch_rows_stripe_bf16(const RowConv& p) { return launch_rows_stripe_dispatch<__nv_bfloat16>(p); }
}  // namespace dwc
