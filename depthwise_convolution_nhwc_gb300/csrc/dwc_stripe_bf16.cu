// dwc_stripe_bf16.cu -- stripe (non-square) filters, bf16 inputs: forward / backward data on the
// row kernel and the filter gradient, both with the filter height read at run time.
#include "dwc_fgrad.cuh"

namespace dwc {
cudaError_t launch_rows_stripe_bf16(const RowConv& p) { return launch_rows_stripe_dispatch<__nv_bfloat16>(p); }
cudaError_t launch_fgrad_stripe_bf16(const FilterGrad& p) { return launch_fgrad_stripe_dispatch<__nv_bfloat16>(p); }
size_t fgrad_stripe_workspace_floats_bf16(int N, int OH, int OW, int C, int FH, int FW) {
    return fgrad_stripe_workspace_t<__nv_bfloat16>(N, OH, OW, C, FH, FW);
}
}  // namespace dwc
