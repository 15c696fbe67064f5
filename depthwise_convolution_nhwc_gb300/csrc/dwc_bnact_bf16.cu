// dwc_bnact_bf16.cu -- BN + Act + forward DWC on the row-streaming kernel, bf16 inputs.
#include "dwc_rows.cuh"

namespace dwc {
cudaError_t launch_rows_bnact_bf16(const RowConv& p, int stride) {
    if (stride == 1) return launch_rows_bnact_dispatch<__nv_bfloat16, 1>(p);
    if (stride == 2) return launch_rows_bnact_dispatch<__nv_bfloat16, 2>(p);
    return cudaErrorNotSupported;
}
}  // namespace dwc
