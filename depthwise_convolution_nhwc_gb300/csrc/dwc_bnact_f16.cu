// dwc_bnact_f16.cu -- BN + Act + forward DWC on the row-streaming kernel, f16 inputs.
#include "dwc_rows.cuh"

namespace dwc {
cudaError_t launch_rows_bnact_f16(const RowConv& p, int stride) {
    if (stride == 1) return launch_rows_bnact_dispatch<__half, 1>(p);
    if (stride == 2) return launch_rows_bnact_dispatch<__half, 2>(p);
    return cudaErrorNotSupported;
}
}  // namespace dwc
