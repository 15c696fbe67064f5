// dwc_bnact_f32.cu -- BN + Act + forward DWC on the row-streaming kernel, f32 inputs.
#include "dwc_rows.cuh"

namespace dwc {
cudaError_t launch_rows_bnact_f32(const RowConv& p, int stride) {
    if (stride == 1) return launch_rows_bnact_dispatch<float, 1>(p);
    if (stride == 2) return launch_rows_bnact_dispatch<float, 2>(p);
    return cudaErrorNotSupported;
}
}  // namespace dwc
