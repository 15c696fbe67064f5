// dwc_rows_bf16.cu -- forward / backward-data kernels, bf16 inputs (tensor-core kernel for
// filters from 9 taps, row-streaming kernel below).
#include "dwc_mma.cuh"

namespace dwc {
cudaError_t launch_rows_bf16(const RowConv& p) { return launch_rows_or_mma<__nv_bfloat16>(p); }
}  // namespace dwc
