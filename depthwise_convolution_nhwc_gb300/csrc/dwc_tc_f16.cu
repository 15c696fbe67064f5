// dwc_tc_f16.cu -- tcgen05 tensor-core forward / backward-data kernels, fp16 inputs (fp32 or
// fp16 outputs).
#include "dwc_tc.cuh"

namespace dwc {
cudaError_t launch_tc_rows_f16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_tc_rows<__half, __half>(p);
    return launch_tc_rows<__half, float>(p);
}
}  // namespace dwc
