// dwc_tc_bf16.cu -- tcgen05 tensor-core forward / backward-data kernels, bf16 inputs (fp32 or
// bf16 outputs).
#include "dwc_tc.cuh"

namespace dwc {
cudaError_t launch_tc_rows_bf16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_tc_rows<__nv_bfloat16, __nv_bfloat16>(p);
    return launch_tc_rows<__nv_bfloat16, float>(p);
}
bool tc_rows_fits(const RowConv& p) {
    TcPlan P;
    return tc_plan(p, P);
}
int tc_rows_launches(const RowConv& p) {
    TcPlan P;
    if (!tc_plan(p, P) || P.a.units == 0) return 0;
    return 2;
}
}  // namespace dwc
