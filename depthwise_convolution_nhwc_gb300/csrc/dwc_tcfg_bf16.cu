// dwc_tcfg_bf16.cu -- tcgen05 tensor-core filter gradient, bf16 inputs.
#include "dwc_tc_fgrad.cuh"

namespace dwc {
cudaError_t launch_tc_fgrad_bf16(const FilterGrad& p) { return launch_tc_fgrad<__nv_bfloat16>(p); }
bool tc_fgrad_fits(const FilterGrad& p) {
    TcFgPlan P;
    return tc_fgrad_plan(p, P);
}
}  // namespace dwc
