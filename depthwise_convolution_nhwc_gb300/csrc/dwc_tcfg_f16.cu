// dwc_tcfg_f16.cu -- tcgen05 tensor-core filter gradient, f16 inputs.
#include "dwc_tc_fgrad.cuh"

namespace dwc {
cudaError_t launch_tc_fgrad_f16(const FilterGrad& p) { return launch_tc_fgrad<__half>(p); }
}  // namespace dwc
