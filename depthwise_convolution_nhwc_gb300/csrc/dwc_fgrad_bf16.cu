// dwc_fgrad_bf16.cu -- filter-gradient kernels, bf16 inputs.
#include "dwc_fgrad.cuh"

namespace dwc {
cudaError_t launch_filter_grad_bf16(const FilterGrad& p) { return launch_fgrad_dispatch<__nv_bfloat16>(p); }
}  // namespace dwc
