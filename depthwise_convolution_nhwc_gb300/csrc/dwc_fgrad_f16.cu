// dwc_fgrad_f16.cu -- filter-gradient kernels, f16 inputs.
#include "dwc_fgrad.cuh"

namespace dwc {
cudaError_t launch_filter_grad_f16(const FilterGrad& p) { return launch_fgrad_dispatch<__half>(p); }
}  // namespace dwc
