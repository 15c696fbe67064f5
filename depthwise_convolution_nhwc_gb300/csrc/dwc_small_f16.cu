// dwc_small_f16.cu -- small-map kernels, f16 inputs.
#include "dwc_small.cuh"

namespace dwc {
cudaError_t launch_small_rows_f16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_small_rows_o16_f16(p);
    return launch_small_rows_t<__half>(p);
}
cudaError_t launch_small_fgrad_f16(const FilterGrad& p) { return launch_small_fgrad_t<__half>(p); }
size_t small_fgrad_workspace_floats_f16(int N, int H, int W, int C, int OH, int OW, int FH, int FW,
                                      int pad) {
    return small_fgrad_workspace_t<__half>(N, H, W, C, OH, OW, FH, FW, pad);
}
}  // namespace dwc
