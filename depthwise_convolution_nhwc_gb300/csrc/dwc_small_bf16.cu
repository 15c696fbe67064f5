// dwc_small_bf16.cu -- small-map kernels, bf16 inputs.
#include "dwc_small.cuh"

namespace dwc {
cudaError_t launch_small_rows_bf16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_small_rows_o16_bf16(p);
    return launch_small_rows_t<__nv_bfloat16>(p);
}
cudaError_t launch_small_fgrad_bf16(const FilterGrad& p) { return launch_small_fgrad_t<__nv_bfloat16>(p); }
size_t small_fgrad_workspace_floats_bf16(int N, int H, int W, int C, int OH, int OW, int FH, int FW,
                                      int pad) {
    return small_fgrad_workspace_t<__nv_bfloat16>(N, H, W, C, OH, OW, FH, FW, pad);
}
}  // namespace dwc
