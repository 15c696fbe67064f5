// dwc_small_f32.cu -- small-map kernels, f32 inputs.
#include "dwc_small.cuh"

namespace dwc {
cudaError_t launch_small_rows_f32(const RowConv& p) { return launch_small_rows_t<float>(p); }
cudaError_t launch_small_fgrad_f32(const FilterGrad& p) { return launch_small_fgrad_t<float>(p); }
size_t small_fgrad_workspace_floats_f32(int N, int H, int W, int C, int OH, int OW, int FH, int FW,
                                      int pad) {
    return small_fgrad_workspace_t<float>(N, H, W, C, OH, OW, FH, FW, pad);
}

bool tiny_fgrad_single_launch(int dtype, int N, int H, int W, int C, int FH, int FW, int pad) {
    if (!tiny_shape(H, W, H, W, FH, FW, pad, pad)) return false;
    switch (dtype) {
        case kF32: return tiny_fgrad_cluster_fits<float>(N, C, FH);
        case kBF16: return tiny_fgrad_cluster_fits<__nv_bfloat16>(N, C, FH);
        default: return tiny_fgrad_cluster_fits<__half>(N, C, FH);
    }
}

bool small_map_serves(int H, int W, int OH, int OW, int FW, int pad_w) {
    if (tiny_shape(H, W, OH, OW, FW, FW, pad_w, pad_w)) return true;
    int maxw = 0, dr = 0;
    return small_rows_wanted(W, OW, FW) && small_shape(H, W, OH, OW, FW, pad_w, maxw, dr);
}
}  // namespace dwc
