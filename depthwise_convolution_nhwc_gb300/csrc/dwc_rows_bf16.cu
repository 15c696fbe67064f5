// dwc_rows_bf16.cu -- forward / backward-data kernels, bf16 inputs (the tcgen05 kernel where
// tc_rows_wanted says so, the warp-level MMA kernel or the row-streaming kernel otherwise).
#include "dwc_mma.cuh"
#include "dwc_s2data.cuh"

namespace dwc {
cudaError_t launch_rows_bf16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_rows_o16_bf16(p);
    return launch_rows_or_mma<__nv_bfloat16>(p);
}

int tensor_core_rows(const RowConv& p) {
    // the choice of launch_rows_or_mma (no 16-bit input shape differs between bf16 and fp16)
    const int pref = family_preference();
    if (((pref == 0 && tc_rows_wanted(p)) || pref == kFamilyTcgen05) && tc_rows_fits(p))
        return kFamilyTcgen05;
    MmaArgs a;
    size_t smem = 0;
    if (((pref == 0 && mma_rows_wanted(p)) || pref == kFamilyMmaSync) && mma_plan(p, a, smem))
        return kFamilyMmaSync;
    return kFamilyCudaCore;
}
cudaError_t launch_rows_s2_bf16(const RowConv& p) {
    if (p.out_dtype != kF32) return launch_rows_s2_o16_bf16(p);
    return launch_rows_s2_dispatch<__nv_bfloat16>(p);
}
cudaError_t launch_s2_bwd_data_bf16(const GeneralConv& p) {
    if (p.out_dtype != kF32) return launch_s2_bwd_data_o16_bf16(p);
    return launch_s2_bwd_data_dispatch<__nv_bfloat16>(p);
}
}  // namespace dwc
