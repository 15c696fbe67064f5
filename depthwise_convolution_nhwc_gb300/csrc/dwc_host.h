// dwc_host.h -- internal host-side interface between the C ABI and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dwc {

enum ElemType { kF32 = 0, kBF16 = 1, kF16 = 2 };

// Devices a process may use with this library (per-device state is kept in fixed tables).
constexpr int kMaxDevices = 64;

inline int elem_bytes(int t) { return t == kF32 ? 4 : 2; }

// One stride-1 convolution over channels-last tensors, as the row-streaming kernel sees it:
//   out[n, oh, ow, c] = sum_{fh, fw} in[n, oh + fh - pad_h, ow + fw - pad_w, c] * filt(fh, fw, c)
// with filt(fh, fw, c) = w[fh, fw, c], or w[FH-1-fh, FW-1-fw, c] when flip is set
// (backward data).  in is N x H x W x C, out is N x OH x OW x C (fp32), w is FH x FW x C.
struct RowConv {
    const void* in;
    const void* w;
    void* out;              // fp32, or the input's 16-bit type when out_dtype says so
    int N, H, W, C;
    int OH, OW;
    int FH, FW;
    int pad_h, pad_w;
    bool flip;
    int dtype;
    cudaStream_t stream;
    unsigned int* status;
    // BN + Act fused in front of the forward pass (act < 0: plain DWC): per-channel batch
    // statistics and affine parameters (C floats each, device memory), epsilon, activation
    // (0 identity, 1 ReLU, 2 ReLU6).
    const float* bn_mean = nullptr;
    const float* bn_var = nullptr;
    const float* bn_gamma = nullptr;
    const float* bn_beta = nullptr;
    float bn_eps = 0.f;
    int act = -1;
    int out_dtype = kF32;   // kF32, or the input's type (kBF16 / kF16) for 16-bit outputs
    int c_lo = 0, c_hi = -1; // channel range a row-kernel launch covers (c_hi < 0: up to C)
    unsigned long long wait_ns = 0;  // limit of every wait in the kernel (0: the default)
    int stall = 0;           // fault injection: CTA 0 of the row kernel issues no copy
};

// Filter-gradient problem: dw[fh, fw, c] = sum_{n,oh,ow} x[n, oh+fh-pad, ow+fw-pad, c] * dy[n,oh,ow,c].
struct FilterGrad {
    const void* x;
    const void* dy;
    float* dw;
    int N, H, W, C;
    int OH, OW;
    int FH, FW;
    int pad;
    int dtype;
    float* workspace;        // partial sums, see filter_grad_workspace_floats
    size_t workspace_floats;
    cudaStream_t stream;
    unsigned int* status;
    unsigned long long wait_ns = 0;  // limit of every wait in the kernel (0: the default)
};

// General problem for the fallback kernels (any stride, any channel count or alignment).
struct GeneralConv {
    const void* a;     // x (fwd, bwd_filter) or dy (bwd_data)
    const void* b;     // w (fwd, bwd_data) or dy (bwd_filter)
    void* out;         // fp32 (always for the filter gradient), or 16-bit per out_dtype
    int N, H, W, C;    // forward input dims
    int OH, OW;
    int FH, FW;
    int stride, pad;
    int dtype;
    float* workspace;
    size_t workspace_floats;
    cudaStream_t stream;
    // BN + Act in front of the forward pass, as in RowConv (act < 0: none)
    const float* bn_mean = nullptr;
    const float* bn_var = nullptr;
    const float* bn_gamma = nullptr;
    const float* bn_beta = nullptr;
    float bn_eps = 0.f;
    int act = -1;
    int out_dtype = kF32;
};

// Limit of the waits inside kernels launched from now on (nanoseconds), and the one-shot
// fault-injection flag of the next row-kernel launch (both set through the C ABI).
unsigned long long wait_limit_ns();
int take_row_stall();

// Device properties cached per device.
struct DeviceInfo {
    int sm_count;
    int max_smem_optin;
};
const DeviceInfo& device_info();

// Stream-ordered scratch memory of one call, from a memory pool the library owns (one per
// device, created on first use; it keeps up to 512 MiB between calls).  scratch_free
// returns the block to the pool in stream order, after the work queued before it.
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream);
void scratch_free(void* p, cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda needed).
CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                      const cuuint32_t* box);

// Row-streaming kernels (stride 1, C even, 16-byte aligned tensors, filter sizes with a
// compiled instantiation).  Return cudaErrorNotSupported when no instantiation fits.
cudaError_t launch_rows_f32(const RowConv& p);
cudaError_t launch_rows_bf16(const RowConv& p);
cudaError_t launch_rows_f16(const RowConv& p);
bool rows_supported(int FH, int FW);
// Stripe (non-square) filters on the row kernel: any height from 1 to 255, odd widths 1..51,
// fp32 outputs; rows_supported / stripe_supported tell the square and the stripe shapes.
cudaError_t launch_rows_stripe_f32(const RowConv& p);
cudaError_t launch_rows_stripe_bf16(const RowConv& p);
cudaError_t launch_rows_stripe_f16(const RowConv& p);
bool stripe_supported(int FH, int FW);
cudaError_t launch_fgrad_stripe_f32(const FilterGrad& p);
cudaError_t launch_fgrad_stripe_bf16(const FilterGrad& p);
cudaError_t launch_fgrad_stripe_f16(const FilterGrad& p);
size_t fgrad_stripe_workspace_floats_f32(int N, int OH, int OW, int C, int FH, int FW);
size_t fgrad_stripe_workspace_floats_bf16(int N, int OH, int OW, int C, int FH, int FW);
size_t fgrad_stripe_workspace_floats_f16(int N, int OH, int OW, int C, int FH, int FW);
// Stride-2 forward row kernels (square filters of 3, 5 or 7 taps; RowConv's OH/OW are the
// strided output dims, pad_h/pad_w the forward pads).
cudaError_t launch_rows_s2_f32(const RowConv& p);
cudaError_t launch_rows_s2_bf16(const RowConv& p);
cudaError_t launch_rows_s2_f16(const RowConv& p);
// BN + Act + forward DWC on the row kernels (square filters of 3, 5 or 7 taps, stride 1 or
// 2, the layout rules of the fast paths; RowConv carries the BN parameters and act >= 0).
cudaError_t launch_rows_bnact_f32(const RowConv& p, int stride);
// BN + Act + forward as two passes (act(BN(x)) once per element into fp32 scratch, then the
// plain fp32 forward): 7x7 filters at stride 1, C a multiple of 4, rows of 28 or more.
bool bnact_split_serves(int FH, int FW, int stride, int C, int W);
cudaError_t launch_bnact_split(const RowConv& p, int stride);
cudaError_t launch_rows_bnact_bf16(const RowConv& p, int stride);
cudaError_t launch_rows_bnact_f16(const RowConv& p, int stride);

// The same launches writing 16-bit outputs of the input's type (RowConv / GeneralConv with
// out_dtype kBF16 or kF16); the entry points above route there themselves.
cudaError_t launch_rows_o16_bf16(const RowConv& p);
cudaError_t launch_rows_o16_f16(const RowConv& p);
cudaError_t launch_rows_s2_o16_bf16(const RowConv& p);
cudaError_t launch_rows_s2_o16_f16(const RowConv& p);
cudaError_t launch_small_rows_o16_bf16(const RowConv& p);
cudaError_t launch_small_rows_o16_f16(const RowConv& p);
cudaError_t launch_s2_bwd_data_o16_bf16(const GeneralConv& p);
cudaError_t launch_s2_bwd_data_o16_f16(const GeneralConv& p);

// Stride-2 backward data (square filters of 3, 5 or 7 taps, C even, 8-byte aligned
// tensors): a = dy, b = w, out = dx of the GeneralConv.
cudaError_t launch_s2_bwd_data_f32(const GeneralConv& p);
cudaError_t launch_s2_bwd_data_bf16(const GeneralConv& p);
cudaError_t launch_s2_bwd_data_f16(const GeneralConv& p);

cudaError_t launch_filter_grad_f32(const FilterGrad& p);
cudaError_t launch_filter_grad_bf16(const FilterGrad& p);
cudaError_t launch_filter_grad_f16(const FilterGrad& p);
bool filter_grad_supported(int FH, int FW);
// Workspace floats the filter-gradient kernels need for inputs of `dtype` (an ElemType;
// 0 if they cannot run this shape), and the CUDA-core kernel's share per dtype.
size_t filter_grad_workspace_floats(int N, int OH, int OW, int C, int FH, int FW, int dtype);
size_t fgrad_workspace_floats_f32(int N, int OH, int OW, int C, int FH, int FW);
size_t fgrad_workspace_floats_bf16(int N, int OH, int OW, int C, int FH, int FW);
size_t fgrad_workspace_floats_f16(int N, int OH, int OW, int C, int FH, int FW);

// Stride-2 filter gradient (square filters of 3, 5 or 7 taps; FilterGrad's OH/OW are the
// strided output dims) and its workspace floats (0 if it cannot run the shape).
cudaError_t launch_filter_grad_s2_f32(const FilterGrad& p);
cudaError_t launch_filter_grad_s2_bf16(const FilterGrad& p);
cudaError_t launch_filter_grad_s2_f16(const FilterGrad& p);
size_t filter_grad_s2_workspace_floats(int N, int OH, int OW, int C, int FH, int FW, int dtype);
size_t fgrad_s2_workspace_floats_f32(int N, int OH, int OW, int C, int FH, int FW);
size_t fgrad_s2_workspace_floats_bf16(int N, int OH, int OW, int C, int FH, int FW);
size_t fgrad_s2_workspace_floats_f16(int N, int OH, int OW, int C, int FH, int FW);

// Small-map kernels (H, W, OH, OW <= 16; stride 1; C a multiple of 16 bytes; 16-byte
// aligned tensors): whole images staged per 32-channel block, only the taps that can meet
// the image are run.  cudaErrorNotSupported when the map is larger or the filter small
// enough for the other kernels to be faster; small_map_serves tells the forward /
// backward-data choice, a nonzero small_fgrad_workspace_floats_* the filter-gradient one.
bool small_map_serves(int H, int W, int OH, int OW, int FW, int pad_w);
// Whether the filter gradient of a 7x7 map ("same" padding, stride 1) runs as one launch
// (the cluster form, 3 taps) rather than a kernel and a slice sum.
bool tiny_fgrad_single_launch(int dtype, int N, int H, int W, int C, int FH, int FW, int pad);
cudaError_t launch_small_rows_f32(const RowConv& p);
cudaError_t launch_small_rows_bf16(const RowConv& p);
cudaError_t launch_small_rows_f16(const RowConv& p);
cudaError_t launch_small_fgrad_f32(const FilterGrad& p);
cudaError_t launch_small_fgrad_bf16(const FilterGrad& p);
cudaError_t launch_small_fgrad_f16(const FilterGrad& p);
size_t small_fgrad_workspace_floats_f32(int N, int H, int W, int C, int OH, int OW, int FH, int FW, int pad);
size_t small_fgrad_workspace_floats_bf16(int N, int H, int W, int C, int OH, int OW, int FH, int FW, int pad);
size_t small_fgrad_workspace_floats_f16(int N, int H, int W, int C, int OH, int OW, int FH, int FW, int pad);

// tcgen05 tensor-core forward / backward-data kernels (16-bit inputs, stride 1; fp32 or the
// input's 16-bit type as output); cudaErrorNotSupported when the shape does not fit.
cudaError_t launch_tc_rows_bf16(const RowConv& p);
cudaError_t launch_tc_rows_f16(const RowConv& p);
bool tc_rows_fits(const RowConv& p);
// Where the tcgen05 kernel is the one to run (timed against the row, warp-level MMA and
// small-map kernels, bf16, fp32 outputs): from 9 taps on rows of at least 28 outputs
// (64x56x56x128: 100 against 115 us at 9 taps, 111 against 162 at 11, 112 against 220 at 13;
// 64x28x28x256: 59 against 66 us at 9 taps, at 7 the row kernel 46 against 58), from 17 taps
// on rows of 17 to 27 outputs, and from 13 taps on rows of 14 to 16 outputs where the batch
// carries enough channel planes (64x14x14x512: 55 against 74 us on the small-map kernel at 13
// taps, 116 against 137 at 31; 32x14x14x512 31x31 a tie; at 9 taps the row kernel 45 against
// 52); 7x7 maps stay on the small-map kernel (64x7x7x1024 31x31: 33 against 262 us).
inline bool tc_rows_wanted(const RowConv& p) {
    return (p.FW >= 9 && p.OW >= 28) || (p.FW >= 17 && p.OW >= 17) ||
           (p.FW >= 13 && p.OW >= 14 && static_cast<long long>(p.N) * p.C >= 16384);
}
// Kernel launches of a tcgen05 call: the preparation and the main kernel (0 when the shape
// has no plan).
int tc_rows_launches(const RowConv& p);
// tc_rows_wanted and a launch plan exists.
inline bool tc_rows_preferred(const RowConv& p) {
    return (p.dtype == kBF16 || p.dtype == kF16) && tc_rows_wanted(p) && tc_rows_fits(p);
}

// Kernel family a 16-bit forward / backward-data call of this shape runs on (kFamily*), and
// whether the filter gradient of 16-bit inputs runs on the tensor-core kernel.
enum KernelFamily { kFamilyGeneral = 0, kFamilyCudaCore = 1, kFamilyTcgen05 = 2, kFamilySmall = 3,
                    kFamilyMmaSync = 4 };
int tensor_core_rows(const RowConv& p);
// Family preference for 16-bit forward / backward-data calls and filter gradients (tests and
// kernel comparisons; 0 = automatic choice), set through dwc_testing_prefer_family.
int family_preference();
// Filter rows per MMA of the tcgen05 kernel (tests): 0 = the plan's choice, 1 = one, 2 = pairs;
// set through dwc_testing_tc_row_pairs.
int tc_row_pairs_mode();
bool tensor_core_fgrad(int N, int C, int OH, int OW, int FH, int FW);
// tcgen05 filter gradient (16-bit inputs, square filters; scratch for the stacked copies of x
// and dy comes from the library's pool): cudaErrorNotSupported when the shape does not fit.
cudaError_t launch_tc_fgrad_bf16(const FilterGrad& p);
cudaError_t launch_tc_fgrad_f16(const FilterGrad& p);
bool tc_fgrad_fits(const FilterGrad& p);
// Where the tcgen05 filter gradient is the one to run (the automatic choice; timed against the
// warp-level MMA and CUDA-core kernels, bf16): from 13 taps on rows of at least 44 outputs
// (wide tiles) or of 17 to 32 outputs (narrow tiles, up to 33 taps).  Its work grows with the
// rows, columns and filter height but not the width (the whole x band of a dy tile is
// multiplied), so small filters stay elsewhere (64x56x56x128: 205 against 229 us at 13 taps,
// 166 against 158 at 11; 64x112x112x64 13x13: 358 against 426; 64x28x28x256: 113 against 131
// us at 13 taps, 198 against 338 at 31; 32x40x40x128 31x31 a tie on a wide tile).
inline bool tc_fgrad_wanted(int FW, int OW) {
    return FW >= 13 && (OW >= 44 || (OW >= 17 && OW <= 32 && FW <= 33));
}
// The tcgen05 filter gradient serves this 16-bit call: the automatic choice or the family
// preference (tcgen05 forced: 2; other families: never).
bool tc_fgrad_taken(const FilterGrad& p);

// The argument and pointer checks of dwc_bwd_filter without its workspace checks; returns a
// dwc_status_t value (0 = DWC_OK).
int validate_bwd_filter(const void* x, const void* dy, const float* dw, int N, int H, int W,
                        int C, int FH, int FW, int stride, int pad, int dtype);

// Fallback kernels.
cudaError_t launch_general_fwd(const GeneralConv& p);
cudaError_t launch_general_bwd_data(const GeneralConv& p);
cudaError_t launch_general_bwd_filter(const GeneralConv& p);
size_t general_bwd_filter_workspace_floats(int N, int OH, int C, int FH, int FW);

// Deterministic fixed-order sum of `slices` partial filter gradients laid out as
// [slices][count] into out[count].
cudaError_t launch_reduce_slices(const float* part, int slices, size_t count, float* out,
                                 cudaStream_t stream);

}  // namespace dwc
