// dwc_api.cu -- the C ABI declared in include/dwc.h: argument validation, choice between
// the fast and the general kernels, TMA descriptor encoding and the device status word.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <climits>
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/dwc.h"
#include "../../include/dwc_testing.h"
#include "dwc_host.h"

namespace dwc {

namespace {

// Status word the kernels set when a wait runs out of time (one per device, in this
// module's global memory; its address is looked up once per device).
__device__ unsigned int g_status_word;

struct PerDevice {
    bool ready = false;
    DeviceInfo info{};
    unsigned int* status = nullptr;
    cudaMemPool_t pool = nullptr;   // scratch of the kernels that need some (created on use)
};

PerDevice g_dev[kMaxDevices];
std::mutex g_mu;
std::atomic<unsigned long long> g_wait_limit_ns{0};  // 0: the kernels' default
std::atomic<int> g_row_stall{0};
std::atomic<int> g_family_pref{0};
std::atomic<int> g_tc_pairs{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// One-time set-up for the current device; nullptr if CUDA is unusable.
PerDevice* device_state() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    PerDevice& s = g_dev[d];
    if (!s.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, d) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        s.info.sm_count = prop.multiProcessorCount;
        s.info.max_smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) {
            (void)cudaGetLastError();  // do not leave the failure to the next launch check
            return nullptr;
        }
        s.status = static_cast<unsigned int*>(addr);
        s.ready = true;
    }
    return &s;
}

}  // namespace

// Memory the pool keeps between calls instead of returning it to the driver.
constexpr uint64_t kScratchKeepBytes = 512ull << 20;

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream) {
    *p = nullptr;
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return cudaErrorInvalidDevice;
    PerDevice* s = device_state();
    if (s == nullptr) return cudaErrorInvalidDevice;
    cudaMemPool_t pool = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (s->pool == nullptr) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = d;
            cudaMemPool_t created = nullptr;
            if (cudaMemPoolCreate(&created, &props) != cudaSuccess) return cudaErrorMemoryAllocation;
            uint64_t keep = kScratchKeepBytes;
            (void)cudaMemPoolSetAttribute(created, cudaMemPoolAttrReleaseThreshold, &keep);
            s->pool = created;
        }
        pool = s->pool;
    }
    return cudaMallocFromPoolAsync(p, bytes, pool, stream);
}

void scratch_free(void* p, cudaStream_t stream) {
    if (p != nullptr) (void)cudaFreeAsync(p, stream);
}

const DeviceInfo& device_info() {
    static const DeviceInfo fallback{152, 232448};  // GB300, used only when no device answers
    PerDevice* s = device_state();
    return s ? s->info : fallback;
}

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                      const cuuint32_t* box) {
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_encode == nullptr) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return CUDA_ERROR_NOT_FOUND;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return g_encode(map, type, rank, base, dims, strides_bytes, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int take_row_stall() { return g_row_stall.exchange(0, std::memory_order_acq_rel); }

int family_preference() { return g_family_pref.load(std::memory_order_relaxed); }

int tc_row_pairs_mode() { return g_tc_pairs.load(std::memory_order_relaxed); }

static unsigned int* status_word() {
    PerDevice* s = device_state();
    return s ? s->status : nullptr;
}

}  // namespace dwc

using namespace dwc;

namespace {

enum Pass { kPassFwd = 0, kPassBwdData = 1, kPassBwdFilter = 2 };

int out_dim(int n_in, int f, int s, int p) {
    const long long num = static_cast<long long>(n_in) + 2LL * p - f;
    if (s < 1 || num < 0) return 0;
    return static_cast<int>(num / s) + 1;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Problem {
    int N, H, W, C, FH, FW, s, p, OH, OW, e, dtype;
};

// Host-side validation shared by every entry point.
dwc_status_t check_problem(int N, int H, int W, int C, int FH, int FW, int stride, int pad,
                           dwc_dtype_t dtype, Problem& P) {
    if (dtype != DWC_F32 && dtype != DWC_BF16 && dtype != DWC_F16) return DWC_ERR_INVALID_ARG;
    if (N < 0 || C < 0 || H < 1 || W < 1 || FH < 1 || FW < 1 || stride < 1 || pad < 0)
        return DWC_ERR_INVALID_ARG;
    P.N = N; P.H = H; P.W = W; P.C = C; P.FH = FH; P.FW = FW; P.s = stride; P.p = pad;
    P.OH = out_dim(H, FH, stride, pad);
    P.OW = out_dim(W, FW, stride, pad);
    if (P.OH < 1 || P.OW < 1) return DWC_ERR_INVALID_ARG;
    P.e = dtype == DWC_F32 ? 4 : 2;
    P.dtype = static_cast<int>(dtype);
    const long long in_elems = static_cast<long long>(N) * H * W * C;
    const long long out_elems = static_cast<long long>(N) * P.OH * P.OW * C;
    if (in_elems > (1LL << 40) || out_elems > (1LL << 40) ||
        static_cast<long long>(FH) * FW * C > (1LL << 36) ||
        static_cast<long long>(N) * P.OH > INT_MAX / 2 ||
        static_cast<long long>(N) * H > INT_MAX / 2)
        return DWC_ERR_UNSUPPORTED;
    return DWC_OK;
}

dwc_status_t check_pointers(const Problem& P, const void* a, long long a_elems, const void* b,
                            long long b_elems, const void* out, long long out_elems,
                            int out_bytes = 4) {
    if ((a_elems > 0 && a == nullptr) || (b_elems > 0 && b == nullptr) ||
        (out_elems > 0 && out == nullptr))
        return DWC_ERR_INVALID_ARG;
    if (!aligned(a, P.e) || !aligned(b, P.e) || !aligned(out, out_bytes)) return DWC_ERR_ALIGNMENT;
    return DWC_OK;
}

// Output type of a forward / backward-data call: fp32, or the input's own 16-bit type.
bool valid_out_dtype(dwc_dtype_t dtype, dwc_dtype_t out_dtype) {
    return out_dtype == DWC_F32 || (out_dtype == dtype && dtype != DWC_F32);
}

bool fast_eligible(const Problem& P, const void* a, const void* b, const void* out) {
    if (P.s != 1) return false;
    if (!rows_supported(P.FH, P.FW) && !stripe_supported(P.FH, P.FW)) return false;
    if (P.C % (16 / P.e) != 0) return false;  // TMA strides must be multiples of 16 bytes
    for (const void* q : {a, b, out})
        if (q != nullptr && !aligned(q, 16)) return false;
    return true;
}

// Stride-2 fast paths (forward, backward data, filter gradient): square odd filters of 3 to
// 13 taps, same layout rules.
bool fast_s2_eligible(const Problem& P, const void* a, const void* b, const void* out) {
    const int F = P.FH;
    if (P.s != 2 || P.FH != P.FW || F < 3 || (F & 1) == 0 || F > 13) return false;
    if (P.C % (16 / P.e) != 0) return false;
    for (const void* q : {a, b, out})
        if (q != nullptr && !aligned(q, 16)) return false;
    return true;
}

// BN + Act + forward fast path: square 3x3, 5x5 or 7x7 filters at stride 1 or 2.
bool bnact_fast_eligible(const Problem& P, const void* a, const void* b, const void* out) {
    if (P.FH != P.FW || (P.FH != 3 && P.FH != 5 && P.FH != 7)) return false;
    return P.s == 1 ? fast_eligible(P, a, b, out) : fast_s2_eligible(P, a, b, out);
}

cudaError_t launch_rows_bnact(const RowConv& rc, int stride) {
    if (bnact_split_serves(rc.FH, rc.FW, stride, rc.C, rc.W)) {
        const cudaError_t err = launch_bnact_split(rc, stride);
        if (err != cudaErrorNotSupported) return err;
    }
    switch (rc.dtype) {
        case kF32: return launch_rows_bnact_f32(rc, stride);
        case kBF16: return launch_rows_bnact_bf16(rc, stride);
        default: return launch_rows_bnact_f16(rc, stride);
    }
}

dwc_status_t map_cuda(cudaError_t err) { return err == cudaSuccess ? DWC_OK : DWC_ERR_CUDA; }

cudaError_t launch_rows(const RowConv& rc) {
    if (rc.FH != rc.FW) {
        // stripe filter: the tensor-core kernel where it serves 16-bit inputs, else the row
        // kernel with the filter height read at run time
        cudaError_t err = cudaErrorNotSupported;
        if (rc.dtype == kBF16) err = launch_rows_bf16(rc);
        if (rc.dtype == kF16) err = launch_rows_f16(rc);
        if (err != cudaErrorNotSupported) return err;
        (void)cudaGetLastError();
        switch (rc.dtype) {
            case kF32: return launch_rows_stripe_f32(rc);
            case kBF16: return launch_rows_stripe_bf16(rc);
            default: return launch_rows_stripe_f16(rc);
        }
    }
    // (a family preference for 16-bit inputs, and the shapes the tcgen05 kernel takes,
    // bypass the small-map kernels)
    const bool pref16 = rc.dtype != kF32 && family_preference() != 0;
    const bool tc16 = !pref16 && tc_rows_preferred(rc);
    if (!pref16 && !tc16 && small_map_serves(rc.H, rc.W, rc.OH, rc.OW, rc.FW, rc.pad_w)) {
        cudaError_t err;
        switch (rc.dtype) {
            case kF32: err = launch_small_rows_f32(rc); break;
            case kBF16: err = launch_small_rows_bf16(rc); break;
            default: err = launch_small_rows_f16(rc); break;
        }
        if (err != cudaErrorNotSupported) return err;
    }
    switch (rc.dtype) {
        case kF32: return launch_rows_f32(rc);
        case kBF16: return launch_rows_bf16(rc);
        default: return launch_rows_f16(rc);
    }
}

cudaError_t launch_fgrad(const FilterGrad& fg) {
    if (fg.FH == fg.FW) {
        cudaError_t err;
        switch (fg.dtype) {
            case kF32: err = launch_small_fgrad_f32(fg); break;
            case kBF16: err = launch_small_fgrad_bf16(fg); break;
            default: err = launch_small_fgrad_f16(fg); break;
        }
        if (err != cudaErrorNotSupported) return err;
    }
    switch (fg.dtype) {
        case kF32: return launch_filter_grad_f32(fg);
        case kBF16: return launch_filter_grad_bf16(fg);
        default: return launch_filter_grad_f16(fg);
    }
}

cudaError_t launch_s2_bwd_data(const GeneralConv& gc) {
    switch (gc.dtype) {
        case kF32: return launch_s2_bwd_data_f32(gc);
        case kBF16: return launch_s2_bwd_data_bf16(gc);
        default: return launch_s2_bwd_data_f16(gc);
    }
}

cudaError_t launch_fgrad_s2(const FilterGrad& fg) {
    switch (fg.dtype) {
        case kF32: return launch_filter_grad_s2_f32(fg);
        case kBF16: return launch_filter_grad_s2_bf16(fg);
        default: return launch_filter_grad_s2_f16(fg);
    }
}

size_t small_fgrad_floats(const Problem& P) {
    if (P.FH != P.FW) return 0;
    switch (P.dtype) {
        case kF32: return small_fgrad_workspace_floats_f32(P.N, P.H, P.W, P.C, P.OH, P.OW, P.FH, P.FW, P.p);
        case kBF16: return small_fgrad_workspace_floats_bf16(P.N, P.H, P.W, P.C, P.OH, P.OW, P.FH, P.FW, P.p);
        default: return small_fgrad_workspace_floats_f16(P.N, P.H, P.W, P.C, P.OH, P.OW, P.FH, P.FW, P.p);
    }
}

// Workspace of the fast filter-gradient kernels: the largest of the kernels that may serve
// the call (the small-map kernel falls back to the others if its launch is refused).
size_t fast_fgrad_floats(const Problem& P) {
    return std::max(filter_grad_workspace_floats(P.N, P.OH, P.OW, P.C, P.FH, P.FW, P.dtype),
                    small_fgrad_floats(P));
}

dwc_status_t fwd_impl(const void* x, const void* w, void* y, int N, int H, int W, int C, int FH,
                      int FW, int stride, int pad, dwc_dtype_t dtype, dwc_dtype_t out_dtype,
                      dwc_stream_t stream) {
    Problem P;
    dwc_status_t st = check_problem(N, H, W, C, FH, FW, stride, pad, dtype, P);
    if (st != DWC_OK) return st;
    if (!valid_out_dtype(dtype, out_dtype)) return DWC_ERR_INVALID_ARG;
    const int od = static_cast<int>(out_dtype);
    const long long nx = static_cast<long long>(N) * H * W * C;
    const long long ny = static_cast<long long>(N) * P.OH * P.OW * C;
    st = check_pointers(P, x, nx, w, static_cast<long long>(FH) * FW * C, y, ny, elem_bytes(od));
    if (st != DWC_OK) return st;
    if (ny == 0) return DWC_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (fast_eligible(P, x, w, y)) {
        RowConv rc{x, w, y, N, H, W, C, P.OH, P.OW, FH, FW, pad, pad, false, P.dtype, s, status_word()};
        rc.out_dtype = od;
        rc.wait_ns = wait_limit_ns();
        rc.stall = take_row_stall();
        const cudaError_t err = launch_rows(rc);
        if (err != cudaErrorNotSupported) return map_cuda(err);
        (void)cudaGetLastError();
    } else if (fast_s2_eligible(P, x, w, y)) {
        RowConv rc{x, w, y, N, H, W, C, P.OH, P.OW, FH, FW, pad, pad, false, P.dtype, s, status_word()};
        rc.out_dtype = od;
        rc.wait_ns = wait_limit_ns();
        cudaError_t err;
        switch (rc.dtype) {
            case kF32: err = launch_rows_s2_f32(rc); break;
            case kBF16: err = launch_rows_s2_bf16(rc); break;
            default: err = launch_rows_s2_f16(rc); break;
        }
        if (err != cudaErrorNotSupported) return map_cuda(err);
        (void)cudaGetLastError();
    }
    GeneralConv gc{x, w, y, N, H, W, C, P.OH, P.OW, FH, FW, stride, pad, P.dtype, nullptr, 0, s};
    gc.out_dtype = od;
    return map_cuda(launch_general_fwd(gc));
}

dwc_status_t bwd_data_impl(const void* dy, const void* w, void* dx, int N, int H, int W, int C,
                           int FH, int FW, int stride, int pad, dwc_dtype_t dtype,
                           dwc_dtype_t out_dtype, dwc_stream_t stream) {
    Problem P;
    dwc_status_t st = check_problem(N, H, W, C, FH, FW, stride, pad, dtype, P);
    if (st != DWC_OK) return st;
    if (!valid_out_dtype(dtype, out_dtype)) return DWC_ERR_INVALID_ARG;
    const int od = static_cast<int>(out_dtype);
    const long long ndy = static_cast<long long>(N) * P.OH * P.OW * C;
    const long long ndx = static_cast<long long>(N) * H * W * C;
    st = check_pointers(P, dy, ndy, w, static_cast<long long>(FH) * FW * C, dx, ndx, elem_bytes(od));
    if (st != DWC_OK) return st;
    if (ndx == 0) return DWC_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (fast_eligible(P, dy, w, dx)) {
        // stride 1: forward pass over dy with the filter rotated by 180 degrees and the
        // complementary padding FH-1-pad (rows) / FW-1-pad (columns); output is H x W.
        RowConv rc{dy, w, dx, N, P.OH, P.OW, C, H, W, FH, FW, FH - 1 - pad, FW - 1 - pad, true,
                   P.dtype, s, status_word()};
        rc.out_dtype = od;
        rc.wait_ns = wait_limit_ns();
        rc.stall = take_row_stall();
        const cudaError_t err = launch_rows(rc);
        if (err != cudaErrorNotSupported) return map_cuda(err);
        (void)cudaGetLastError();
    }
    GeneralConv gc{dy, w, dx, N, H, W, C, P.OH, P.OW, FH, FW, stride, pad, P.dtype, nullptr, 0, s};
    gc.out_dtype = od;
    if (fast_s2_eligible(P, dy, w, dx)) {
        const cudaError_t err = launch_s2_bwd_data(gc);
        if (err != cudaErrorNotSupported) return map_cuda(err);
        (void)cudaGetLastError();
    }
    return map_cuda(launch_general_bwd_data(gc));
}

}  // namespace

extern "C" {

dwc_status_t dwc_fwd(const void* x, const void* w, float* y, int N, int H, int W, int C, int FH,
                     int FW, int stride, int pad, dwc_dtype_t dtype, dwc_stream_t stream) {
    return fwd_impl(x, w, y, N, H, W, C, FH, FW, stride, pad, dtype, DWC_F32, stream);
}

dwc_status_t dwc_fwd_ex(const void* x, const void* w, void* y, int N, int H, int W, int C, int FH,
                        int FW, int stride, int pad, dwc_dtype_t dtype, dwc_dtype_t out_dtype,
                        dwc_stream_t stream) {
    return fwd_impl(x, w, y, N, H, W, C, FH, FW, stride, pad, dtype, out_dtype, stream);
}

dwc_status_t dwc_bwd_data_ex(const void* dy, const void* w, void* dx, int N, int H, int W, int C,
                             int FH, int FW, int stride, int pad, dwc_dtype_t dtype,
                             dwc_dtype_t out_dtype, dwc_stream_t stream) {
    return bwd_data_impl(dy, w, dx, N, H, W, C, FH, FW, stride, pad, dtype, out_dtype, stream);
}

dwc_status_t dwc_fwd_bn_act(const void* x, const float* mean, const float* var,
                            const float* gamma, const float* beta, float eps, dwc_act_t act,
                            const void* w, float* y, int N, int H, int W, int C, int FH, int FW,
                            int stride, int pad, dwc_dtype_t dtype, dwc_stream_t stream) {
    Problem P;
    dwc_status_t st = check_problem(N, H, W, C, FH, FW, stride, pad, dtype, P);
    if (st != DWC_OK) return st;
    if (act != DWC_ACT_NONE && act != DWC_ACT_RELU && act != DWC_ACT_RELU6)
        return DWC_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !(eps < INFINITY)) return DWC_ERR_INVALID_ARG;
    const long long nx = static_cast<long long>(N) * H * W * C;
    const long long ny = static_cast<long long>(N) * P.OH * P.OW * C;
    st = check_pointers(P, x, nx, w, static_cast<long long>(FH) * FW * C, y, ny);
    if (st != DWC_OK) return st;
    for (const float* q : {mean, var, gamma, beta}) {
        if (C > 0 && q == nullptr) return DWC_ERR_INVALID_ARG;
        if (!aligned(q, 4)) return DWC_ERR_ALIGNMENT;
    }
    if (ny == 0) return DWC_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (bnact_fast_eligible(P, x, w, y)) {
        RowConv rc{x, w, y, N, H, W, C, P.OH, P.OW, FH, FW, pad, pad, false, P.dtype, s, status_word(),
                   mean, var, gamma, beta, eps, static_cast<int>(act)};
        rc.wait_ns = wait_limit_ns();
        const cudaError_t err = launch_rows_bnact(rc, stride);
        if (err != cudaErrorNotSupported) return map_cuda(err);
        (void)cudaGetLastError();
    }
    GeneralConv gc{x, w, y, N, H, W, C, P.OH, P.OW, FH, FW, stride, pad, P.dtype, nullptr, 0, s,
                   mean, var, gamma, beta, eps, static_cast<int>(act)};
    return map_cuda(launch_general_fwd(gc));
}

dwc_status_t dwc_bwd_data(const void* dy, const void* w, float* dx, int N, int H, int W, int C,
                          int FH, int FW, int stride, int pad, dwc_dtype_t dtype,
                          dwc_stream_t stream) {
    return bwd_data_impl(dy, w, dx, N, H, W, C, FH, FW, stride, pad, dtype, DWC_F32, stream);
}

}  // extern "C"

namespace dwc {

// The argument and pointer checks of dwc_bwd_filter (without the workspace ones), for the
// entry points that supply the workspace themselves.
int validate_bwd_filter(const void* x, const void* dy, const float* dw, int N, int H, int W,
                        int C, int FH, int FW, int stride, int pad, int dtype) {
    Problem P;
    const dwc_status_t st = check_problem(N, H, W, C, FH, FW, stride, pad,
                                          static_cast<dwc_dtype_t>(dtype), P);
    if (st != DWC_OK) return st;
    return check_pointers(P, x, static_cast<long long>(N) * H * W * C, dy,
                          static_cast<long long>(N) * P.OH * P.OW * C, dw,
                          static_cast<long long>(FH) * FW * C);
}

}  // namespace dwc

extern "C" {

size_t dwc_bwd_filter_workspace_size(int N, int H, int W, int C, int FH, int FW, int stride,
                                     int pad, dwc_dtype_t dtype) {
    Problem P;
    if (check_problem(N, H, W, C, FH, FW, stride, pad, dtype, P) != DWC_OK) return 0;
    size_t floats = general_bwd_filter_workspace_floats(N, P.OH, C, FH, FW);
    if (fast_eligible(P, nullptr, nullptr, nullptr)) floats = std::max(floats, fast_fgrad_floats(P));
    if (fast_s2_eligible(P, nullptr, nullptr, nullptr))
        floats = std::max(floats, filter_grad_s2_workspace_floats(N, P.OH, P.OW, C, FH, FW, P.dtype));
    return floats * sizeof(float);
}

dwc_status_t dwc_bwd_filter(const void* x, const void* dy, float* dw, int N, int H, int W, int C,
                            int FH, int FW, int stride, int pad, dwc_dtype_t dtype,
                            void* workspace, size_t workspace_bytes, dwc_stream_t stream) {
    Problem P;
    dwc_status_t st = check_problem(N, H, W, C, FH, FW, stride, pad, dtype, P);
    if (st != DWC_OK) return st;
    const long long nx = static_cast<long long>(N) * H * W * C;
    const long long ndy = static_cast<long long>(N) * P.OH * P.OW * C;
    const long long ndw = static_cast<long long>(FH) * FW * C;
    st = check_pointers(P, x, nx, dy, ndy, dw, ndw);
    if (st != DWC_OK) return st;
    if (ndw == 0) return DWC_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0) return map_cuda(cudaMemsetAsync(dw, 0, sizeof(float) * ndw, s));
    const size_t need = dwc_bwd_filter_workspace_size(N, H, W, C, FH, FW, stride, pad, dtype);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16)))
        return DWC_ERR_WORKSPACE;
    float* ws = static_cast<float*>(workspace);
    const size_t ws_floats = workspace_bytes / sizeof(float);
    if (fast_eligible(P, x, dy, dw) && fast_fgrad_floats(P) > 0) {
        FilterGrad fg{x, dy, dw, N, H, W, C, P.OH, P.OW, FH, FW, pad, P.dtype, ws, ws_floats, s,
                      status_word(), wait_limit_ns()};
        const cudaError_t err = launch_fgrad(fg);
        if (err != cudaErrorNotSupported) return map_cuda(err);
        (void)cudaGetLastError();
    } else if (fast_s2_eligible(P, x, dy, dw) &&
               filter_grad_s2_workspace_floats(N, P.OH, P.OW, C, FH, FW, P.dtype) > 0) {
        FilterGrad fg{x, dy, dw, N, H, W, C, P.OH, P.OW, FH, FW, pad, P.dtype, ws, ws_floats, s,
                      status_word(), wait_limit_ns()};
        const cudaError_t err = launch_fgrad_s2(fg);
        if (err != cudaErrorNotSupported) return map_cuda(err);
        (void)cudaGetLastError();
    }
    GeneralConv gc{x, dy, dw, N, H, W, C, P.OH, P.OW, FH, FW, stride, pad, P.dtype, ws, ws_floats, s};
    return map_cuda(launch_general_bwd_filter(gc));
}

dwc_status_t dwc_device_status(dwc_stream_t stream) {
    unsigned int* word = status_word();
    if (word == nullptr) return DWC_ERR_CUDA;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DWC_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DWC_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return DWC_ERR_CUDA;
        return DWC_ERR_TIMEOUT;
    }
    return DWC_OK;
}

const char* dwc_status_string(dwc_status_t status) {
    switch (status) {
        case DWC_OK: return "ok";
        case DWC_ERR_INVALID_ARG: return "invalid argument";
        case DWC_ERR_UNSUPPORTED: return "problem size beyond the library's limits";
        case DWC_ERR_ALIGNMENT: return "tensor pointer not aligned to its element size";
        case DWC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case DWC_ERR_CUDA: return "CUDA runtime or launch error";
        case DWC_ERR_TIMEOUT: return "a kernel wait ran out of time";
        default: return "unknown status";
    }
}

int dwc_version(void) { return 200; }

unsigned long long dwc_set_wait_limit_ns(unsigned long long ns) {
    return g_wait_limit_ns.exchange(ns, std::memory_order_acq_rel);
}

void dwc_testing_stall_next_row_launch(void) { g_row_stall.store(1, std::memory_order_release); }

int dwc_testing_prefer_family(int family) {
    if (family != 0 && family != kFamilyCudaCore && family != kFamilyTcgen05 &&
        family != kFamilyMmaSync)
        return -1;
    return g_family_pref.exchange(family, std::memory_order_acq_rel);
}

int dwc_testing_tc_row_pairs(int mode) {
    if (mode < 0 || mode > 2) return -1;
    return g_tc_pairs.exchange(mode, std::memory_order_acq_rel);
}

int dwc_path(int pass, const void* a, const void* b, const void* out, int N, int H, int W, int C,
             int FH, int FW, int stride, int pad, dwc_dtype_t dtype) {
    Problem P;
    if (pass < 0 || pass > 3) return -1;
    if (check_problem(N, H, W, C, FH, FW, stride, pad, dtype, P) != DWC_OK) return -1;
    if (pass == 3) return bnact_fast_eligible(P, a, b, out) ? 1 : 0;
    if (fast_s2_eligible(P, a, b, out)) {
        if (pass == kPassBwdFilter)
            return filter_grad_s2_workspace_floats(N, P.OH, P.OW, C, FH, FW, P.dtype) > 0 ? 1 : 0;
        return 1;
    }
    if (P.s == 2) return 0;
    if (!fast_eligible(P, a, b, out)) return 0;
    if (pass == kPassBwdFilter) {
        if (fast_fgrad_floats(P) == 0) return 0;
        if (small_fgrad_floats(P) > 0) return 3;
        if (P.e == 2 && FH == FW) {
            FilterGrad fg{};
            fg.N = N; fg.H = H; fg.W = W; fg.C = C; fg.OH = P.OH; fg.OW = P.OW;
            fg.FH = FH; fg.FW = FW; fg.pad = pad; fg.dtype = P.dtype;
            const int pref = family_preference();
            if (tc_fgrad_taken(fg)) return 2;
            if ((pref == 0 || pref == 4) && tensor_core_fgrad(N, C, P.OH, P.OW, FH, FW)) return 4;
        }
        return 1;
    }
    const bool pref16 = P.e == 2 && family_preference() != 0;
    // the same RowConv the entry points build (backward data: over dy, output H x W)
    const RowConv rc = pass == kPassFwd
        ? RowConv{a, b, nullptr, N, H, W, C, P.OH, P.OW, FH, FW, pad, pad, false, P.dtype,
                  nullptr, nullptr}
        : RowConv{a, b, nullptr, N, P.OH, P.OW, C, H, W, FH, FW, FH - 1 - pad, FW - 1 - pad,
                  true, P.dtype, nullptr, nullptr};
    const bool tc16 = P.e == 2 && !pref16 && tc_rows_preferred(rc);
    if (FH == FW && !pref16 && !tc16 &&
        (pass == kPassFwd ? small_map_serves(H, W, P.OH, P.OW, FW, pad)
                          : small_map_serves(P.OH, P.OW, H, W, FW, FW - 1 - pad)))
        return 3;
    if (P.e == 2) return tensor_core_rows(rc);
    return 1;
}

int dwc_kernel_launches(int pass, int N, int H, int W, int C, int FH, int FW, int stride, int pad,
                        dwc_dtype_t dtype) {
    const int fam = dwc_path(pass, nullptr, nullptr, nullptr, N, H, W, C, FH, FW, stride, pad, dtype);
    if (fam < 0) return -1;
    Problem P;
    if (check_problem(N, H, W, C, FH, FW, stride, pad, dtype, P) != DWC_OK) return -1;
    const long long out = pass == kPassBwdFilter ? static_cast<long long>(FH) * FW * C
                        : pass == kPassBwdData ? static_cast<long long>(N) * H * W * C
                                               : static_cast<long long>(N) * P.OH * P.OW * C;
    if (out == 0) return 0;
    // filter gradients: the kernel and the fixed-order sum of its slices (or a fill of dW
    // with zeros when nothing meets it: a memset, not a kernel of this library); the tcgen05
    // filter gradient: the stacked copies of x and dy (one kernel), then the main kernel;
    // 7x7 maps: one kernel (its clusters sum the slices)
    if (pass == kPassBwdFilter) {
        if (N == 0) return 0;
        if (fam == 3 && stride == 1 && tiny_fgrad_single_launch(P.dtype, N, H, W, C, FH, FW, pad)) return 1;
        return 2;
    }
    if (pass == 3) {
        // 7x7 at stride 1 on the fast path: act(BN(x)) into scratch (and 16-bit filters
        // widened), then the plain fp32 forward (a second launch for a tail of at most 32
        // channels past a multiple of 64)
        if (fam == 1 && bnact_split_serves(FH, FW, stride, C, W)) {
            const int rem = C % 64;
            return (dtype == DWC_F32 ? 2 : 3) + (C > 64 && rem != 0 && rem <= 32 ? 1 : 0);
        }
        return 1;
    }
    if (fam == 2) {
        const RowConv rc = pass == kPassFwd
            ? RowConv{nullptr, nullptr, nullptr, N, H, W, C, P.OH, P.OW, FH, FW, pad, pad, false,
                      P.dtype, nullptr, nullptr}
            : RowConv{nullptr, nullptr, nullptr, N, P.OH, P.OW, C, H, W, FH, FW, FH - 1 - pad,
                      FW - 1 - pad, true, P.dtype, nullptr, nullptr};
        return tc_rows_launches(rc);
    }
    // row kernel, 3 to 7 taps (square): a channel tail of at most 32 past a multiple of 64
    // runs as a second launch on lane groups (7 taps)
    const bool rows = fam == 1 && FH == FW && FH <= 7 && !(stride == 2 && pass == kPassBwdData);
    const int rem = C % 64;
    if (rows && C > 64 && rem != 0 && rem <= 32 && FH == 7) return 2;
    return 1;
}

}  // extern "C"
