// dwc_noalloc.cu -- filter gradient for callers that cannot allocate device memory.
//
// dwc_bwd_filter needs a device workspace for its per-slice partial sums, which the caller
// allocates.  Some callers cannot do that: code running inside a fixed memory budget that
// forbids new device allocations, allocator-less runtimes and plug-in hosts that hand the
// library only the input and output buffers, or code paths where a cudaMalloc would
// synchronise the device at a bad moment.  dwc_bwd_filter_noalloc serves them with a
// workspace that lives in a file-scope device array of fixed size, reserved once when
// the library's device code is loaded and held by every GPU that loads it until the
// process exits.  No call allocates or frees anything.
//
// Sharing rules: every call uses the same array and leaves its partial sums there.  The
// filter-gradient kernels overwrite every partial sum they later read, so nothing in the
// array has to start at zero and no clearing is done.  Two calls whose kernels overlap on
// the GPU (for example on different streams without ordering between them) race on the
// array and produce wrong results; order them on one stream or with events.
#include <mutex>

#include "../../include/dwc.h"
#include "dwc_host.h"

namespace {

// 8 Mi floats = 32 MiB: enough for the filter gradient of every benchmark shape (the
// largest, 31x31 filters over 1024 channels, needs about 3 Mi floats).
constexpr size_t kScratchFloats = size_t(8) << 20;

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
// In host code the array's name is only a host-side handle, so it must not be passed to a
// kernel directly; cudaGetSymbolAddress returns the real device address.
float* scratch_for_current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[d] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            (void)cudaGetLastError();  // the next call's launch check must not see this failure
            return nullptr;
        }
        g_scratch_ptr[d] = static_cast<float*>(p);
    }
    return g_scratch_ptr[d];
}

}  // namespace

extern "C" dwc_status_t dwc_bwd_filter_noalloc(const void* x, const void* dy, float* dw, int N,
                                               int H, int W, int C, int FH, int FW, int stride,
                                               int pad, dwc_dtype_t dtype, dwc_stream_t stream) {
    // argument and pointer errors first, exactly as dwc_bwd_filter reports them; only a
    // valid call that does not fit the fixed array is DWC_ERR_UNSUPPORTED
    const int st = dwc::validate_bwd_filter(x, dy, dw, N, H, W, C, FH, FW, stride, pad,
                                            static_cast<int>(dtype));
    if (st != DWC_OK) return static_cast<dwc_status_t>(st);
    const size_t need = dwc_bwd_filter_workspace_size(N, H, W, C, FH, FW, stride, pad, dtype);
    if (need == 0)  // empty problems and shapes that need no workspace
        return dwc_bwd_filter(x, dy, dw, N, H, W, C, FH, FW, stride, pad, dtype, nullptr, 0,
                              stream);
    if (need > kScratchFloats * sizeof(float)) return DWC_ERR_UNSUPPORTED;
    float* scratch = scratch_for_current_device();
    if (scratch == nullptr) return DWC_ERR_CUDA;
    return dwc_bwd_filter(x, dy, dw, N, H, W, C, FH, FW, stride, pad, dtype, scratch,
                          kScratchFloats * sizeof(float), stream);
}
