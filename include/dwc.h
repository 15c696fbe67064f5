/*
 * dwc.h -- C ABI of the GB300 depthwise 2-D convolution library (libdwc_gb300.so).
 *
 * Operation ("Flash-DWC: Making Depthwise Convolution Compute-Efficient on GPUs",
 * §2.1 and Fig. 1): every channel c has its own FH x FW filter and
 *
 *     Y[n, oh, ow, c] = sum_{fh < FH, fw < FW} X[n, oh*s + fh - p, ow*s + fw - p, c] * W[fh, fw, c]
 *
 * with taps outside the image contributing zero (zero padding p on all four sides, one
 * stride s for both axes), OH = floor((H + 2p - FH) / s) + 1, OW = floor((W + 2p - FW) / s) + 1.
 * The forward pass is a cross-correlation (no filter flip).
 *
 * Layout (§2.3, "unified channels-last layout"), all tensors dense and row-major:
 *     X, dX : N x H  x W  x C      (input of the forward pass and its gradient)
 *     Y, dY : N x OH x OW x C      (output of the forward pass and its gradient)
 *     W, dW : FH x FW x C          (filter and its gradient; channel last)
 *
 * Data types: the inputs (X, W, dY) of one call share one dtype (fp32, bf16 or fp16);
 * every output (Y, dX, dW) is fp32, except that dwc_fwd_ex / dwc_bwd_data_ex may write Y /
 * dX in the 16-bit input's own type.  All arithmetic is fp32 multiply-add; 16-bit inputs
 * are widened to fp32 exactly before use.
 *
 * Pointers and ownership: every tensor pointer is a DEVICE pointer allocated and owned by
 * the caller.  Inputs are only read; outputs are overwritten (never accumulated into).
 * Outputs must not overlap inputs.  Calls are asynchronous on `stream` (0 = legacy default
 * stream): they enqueue work and return; the caller synchronises.  Device memory: the
 * 16-bit calls that run on the tcgen05 tensor-core kernels (see dwc_path) take scratch with
 * cudaMallocFromPoolAsync on `stream` -- forward and backward data for a re-laid-out copy of
 * their input and the filter's Toeplitz runs (about 1.5x the input's bytes), the filter
 * gradient for re-laid-out copies of x and dy (about 1.3x their bytes) -- from a memory pool
 * the library creates per device on first use and that keeps up to 512 MiB between calls;
 * the scratch returns to the pool in stream order (cudaFreeAsync) after the call's kernels.
 * If the allocation fails the call runs on another kernel.  dwc_fwd_bn_act with 7x7 filters
 * at stride 1 on rows of 28 or more takes scratch from the same pool for an fp32 copy of
 * act(BN(X)) (4 bytes per input element, plus the filter widened to fp32 for 16-bit
 * inputs).  No other call allocates device memory (dwc_bwd_filter otherwise takes a caller
 * workspace).
 *
 * Stream order and dependent launches: the library launches its kernels with programmatic
 * stream serialization.  Each kernel lets the next kernel of the stream be scheduled as it
 * starts, and waits (griddepcontrol.wait) for the kernel before it to complete before it
 * touches memory, so the results are those of plain stream order.  A caller kernel launched
 * right after a call WITH the programmatic-serialization attribute must likewise wait
 * (griddepcontrol.wait / cudaGridDependencySynchronize) before reading the call's outputs,
 * as the CUDA model asks of every programmatic dependent; ordinary launches, events, copies
 * and CUDA-graph capture see plain stream order.
 *
 * Errors: every call validates its arguments on the host and returns a dwc_status_t
 * without launching anything when they are wrong.  No call aborts or throws.  A CUDA
 * launch failure is returned as DWC_ERR_CUDA.  Kernels never spin without limit: a wait
 * inside a kernel that runs out of time sets a device-side status bit and the kernel
 * ends; dwc_device_status() reports it as DWC_ERR_TIMEOUT.
 *
 * Every fp32 tensor must be 4-byte aligned and every 16-bit tensor 2-byte aligned.  The
 * fast kernels are used when C is a multiple of 4 (fp32) or 8 (16-bit), all pointers are
 * 16-byte aligned and either
 *   - stride == 1 with a square filter of odd size 3..51, or a stripe (non-square) filter
 *     of odd width 1..51 and any height 1..255, or
 *   - stride == 2 with a square odd filter of 3 to 13 taps;
 * everything else (strides above 2, even widths, ...) runs on the general kernels (same
 * results, slower).
 */
#ifndef DWC_GB300_H
#define DWC_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dwc_stream_t; /* a cudaStream_t */

typedef enum {
    DWC_F32 = 0,  /* IEEE fp32 inputs */
    DWC_BF16 = 1, /* bfloat16 inputs, fp32 accumulation and output */
    DWC_F16 = 2   /* IEEE fp16 inputs, fp32 accumulation and output */
} dwc_dtype_t;

typedef enum {
    DWC_OK = 0,
    DWC_ERR_INVALID_ARG = 1, /* null pointer, negative size, stride < 1, pad < 0, empty filter,
                                unknown dtype, output does not fit (OH or OW < 1) */
    DWC_ERR_UNSUPPORTED = 2, /* a size beyond the library's limits (int32 index overflow) */
    DWC_ERR_ALIGNMENT = 3,   /* a tensor pointer is not aligned to its element size */
    DWC_ERR_WORKSPACE = 4,   /* workspace missing or smaller than the query says */
    DWC_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
    DWC_ERR_TIMEOUT = 6      /* a kernel gave up waiting (reported by dwc_device_status) */
} dwc_status_t;

/* Forward pass Y = DWC(X, W) (§2.1, Fig. 1; §3 and §4 of the paper give the GPU dataflow).
 *   x : N x H x W x C, dtype      w : FH x FW x C, dtype      y : N x OH x OW x C, fp32 (out)
 */
dwc_status_t dwc_fwd(const void* x, const void* w, float* y,
                     int N, int H, int W, int C, int FH, int FW, int stride, int pad,
                     dwc_dtype_t dtype, dwc_stream_t stream);

/* Forward pass and backward data with a chosen output type.  Same operations, arguments and
 * errors as dwc_fwd / dwc_bwd_data, plus:
 *   out_dtype : DWC_F32, or the input's own 16-bit type (DWC_BF16 for bf16 inputs, DWC_F16 for
 *               fp16 inputs).  A 16-bit output holds the fp32 result rounded to nearest even
 *               once, at the store; it halves the output's HBM traffic.  Any other combination
 *               (e.g. fp32 inputs with a 16-bit output) returns DWC_ERR_INVALID_ARG.
 *   y, dx     : N x OH x OW x C / N x H x W x C elements of out_dtype, aligned to its size.
 * (The paper keeps fp32 outputs; 16-bit outputs are an option of this library.  The filter
 * gradient stays fp32: it is small and is an accumulation.) */
dwc_status_t dwc_fwd_ex(const void* x, const void* w, void* y,
                        int N, int H, int W, int C, int FH, int FW, int stride, int pad,
                        dwc_dtype_t dtype, dwc_dtype_t out_dtype, dwc_stream_t stream);
dwc_status_t dwc_bwd_data_ex(const void* dy, const void* w, void* dx,
                             int N, int H, int W, int C, int FH, int FW, int stride, int pad,
                             dwc_dtype_t dtype, dwc_dtype_t out_dtype, dwc_stream_t stream);

/* Activation applied after the batch normalisation of dwc_fwd_bn_act. */
typedef enum {
    DWC_ACT_NONE = 0,  /* identity */
    DWC_ACT_RELU = 1,  /* max(v, 0) */
    DWC_ACT_RELU6 = 2  /* min(max(v, 0), 6) */
} dwc_act_t;

/* BN + Act + forward DWC fused in one pass ("kernel fusion", §5.2 of the paper: a DWC is
 * commonly preceded by batch normalisation and an activation; the fused kernel normalises
 * and activates each input value as it reads it, so the activated tensor never goes
 * through HBM):
 *   Z[n, h, w, c] = act((X[n, h, w, c] - mean[c]) / sqrt(var[c] + eps) * gamma[c] + beta[c])
 *   Y = DWC(Z, W), whose zero padding applies to Z (a tap in the padding reads 0, not
 *       act(BN(0))).
 * Forward pass only: the batch statistics are inputs (computed beforehand, or running
 * statistics at inference); the backward passes through BN and Act are not part of it.
 *   x : N x H x W x C, dtype      w : FH x FW x C, dtype      y : N x OH x OW x C, fp32 (out)
 *   mean, var, gamma, beta : C fp32 values each, device memory, read only; eps >= 0.
 * The fused fast path covers square 3x3, 5x5 and 7x7 filters at stride 1 or 2 under the
 * layout rules of the fast kernels; other problems run a general fused kernel.  Errors as
 * dwc_fwd; DWC_ERR_INVALID_ARG also for a null BN pointer (C > 0), an unknown activation or
 * a negative or non-finite eps; DWC_ERR_ALIGNMENT for a BN pointer not 4-byte aligned.
 * Exception to "one pass": 7x7 filters at stride 1 (C a multiple of 4, rows of 28 or more
 * pixels) measured faster as two
 * passes (the fused 7x7 kernel's per-element transforms cost more than the HBM round trip of
 * Z), so there Z is written once as fp32 to stream-ordered scratch memory from the library's
 * pool and the plain forward reads it: the same arithmetic and results. */
dwc_status_t dwc_fwd_bn_act(const void* x, const float* mean, const float* var,
                            const float* gamma, const float* beta, float eps, dwc_act_t act,
                            const void* w, float* y, int N, int H, int W, int C, int FH, int FW,
                            int stride, int pad, dwc_dtype_t dtype, dwc_stream_t stream);

/* Backward data ("BDC", §5.1): dX = the adjoint of the forward pass in X, i.e.
 *   dX[n, ih, iw, c] = sum over (oh, ow, fh, fw) with oh*s + fh - p = ih and ow*s + fw - p = iw
 *                      of dY[n, oh, ow, c] * W[fh, fw, c];
 * for stride 1 this is the forward pass over dY with W rotated by 180 degrees and pad
 * FH-1-p (the rotation is folded into the kernel's filter indexing; no copy is made).
 *   dy : N x OH x OW x C, dtype   w : FH x FW x C, dtype   dx : N x H x W x C, fp32 (out)
 * N, H, W, C, FH, FW, stride, pad describe the FORWARD problem (H, W = forward input size).
 */
dwc_status_t dwc_bwd_data(const void* dy, const void* w, float* dx,
                          int N, int H, int W, int C, int FH, int FW, int stride, int pad,
                          dwc_dtype_t dtype, dwc_stream_t stream);

/* Bytes of device workspace dwc_bwd_filter needs for this problem on the CURRENT device
 * (0 means none).  Returns 0 for invalid arguments as well; dwc_bwd_filter then reports the
 * argument error. */
size_t dwc_bwd_filter_workspace_size(int N, int H, int W, int C, int FH, int FW, int stride,
                                     int pad, dwc_dtype_t dtype);

/* Backward filter ("BFC", §5.1): dW[fh, fw, c] = sum_{n, oh, ow} X[n, oh*s+fh-p, ow*s+fw-p, c]
 *                                                             * dY[n, oh, ow, c].
 * The accumulation axis N*OH*OW is split into slices (§5.1, "accumulation-axis
 * parallelism"); slice partials go to `workspace` and are summed in a fixed order, so the
 * result is bit-identical from run to run (no atomics).  (On 7x7 maps with 3 taps the
 * slices of a channel block form one thread-block cluster and are summed through
 * distributed shared memory, in a fixed order too; the workspace is then left untouched.)
 *   x : N x H x W x C, dtype   dy : N x OH x OW x C, dtype   dw : FH x FW x C, fp32 (out)
 *   workspace : device buffer of at least dwc_bwd_filter_workspace_size(...) bytes, owned by
 *               the caller, 16-byte aligned, contents ignored on entry and clobbered.
 */
dwc_status_t dwc_bwd_filter(const void* x, const void* dy, float* dw,
                            int N, int H, int W, int C, int FH, int FW, int stride, int pad,
                            dwc_dtype_t dtype, void* workspace, size_t workspace_bytes,
                            dwc_stream_t stream);

/* Filter gradient without any allocation (no counterpart in the paper: an addition of this
 * library).  Same operation, arguments, results and errors as dwc_bwd_filter, but the
 * workspace is a fixed device array inside the library instead of a caller buffer.
 *
 * Who needs it: callers that cannot call cudaMalloc, e.g. code running under a fixed
 * device-memory budget or a caching allocator that must not grow, plug-in hosts that hand
 * the library only its input and output buffers, and code that must not trigger the
 * implicit synchronisation an allocation can cause.
 *
 * Limit: the array holds 8 Mi floats (32 MiB); it is reserved on a GPU when the library's
 * device code is loaded there (at the latest by the first call of this function on that
 * GPU) and stays reserved until the process exits.  A problem whose
 * dwc_bwd_filter_workspace_size() exceeds 32 MiB is rejected with DWC_ERR_UNSUPPORTED
 * before anything is launched (every benchmark shape of this library fits); argument and
 * pointer errors are reported first, as dwc_bwd_filter reports them.
 *
 * Set-up: the first call on each device looks up the array's device address with that
 * device current (cudaGetSymbolAddress); make that first call before any stream capture.
 * Sharing: all calls use the same array and leave their partial sums in it; nothing in it
 * needs to start at zero.  Calls whose kernels overlap on the GPU (e.g. on two unordered
 * streams) race on the array: order them on one stream or with events.  The call itself
 * allocates and frees nothing.
 * Check dwc_device_status() before trusting dW: a kernel whose bounded wait ran out leaves
 * some partial sums unwritten, and the final sum then adds an earlier call's leftovers, so
 * dW can look finite and plausible although it is wrong. */
dwc_status_t dwc_bwd_filter_noalloc(const void* x, const void* dy, float* dw,
                                    int N, int H, int W, int C, int FH, int FW, int stride,
                                    int pad, dwc_dtype_t dtype, dwc_stream_t stream);

/* Synchronises `stream`, then reads and clears the device status word that the kernels
 * set when a wait runs out of time.  DWC_OK if no kernel reported a problem since the last
 * call, DWC_ERR_TIMEOUT if one did, DWC_ERR_CUDA if the synchronisation failed. */
dwc_status_t dwc_device_status(dwc_stream_t stream);

/* Upper bound, in nanoseconds, on every wait inside the kernels launched after this call (on
 * any device and stream); 0 restores the default of 2 seconds.  A healthy wait lasts
 * microseconds: the limit only decides how soon a kernel whose data never arrives gives up
 * and reports DWC_ERR_TIMEOUT through dwc_device_status().  Returns the previous setting. */
unsigned long long dwc_set_wait_limit_ns(unsigned long long ns);

/* Multiply-add rate microbenchmark of the CUDA cores, the measured compute peak against
 * which the CUDA-core kernels' roofline is stated (no counterpart in the paper).  Launches
 * `blocks` x 256 threads on `stream`; every thread runs `iters` iterations of 8 independent
 * chains of one multiply-add instruction:
 *   kind 0: fp32 FMA (1 multiply-add per instruction)
 *   kind 1: packed fp32x2 FMA (2 per instruction)
 *   kind 2: packed fp16x2 FMA (2 per instruction)
 *   kind 3: packed bf16x2 FMA (2 per instruction)
 * so one launch performs blocks * 256 * iters * 8 * (1 or 2) multiply-adds (2 FLOPs each);
 * the caller times it with events on `stream`.  `out` (device, blocks * 256 floats) receives
 * one value per thread.  DWC_ERR_INVALID_ARG for an unknown kind, blocks or iters < 1 or a
 * null `out`. */
dwc_status_t dwc_fma_rate_probe(int kind, int blocks, int iters, float* out, dwc_stream_t stream);

/* Static text for a status code (never NULL). */
const char* dwc_status_string(dwc_status_t status);

/* Library version as 10000*major + 100*minor + patch. */
int dwc_version(void);

/* Which kernel family a call with these arguments would use: 1 = fast CUDA-core kernels
 * (row-streaming, stride-2 and filter-gradient kernels, for the shapes listed at the top
 * of this file), 2 = tensor-core kernels on the 5th-generation MMA (tcgen05, accumulators in
 * tensor memory; 16-bit inputs only), 3 = small-map kernels (maps up to 16 x 16), 4 =
 * tensor-core kernels on the warp-level MMA (mma.sync; 16-bit inputs only), 0 = general
 * kernels, -1 = invalid arguments.  `pass` is 0 for
 * dwc_fwd, 1 for dwc_bwd_data, 2 for dwc_bwd_filter, 3 for dwc_fwd_bn_act.  Pointer
 * alignment is checked with the pointers given (they may be NULL to mean "16-byte
 * aligned"). */
int dwc_path(int pass, const void* a, const void* b, const void* out,
             int N, int H, int W, int C, int FH, int FW, int stride, int pad, dwc_dtype_t dtype);

/* Kernel launches of this library that a call with these arguments and 16-byte aligned
 * pointers makes (the tcgen05 forward / backward data: a preparation kernel and the main
 * kernel; the tcgen05 filter gradient: one preparation kernel and the main kernel; the
 * filter gradient of 7x7 maps with 3 taps: one kernel; other filter gradients: the
 * kernel and the sum of its slices), 0 for an empty output, -1 for
 * invalid arguments.  `pass` as for dwc_path.  For profiling and launch accounting. */
int dwc_kernel_launches(int pass, int N, int H, int W, int C, int FH, int FW, int stride, int pad,
                        dwc_dtype_t dtype);

#ifdef __cplusplus
}
#endif

#endif /* DWC_GB300_H */
