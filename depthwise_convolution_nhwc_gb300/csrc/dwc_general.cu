// dwc_general.cu -- fallback kernels for any stride, channel count, alignment or filter
// size, and the fixed-order reduction of filter-gradient slices.
//
// These follow the definitions directly ("Flash-DWC: Making Depthwise Convolution
// Compute-Efficient on GPUs", §2.1 / Fig. 1 for the forward pass, §5.1 for the two backward
// passes, §5.2 for BN + Act in front of the forward pass) with one thread per output element and fp32 accumulation; they serve the shapes
// the row-streaming kernels do not cover (strides above 1, odd channel counts, unaligned
// pointers, even or very large filters).
#include <algorithm>

#include "dwc_device.cuh"
#include "dwc_host.h"

namespace dwc {

template <typename T, class OutT>
__global__ void general_fwd_kernel(const T* __restrict__ x, const T* __restrict__ w,
                                   OutT* __restrict__ y, int N, int H, int W, int C, int OH,
                                   int OW, int FH, int FW, int s, int p) {
    const long long total = static_cast<long long>(N) * OH * OW * C;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        long long q = i;
        const int c = static_cast<int>(q % C); q /= C;
        const int ow = static_cast<int>(q % OW); q /= OW;
        const int oh = static_cast<int>(q % OH); q /= OH;
        const int n = static_cast<int>(q);
        // only the taps that land inside the image: fh in [p - oh*s, H + p - oh*s)
        const int fh0 = max(0, p - oh * s), fh1 = min(FH, H + p - oh * s);
        const int fw0 = max(0, p - ow * s), fw1 = min(FW, W + p - ow * s);
        float acc = 0.f;
        for (int fh = fh0; fh < fh1; ++fh) {
            const int ih = oh * s + fh - p;
            for (int fw = fw0; fw < fw1; ++fw) {
                const int iw = ow * s + fw - p;
                acc = fmaf(to_f32(x[((static_cast<size_t>(n) * H + ih) * W + iw) * C + c]),
                           to_f32(w[(static_cast<size_t>(fh) * FW + fw) * C + c]), acc);
            }
        }
        store_out(y + i, acc);
    }
}

// y = DWC(act(BN(x)), w): the forward kernel with every in-image input value normalised with
// its channel's batch statistics and activated first (taps in the padding read zero, as
// the DWC pads the activated tensor).  act: 0 identity, 1 ReLU, 2 ReLU6.
template <typename T>
__global__ void general_fwd_bnact_kernel(const T* __restrict__ x, const T* __restrict__ w,
                                         float* __restrict__ y, int N, int H, int W, int C,
                                         int OH, int OW, int FH, int FW, int s, int p,
                                         const float* __restrict__ mean,
                                         const float* __restrict__ var,
                                         const float* __restrict__ gamma,
                                         const float* __restrict__ beta, float eps, int act) {
    const long long total = static_cast<long long>(N) * OH * OW * C;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        long long q = i;
        const int c = static_cast<int>(q % C); q /= C;
        const int ow = static_cast<int>(q % OW); q /= OW;
        const int oh = static_cast<int>(q % OH); q /= OH;
        const int n = static_cast<int>(q);
        const float scale = gamma[c] * rsqrtf(var[c] + eps);
        const float shift = beta[c] - mean[c] * scale;
        const int fh0 = max(0, p - oh * s), fh1 = min(FH, H + p - oh * s);
        const int fw0 = max(0, p - ow * s), fw1 = min(FW, W + p - ow * s);
        float acc = 0.f;
        for (int fh = fh0; fh < fh1; ++fh) {
            const int ih = oh * s + fh - p;
            for (int fw = fw0; fw < fw1; ++fw) {
                const int iw = ow * s + fw - p;
                float z = fmaf(to_f32(x[((static_cast<size_t>(n) * H + ih) * W + iw) * C + c]),
                               scale, shift);
                if (act >= 1) z = fmaxf(z, 0.f);
                if (act == 2) z = fminf(z, 6.f);
                acc = fmaf(z, to_f32(w[(static_cast<size_t>(fh) * FW + fw) * C + c]), acc);
            }
        }
        y[i] = acc;
    }
}

// dx[n, ih, iw, c] = sum over taps whose forward product read x[n, ih, iw, c].
template <typename T, class OutT>
__global__ void general_bwd_data_kernel(const T* __restrict__ dy, const T* __restrict__ w,
                                        OutT* __restrict__ dx, int N, int H, int W, int C,
                                        int OH, int OW, int FH, int FW, int s, int p) {
    const long long total = static_cast<long long>(N) * H * W * C;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        long long q = i;
        const int c = static_cast<int>(q % C); q /= C;
        const int iw = static_cast<int>(q % W); q /= W;
        const int ih = static_cast<int>(q % H); q /= H;
        const int n = static_cast<int>(q);
        // taps whose output lies inside: 0 <= ih + p - fh <= (OH - 1) * s
        const int fh0 = max(0, ih + p - (OH - 1) * s), fh1 = min(FH, ih + p + 1);
        const int fw0 = max(0, iw + p - (OW - 1) * s), fw1 = min(FW, iw + p + 1);
        float acc = 0.f;
        for (int fh = fh0; fh < fh1; ++fh) {
            const int th = ih + p - fh;
            if (th % s) continue;
            const int oh = th / s;
            for (int fw = fw0; fw < fw1; ++fw) {
                const int tw = iw + p - fw;
                if (tw % s) continue;
                const int ow = tw / s;
                acc = fmaf(to_f32(dy[((static_cast<size_t>(n) * OH + oh) * OW + ow) * C + c]),
                           to_f32(w[(static_cast<size_t>(fh) * FW + fw) * C + c]), acc);
            }
        }
        store_out(dx + i, acc);
    }
}

// part[z, fh, fw, c] = sum over output rows of slice z of x * dy.
template <typename T>
__global__ void general_bwd_filter_kernel(const T* __restrict__ x, const T* __restrict__ dy,
                                          float* __restrict__ part, int N, int H, int W, int C,
                                          int OH, int OW, int FH, int FW, int s, int p,
                                          int rows_per_slice, int Z) {
    pdl_trigger();   // the slice sum may be scheduled now (it waits for this grid)
    const long long per_z = static_cast<long long>(FH) * FW * C;
    const long long total = per_z * Z;
    const long long rows = static_cast<long long>(N) * OH;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int z = static_cast<int>(i / per_z);
        long long q = i % per_z;
        const int c = static_cast<int>(q % C); q /= C;
        const int fw = static_cast<int>(q % FW); q /= FW;
        const int fh = static_cast<int>(q);
        float acc = 0.f;
        const long long r1 = std::min<long long>(static_cast<long long>(z + 1) * rows_per_slice, rows);
        for (long long r = static_cast<long long>(z) * rows_per_slice; r < r1; ++r) {
            const int n = static_cast<int>(r / OH), oh = static_cast<int>(r % OH);
            const int ih = oh * s + fh - p;
            if (ih < 0 || ih >= H) continue;
            for (int ow = 0; ow < OW; ++ow) {
                const int iw = ow * s + fw - p;
                if (iw < 0 || iw >= W) continue;
                acc = fmaf(to_f32(x[((static_cast<size_t>(n) * H + ih) * W + iw) * C + c]),
                           to_f32(dy[((static_cast<size_t>(n) * OH + oh) * OW + ow) * C + c]), acc);
            }
        }
        part[i] = acc;
    }
}

// out[i] = sum_z part[z * count + i].  A block covers 32 consecutive outputs (one per lane,
// so every slice row is read with coalesced 128-byte loads); warp k sums the contiguous
// slice range [k*zc, (k+1)*zc) and warp 0 adds the 8 partial sums in warp order.  The order
// of additions depends only on `slices`, so runs are bit-identical.
constexpr int kReduceWarps = 8;

__global__ void __launch_bounds__(kReduceWarps * 32)
reduce_slices_kernel(const float* __restrict__ part, int slices, size_t count,
                     float* __restrict__ out) {
    pdl_wait();   // the kernel that wrote the slices has finished
    __shared__ float partial[kReduceWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int zc = (slices + kReduceWarps - 1) / kReduceWarps;
    const int z0 = min(slices, warp * zc), z1 = min(slices, z0 + zc);
    for (size_t base = static_cast<size_t>(blockIdx.x) * 32; base < count;
         base += static_cast<size_t>(gridDim.x) * 32) {
        const size_t i = base + lane;
        float s = 0.f;
        if (i < count) {
#pragma unroll 8
            for (int z = z0; z < z1; ++z) s += part[static_cast<size_t>(z) * count + i];
        }
        partial[warp][lane] = s;
        __syncthreads();
        if (warp == 0 && i < count) {
            float t = partial[0][lane];
#pragma unroll
            for (int k = 1; k < kReduceWarps; ++k) t += partial[k][lane];
            out[i] = t;
        }
        __syncthreads();
    }
}

// The same sum, four consecutive outputs per lane (16-byte loads and stores; a block covers
// 128 outputs), for counts that are a multiple of 4 with 16-byte aligned buffers.  Each
// output's additions come in the same order as in reduce_slices_kernel, so the two give
// identical results.
__global__ void __launch_bounds__(kReduceWarps * 32)
reduce_slices4_kernel(const float4* __restrict__ part, int slices, size_t count4,
                      float4* __restrict__ out) {
    pdl_wait();   // the kernel that wrote the slices has finished
    __shared__ float4 partial[kReduceWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int zc = (slices + kReduceWarps - 1) / kReduceWarps;
    const int z0 = min(slices, warp * zc), z1 = min(slices, z0 + zc);
    for (size_t base = static_cast<size_t>(blockIdx.x) * 32; base < count4;
         base += static_cast<size_t>(gridDim.x) * 32) {
        const size_t i = base + lane;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < count4) {
#pragma unroll 8
            for (int z = z0; z < z1; ++z) {
                const float4 v = part[static_cast<size_t>(z) * count4 + i];
                s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
            }
        }
        partial[warp][lane] = s;
        __syncthreads();
        if (warp == 0 && i < count4) {
            float4 t = partial[0][lane];
#pragma unroll
            for (int k = 1; k < kReduceWarps; ++k) {
                const float4 v = partial[k][lane];
                t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
            }
            out[i] = t;
        }
        __syncthreads();
    }
}

// Launched as a programmatic dependent of the kernel before it in the stream (the one that
// wrote the slices): it is scheduled while that kernel runs and waits in pdl_wait(), which
// saved 1-3 us per filter-gradient pass (fp32 64x56x56x128 7x7: 80.5 -> 77.6 us).
cudaError_t launch_reduce_slices(const float* part, int slices, size_t count, float* out,
                                 cudaStream_t stream) {
    if (count == 0) return cudaSuccess;
    const size_t cap = static_cast<size_t>(device_info().sm_count) * 8;   // one wave
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kReduceWarps * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (count % 4 == 0 && reinterpret_cast<uintptr_t>(part) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(out) % 16 == 0) {
        const size_t count4 = count / 4;
        cfg.gridDim = dim3(static_cast<unsigned>(std::min<size_t>((count4 + 31) / 32, cap)));
        return cudaLaunchKernelEx(&cfg, reduce_slices4_kernel, reinterpret_cast<const float4*>(part), slices,
                                  count4, reinterpret_cast<float4*>(out));
    }
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<size_t>((count + 31) / 32, cap)));
    return cudaLaunchKernelEx(&cfg, reduce_slices_kernel, part, slices, count, out);
}

static unsigned grid_for(long long total, int threads) {
    const long long cap = static_cast<long long>(device_info().sm_count) * 16;
    return static_cast<unsigned>(std::max<long long>(1, std::min(cap, (total + threads - 1) / threads)));
}

template <typename T>
static cudaError_t general_fwd_t(const GeneralConv& p) {
    const long long total = static_cast<long long>(p.N) * p.OH * p.OW * p.C;
    if (total == 0) return cudaSuccess;
    if (p.act >= 0) {
        general_fwd_bnact_kernel<T><<<grid_for(total, 256), 256, 0, p.stream>>>(
            static_cast<const T*>(p.a), static_cast<const T*>(p.b), static_cast<float*>(p.out), p.N, p.H, p.W, p.C,
            p.OH, p.OW, p.FH, p.FW, p.stride, p.pad, p.bn_mean, p.bn_var, p.bn_gamma, p.bn_beta,
            p.bn_eps, p.act);
        return cudaGetLastError();
    }
    if (p.out_dtype != kF32)
        general_fwd_kernel<T, T><<<grid_for(total, 256), 256, 0, p.stream>>>(
            static_cast<const T*>(p.a), static_cast<const T*>(p.b), static_cast<T*>(p.out), p.N, p.H,
            p.W, p.C, p.OH, p.OW, p.FH, p.FW, p.stride, p.pad);
    else
        general_fwd_kernel<T, float><<<grid_for(total, 256), 256, 0, p.stream>>>(
            static_cast<const T*>(p.a), static_cast<const T*>(p.b), static_cast<float*>(p.out), p.N,
            p.H, p.W, p.C, p.OH, p.OW, p.FH, p.FW, p.stride, p.pad);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t general_bwd_data_t(const GeneralConv& p) {
    const long long total = static_cast<long long>(p.N) * p.H * p.W * p.C;
    if (total == 0) return cudaSuccess;
    if (p.out_dtype != kF32)
        general_bwd_data_kernel<T, T><<<grid_for(total, 256), 256, 0, p.stream>>>(
            static_cast<const T*>(p.a), static_cast<const T*>(p.b), static_cast<T*>(p.out), p.N, p.H,
            p.W, p.C, p.OH, p.OW, p.FH, p.FW, p.stride, p.pad);
    else
        general_bwd_data_kernel<T, float><<<grid_for(total, 256), 256, 0, p.stream>>>(
            static_cast<const T*>(p.a), static_cast<const T*>(p.b), static_cast<float*>(p.out), p.N,
            p.H, p.W, p.C, p.OH, p.OW, p.FH, p.FW, p.stride, p.pad);
    return cudaGetLastError();
}

static int general_slices(int N, int OH, int C, int FH, int FW) {
    const long long outs = static_cast<long long>(FH) * FW * C;
    const long long target = static_cast<long long>(device_info().sm_count) * 1024;
    long long z = (target + outs - 1) / std::max<long long>(outs, 1);
    const long long rows = static_cast<long long>(N) * OH;
    z = std::max<long long>(1, std::min<long long>(z, std::max<long long>(rows, 1)));
    return static_cast<int>(z);
}

size_t general_bwd_filter_workspace_floats(int N, int OH, int C, int FH, int FW) {
    return static_cast<size_t>(general_slices(N, OH, C, FH, FW)) * FH * FW * C;
}

template <typename T>
static cudaError_t general_bwd_filter_t(const GeneralConv& p) {
    const size_t count = static_cast<size_t>(p.FH) * p.FW * p.C;
    if (count == 0) return cudaSuccess;
    const long long rows = static_cast<long long>(p.N) * p.OH;
    float* dw = static_cast<float*>(p.out);
    if (rows == 0 || p.OW == 0) return cudaMemsetAsync(dw, 0, count * sizeof(float), p.stream);
    int Z = general_slices(p.N, p.OH, p.C, p.FH, p.FW);
    const int rps = static_cast<int>((rows + Z - 1) / Z);
    Z = static_cast<int>((rows + rps - 1) / rps);
    if (p.workspace == nullptr || p.workspace_floats < count * Z) return cudaErrorInvalidValue;
    const long long total = static_cast<long long>(count) * Z;
    general_bwd_filter_kernel<T><<<grid_for(total, 256), 256, 0, p.stream>>>(
        static_cast<const T*>(p.a), static_cast<const T*>(p.b), p.workspace, p.N, p.H, p.W, p.C,
        p.OH, p.OW, p.FH, p.FW, p.stride, p.pad, rps, Z);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return launch_reduce_slices(p.workspace, Z, count, dw, p.stream);
}

#define DWC_BY_DTYPE(fn, p)                                         \
    switch ((p).dtype) {                                            \
        case kF32: return fn<float>(p);                             \
        case kBF16: return fn<__nv_bfloat16>(p);                    \
        case kF16: return fn<__half>(p);                            \
        default: return cudaErrorInvalidValue;                      \
    }

cudaError_t launch_general_fwd(const GeneralConv& p) { DWC_BY_DTYPE(general_fwd_t, p) }
cudaError_t launch_general_bwd_data(const GeneralConv& p) { DWC_BY_DTYPE(general_bwd_data_t, p) }
cudaError_t launch_general_bwd_filter(const GeneralConv& p) { DWC_BY_DTYPE(general_bwd_filter_t, p) }

}  // namespace dwc
