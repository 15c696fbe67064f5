// dwc_bnact_split.cu -- BN + Act + forward DWC as two passes, for 7x7 filters at stride 1.
//
// The fused row kernel applies the per-channel affine map and the activation to every
// staged input value in every warp that reads it: about 7 times per element at 7x7 (each
// input row is staged for 4 bands, and neighbouring warps share 6 columns of halo), which
// adds about half again to a kernel already limited by instruction issue (fp32
// 64x56x56x128: 122 us fused against 70 us for the plain forward).  Here one pass writes
// act(BN(x)) once per element as fp32 into scratch memory and the plain fp32 forward runs on
// it: the extra HBM traffic (read x, write and read the fp32 copy) costs less than the
// transforms.  The arithmetic is the fused kernel's: z = fma(x, scale, shift) in fp32 with
// scale = gamma / sqrt(var + eps), shift = beta - mean * scale, then the activation, and the
// forward zero-pads z; 16-bit inputs and filters are widened exactly.  Measured (CUDA events):
// fp32 64x56x56x128 122 -> 109 us, 64x28x28x256 75 -> 65 us, bf16 64x56x56x128 131 -> 106 us;
// on 14-wide maps the two forms tie (40 us), so rows narrower than 28 keep the fused kernel.
#include "dwc_device.cuh"
#include "dwc_host.h"

namespace dwc {
namespace {

template <typename T>
__device__ __forceinline__ float widen(T v) {
    if constexpr (std::is_same<T, float>::value) return v;
    else if constexpr (std::is_same<T, __nv_bfloat16>::value) return __bfloat162float(v);
    else return __half2float(v);
}

template <typename T>
struct Quad;
template <>
struct Quad<float> {
    __device__ static __forceinline__ float4 load(const float* p) { return *reinterpret_cast<const float4*>(p); }
};
template <>
struct Quad<__nv_bfloat16> {
    __device__ static __forceinline__ float4 load(const __nv_bfloat16* p) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
};
template <>
struct Quad<__half> {
    __device__ static __forceinline__ float4 load(const __half* p) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
};

__device__ __forceinline__ float act_of(float t, int act) {
    if (act >= 1) t = fmaxf(t, 0.f);
    if (act == 2) t = fminf(t, 6.f);
    return t;
}

// z = act(x * scale[c] + shift[c]) for 4 consecutive channels per thread (C % 4 == 0).  The
// grid's thread count is a multiple of C / 4, so a thread keeps one channel quad (its scale
// and shift computed once) and strides over pixels.
template <typename T>
__global__ void __launch_bounds__(256) bnact_apply_kernel(const T* __restrict__ x, float4* __restrict__ z,
                                                          long long pixels, int C,
                                                          const float* __restrict__ mean,
                                                          const float* __restrict__ var,
                                                          const float* __restrict__ gamma,
                                                          const float* __restrict__ beta, float eps,
                                                          int act) {
    const int g4 = C / 4;
    const long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const int q = static_cast<int>(t % g4);
    const long long pstride = nthreads / g4;
    float sc[4], sh[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int c = 4 * q + k;
        sc[k] = gamma[c] * rsqrtf(var[c] + eps);
        sh[k] = beta[c] - mean[c] * sc[k];
    }
    for (long long p = t / g4; p < pixels; p += pstride) {
        const size_t i = static_cast<size_t>(p) * C + 4 * q;
        const float4 v = Quad<T>::load(x + i);
        z[i / 4] = make_float4(act_of(fmaf(v.x, sc[0], sh[0]), act), act_of(fmaf(v.y, sc[1], sh[1]), act),
                               act_of(fmaf(v.z, sc[2], sh[2]), act), act_of(fmaf(v.w, sc[3], sh[3]), act));
    }
}

template <typename T>
__global__ void __launch_bounds__(256) widen_kernel(const T* __restrict__ w, float* __restrict__ w32, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        w32[i] = widen(w[i]);
}

template <typename T>
cudaError_t apply_t(const RowConv& p, float* z, float* w32) {
    const long long pixels = static_cast<long long>(p.N) * p.H * p.W;
    const int g4 = p.C / 4;
    // blocks per period: the smallest block count whose threads are a multiple of C / 4
    int a0 = g4, b0 = 256;
    while (b0 != 0) { const int r = a0 % b0; a0 = b0; b0 = r; }
    const long long unit = g4 / a0;
    const long long want = (pixels * g4 + 255) / 256;
    const long long cap = static_cast<long long>(device_info().sm_count) * 8;
    const long long blocks = std::max<long long>(unit, std::min(want, cap) / unit * unit);
    if (blocks >= (1LL << 31)) return cudaErrorNotSupported;
    bnact_apply_kernel<T><<<static_cast<unsigned>(blocks), 256, 0, p.stream>>>(
        static_cast<const T*>(p.in), reinterpret_cast<float4*>(z), pixels, p.C, p.bn_mean, p.bn_var,
        p.bn_gamma, p.bn_beta, p.bn_eps, p.act);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || w32 == nullptr) return err;
    const int nw = p.FH * p.FW * p.C;
    widen_kernel<T><<<static_cast<unsigned>((nw + 255) / 256), 256, 0, p.stream>>>(
        static_cast<const T*>(p.w), w32, nw);
    return cudaGetLastError();
}

}  // namespace

bool bnact_split_serves(int FH, int FW, int stride, int C, int W) {
    return FH == 7 && FW == 7 && stride == 1 && C % 4 == 0 && W >= 28;
}

cudaError_t launch_bnact_split(const RowConv& p, int stride) {
    if (!bnact_split_serves(p.FH, p.FW, stride, p.C, p.W) || p.act < 0 || p.flip) return cudaErrorNotSupported;
    const size_t nx = static_cast<size_t>(p.N) * p.H * p.W * p.C;
    const size_t zbytes = (nx * sizeof(float) + 255) & ~static_cast<size_t>(255);
    const size_t wbytes = p.dtype == kF32 ? 0 : static_cast<size_t>(p.FH) * p.FW * p.C * sizeof(float);
    void* buf = nullptr;
    cudaError_t err = scratch_alloc(&buf, zbytes + wbytes, p.stream);
    if (err != cudaSuccess) return err;
    float* z = static_cast<float*>(buf);
    float* w32 = wbytes ? reinterpret_cast<float*>(static_cast<unsigned char*>(buf) + zbytes) : nullptr;
    switch (p.dtype) {
        case kF32: err = apply_t<float>(p, z, nullptr); break;
        case kBF16: err = apply_t<__nv_bfloat16>(p, z, w32); break;
        default: err = apply_t<__half>(p, z, w32); break;
    }
    if (err == cudaSuccess) {
        RowConv q = p;
        q.in = z;
        q.w = w32 ? w32 : p.w;
        q.dtype = kF32;
        q.out_dtype = kF32;
        q.act = -1;
        q.bn_mean = q.bn_var = q.bn_gamma = q.bn_beta = nullptr;
        err = launch_rows_f32(q);
    }
    scratch_free(buf, p.stream);
    return err;
}

}  // namespace dwc
