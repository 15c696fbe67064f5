// dwc_probe.cu -- multiply-add rate microbenchmark of the CUDA cores (the compute peak that
// the roofline of the CUDA-core kernels is measured against) behind dwc_fma_rate_probe.
//
// Every thread runs `iters` iterations of kChains independent dependency chains
// acc = acc * a + b of one multiply-add instruction kind; with enough warps per scheduler
// the chains hide the instruction latency, so the launch time measures the issue rate of
// that instruction.  a = 0.5 and b = 0.25 keep every chain at its fixed point 0.5 (no
// overflow, no subnormals in any of the types).  One value per thread is stored so that no
// chain can be removed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dwc.h"

namespace {

constexpr int kChains = 8;
constexpr int kThreads = 256;

template <int KIND>
__global__ void __launch_bounds__(kThreads) fma_rate_kernel(float* out, int iters) {
    float result = 0.f;
    if constexpr (KIND == 0) {  // fp32 FFMA
        float acc[kChains];
#pragma unroll
        for (int j = 0; j < kChains; ++j) acc[j] = 0.125f * (j + threadIdx.x % 3);
        const float a = 0.5f, b = 0.25f;
#pragma unroll 1
        for (int i = 0; i < iters; ++i)
#pragma unroll
            for (int j = 0; j < kChains; ++j)
                asm("fma.rn.f32 %0, %0, %1, %2;" : "+f"(acc[j]) : "f"(a), "f"(b));
#pragma unroll
        for (int j = 0; j < kChains; ++j) result += acc[j];
    } else if constexpr (KIND == 1) {  // packed fp32x2 FFMA2
        unsigned long long acc[kChains];
        unsigned long long a, b;
        asm("mov.b64 %0, {%1, %1};" : "=l"(a) : "f"(0.5f));
        asm("mov.b64 %0, {%1, %1};" : "=l"(b) : "f"(0.25f));
#pragma unroll
        for (int j = 0; j < kChains; ++j) {
            const float v = 0.125f * (j + threadIdx.x % 3);
            asm("mov.b64 %0, {%1, %1};" : "=l"(acc[j]) : "f"(v));
        }
#pragma unroll 1
        for (int i = 0; i < iters; ++i)
#pragma unroll
            for (int j = 0; j < kChains; ++j)
                asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[j]) : "l"(a), "l"(b));
#pragma unroll
        for (int j = 0; j < kChains; ++j) {
            float lo, hi;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc[j]));
            result += lo + hi;
        }
    } else {  // packed 16-bit: 2 = fp16x2 HFMA2, 3 = bf16x2
        uint32_t acc[kChains];
        uint32_t a, b;
        if constexpr (KIND == 2) {
            const __half2 ha = __float2half2_rn(0.5f), hb = __float2half2_rn(0.25f);
            a = *reinterpret_cast<const uint32_t*>(&ha);
            b = *reinterpret_cast<const uint32_t*>(&hb);
        } else {
            const __nv_bfloat162 ha = __float2bfloat162_rn(0.5f), hb = __float2bfloat162_rn(0.25f);
            a = *reinterpret_cast<const uint32_t*>(&ha);
            b = *reinterpret_cast<const uint32_t*>(&hb);
        }
#pragma unroll
        for (int j = 0; j < kChains; ++j) acc[j] = (threadIdx.x % 3 == 0) ? a : b;
#pragma unroll 1
        for (int i = 0; i < iters; ++i)
#pragma unroll
            for (int j = 0; j < kChains; ++j) {
                if constexpr (KIND == 2)
                    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(acc[j]) : "r"(a), "r"(b));
                else
                    asm("fma.rn.bf16x2 %0, %0, %1, %2;" : "+r"(acc[j]) : "r"(a), "r"(b));
            }
#pragma unroll
        for (int j = 0; j < kChains; ++j) {
            if constexpr (KIND == 2) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&acc[j]));
                result += f.x + f.y;
            } else {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&acc[j]));
                result += f.x + f.y;
            }
        }
    }
    out[static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x] = result;
}

}  // namespace

extern "C" dwc_status_t dwc_fma_rate_probe(int kind, int blocks, int iters, float* out,
                                           dwc_stream_t stream) {
    if (kind < 0 || kind > 3 || blocks < 1 || iters < 1 || out == nullptr)
        return DWC_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(out) % 4 != 0) return DWC_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (kind) {
        case 0: fma_rate_kernel<0><<<blocks, kThreads, 0, s>>>(out, iters); break;
        case 1: fma_rate_kernel<1><<<blocks, kThreads, 0, s>>>(out, iters); break;
        case 2: fma_rate_kernel<2><<<blocks, kThreads, 0, s>>>(out, iters); break;
        default: fma_rate_kernel<3><<<blocks, kThreads, 0, s>>>(out, iters); break;
    }
    return cudaGetLastError() == cudaSuccess ? DWC_OK : DWC_ERR_CUDA;
}
