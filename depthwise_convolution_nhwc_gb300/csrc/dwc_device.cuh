// dwc_device.cuh -- device-side building blocks shared by the DWC kernels (sm_103a).
//
// mbarrier + TMA (cp.async.bulk.tensor) staging with bounded waits, packed fp32x2 FMA,
// and 16-bit -> fp32 pair conversion.  Every wait on an mbarrier has a time limit: when
// it runs out the kernel records DWC_DEVSTAT_TIMEOUT in the status word it was given
// and winds down instead of spinning forever.
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dwc_host.h"

namespace dwc {

// Bits of the device status word (a 32-bit word in global memory, read by the host).
enum : unsigned int {
    DWC_DEVSTAT_TIMEOUT = 1u,   // an mbarrier wait ran out of time
};

// Default upper bound on one mbarrier wait.  A healthy wait lasts microseconds; the limit
// only ends a kernel whose copies never arrive.  Launches carry the limit as an argument
// (dwc_set_wait_limit_ns changes it for later launches).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if `limit_ns` ran out
// (the caller then records the timeout and winds down).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Position in a ring of `n` pipeline stages: the slot and the parity of its current use.
// Advanced by one stage at a time, so no division is ever needed in the hot loops.
struct Ring {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void next(uint32_t n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// Programmatic dependent launch: a kernel whose output the next kernel of the stream sums
// (the filter gradients' partial slices) lets that kernel be scheduled while it still runs;
// the dependent waits, before reading anything, until this grid has finished and its writes
// are visible.  Both are no-ops for kernels launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kern` as a programmatic dependent of the kernel before it in the stream.  The
// kernel must call pdl_wait() before it touches global memory: the previous grid (whatever
// wrote its inputs or still reads its outputs) has then finished.
template <class K, class... Args>
cudaError_t launch_pdl(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

__device__ __forceinline__ void record_status(unsigned int* status, unsigned int bits) {
    if (status) atomicOr(status, bits);
}

// --- TMA tiled loads (global -> shared, completion counted on an mbarrier) -------------
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// --- division by a launch-time constant ---------------------------------------------------
// q / d for q < 2^31 and a divisor fixed on the host, with one multiply-high, an add and a
// shift instead of the runtime's general division (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994): s = ceil(log2 d),
// m = floor(2^32 * (2^s - d) / d) + 1, then q / d = (umulhi(q, m) + q) >> s, where the sum
// stays below 2^32 because umulhi(q, m) <= q < 2^31.
struct FastDiv {
    uint32_t d = 1, m = 1, s = 0;
    __host__ void init(uint32_t div) {
        d = div < 1 ? 1 : div;
        s = 0;
        while ((1ull << s) < d) ++s;
        m = static_cast<uint32_t>((((1ull << 32) * ((1ull << s) - d)) / d) + 1);
    }
    __device__ __forceinline__ uint32_t div(uint32_t q) const { return (__umulhi(q, m) + q) >> s; }
    // quotient, and q - quotient * d in `rem`
    __device__ __forceinline__ uint32_t divmod(uint32_t q, uint32_t& rem) const {
        const uint32_t t = div(q);
        rem = q - t * d;
        return t;
    }
};

// --- arithmetic ------------------------------------------------------------------------
// acc += a * b on two fp32 lanes at once (one packed FMA instruction on sm_100+).
__device__ __forceinline__ void fma2(float2& acc, float2 a, float2 b) {
    acc = __ffma2_rn(a, b, acc);
}

// Arithmetic on a pair of adjacent channels held as one 64-bit register (two fp32 lanes).
// Keeping the pair as a single 64-bit value from the shared-memory load to the packed FMA
// lets the register allocator place it in an aligned register pair once, instead of
// assembling pairs around every packed FMA (on the 7x7 forward, float2 values with the
// packed-FMA builtin timed the same and two scalar FMAs per pair 28 % slower).
struct Pair64 {
    using V = unsigned long long;
    __device__ static __forceinline__ V zero() { return 0ull; }
    __device__ static __forceinline__ void fma(V& acc, V a, V b) {
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
    }
    __device__ static __forceinline__ V pack(float lo, float hi) {
        V r;
        asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
        return r;
    }
    __device__ static __forceinline__ float2 unpack(V v) {
        float2 f;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
        return f;
    }
    __device__ static __forceinline__ V load(const float* p) {
        return *reinterpret_cast<const unsigned long long*>(p);
    }
    __device__ static __forceinline__ V load(const __nv_bfloat16* p) {
        // bf16 -> fp32 is exact: the 16 bits become the high half of the fp32 word
        const unsigned u = *reinterpret_cast<const unsigned*>(p);
        V r;
        asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(u << 16), "r"(u & 0xffff0000u));
        return r;
    }
    __device__ static __forceinline__ V load(const __half* p) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(p));
        return pack(f.x, f.y);
    }
};

// Element type traits: how two adjacent channels are loaded from shared memory and
// widened to fp32 (exact for bf16 and fp16).
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    using pair_t = float2;
    static constexpr int kBytes = 4;
    static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    __device__ static __forceinline__ float2 load_pair(const float* p) {
        return *reinterpret_cast<const float2*>(p);
    }
};

template <>
struct Elem<__nv_bfloat16> {
    using pair_t = __nv_bfloat162;
    static constexpr int kBytes = 2;
    static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // bf16 -> fp32 is exact: the fp32 bit pattern is the bf16 one shifted up by 16, so the
    // pair widens with one shift and one mask
    __device__ static __forceinline__ float2 load_pair(const __nv_bfloat16* p) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
};

template <>
struct Elem<__half> {
    using pair_t = __half2;
    static constexpr int kBytes = 2;
    static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    __device__ static __forceinline__ float2 load_pair(const __half* p) {
        return __half22float2(*reinterpret_cast<const __half2*>(p));
    }
};

// Scalar widening for the generic kernels.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }

// Streaming store of an fp32 pair (outputs are written once and not re-read).
__device__ __forceinline__ void store_pair_streaming(float* p, float2 v) {
    __stcs(reinterpret_cast<float2*>(p), v);
}

// Streaming store of an fp32 pair as the output type: fp32 as is, bf16 / fp16 rounded to
// nearest even (the fp32 accumulators round once, at the store).
__device__ __forceinline__ void store_out_pair(float* p, float2 v) { store_pair_streaming(p, v); }
__device__ __forceinline__ void store_out_pair(__nv_bfloat16* p, float2 v) {
    const __nv_bfloat162 h = __float22bfloat162_rn(v);
    __stcs(reinterpret_cast<unsigned int*>(p), *reinterpret_cast<const unsigned int*>(&h));
}
__device__ __forceinline__ void store_out_pair(__half* p, float2 v) {
    const __half2 h = __float22half2_rn(v);
    __stcs(reinterpret_cast<unsigned int*>(p), *reinterpret_cast<const unsigned int*>(&h));
}
// one value, for the general kernels
__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store_out(__half* p, float v) { *p = __float2half_rn(v); }


// ------------------------------------------------------------------ host-side occupancy

// Once-only flags of one kernel, one per device: cudaFuncSetAttribute applies to the current
// device only, so a process that uses several GPUs opts a kernel in on each of them.
struct DeviceOnce {
    std::atomic<bool> done[kMaxDevices] = {};
};

// Let `kern` use the device's whole opt-in shared memory on the current device (once per
// device; a failed attempt is retried at the next launch).  `once` belongs to the kernel:
// instantiations of one kernel template share a function type, so the caller keeps one
// DeviceOnce per instantiation (a function-local static next to the launch).
template <class K>
cudaError_t opt_in_smem(K kern, DeviceOnce& once, int max_smem_optin) {
    int d = 0;
    cudaError_t err = cudaGetDevice(&d);
    if (err != cudaSuccess) return err;
    const bool tracked = d >= 0 && d < kMaxDevices;
    if (tracked && once.done[d].load(std::memory_order_acquire)) return cudaSuccess;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin);
    if (err == cudaSuccess && tracked) once.done[d].store(true, std::memory_order_release);
    return err;
}

// Registers per thread of a kernel (allocation granularity of 8), or `fallback` when the
// runtime cannot say (no device).
template <class K>
int kernel_regs(K kern, int fallback) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
        (void)cudaGetLastError();
        return fallback;
    }
    return (fa.numRegs + 7) / 8 * 8;
}

// Resident CTAs per SM from dynamic shared memory, threads and registers (the register file
// is allocated per warp in units of 256 registers; 1 KB of shared memory is reserved per CTA).
inline int resident_ctas(size_t smem, int threads, int regs) {
    const int warps = (threads + 31) / 32;
    const int by_smem = static_cast<int>(233472 / (smem + 1024));
    const int by_threads = 2048 / (warps * 32);
    const int by_regs = 65536 / (((regs * 32 + 255) / 256) * 256 * warps);
    int r = by_smem < by_threads ? by_smem : by_threads;
    if (by_regs < r) r = by_regs;
    return r < 1 ? 1 : r;
}

}  // namespace dwc
