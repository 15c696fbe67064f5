// dwc_mma.cuh -- tensor-core forward / backward-data kernel for 16-bit inputs (bf16, fp16),
// fp32 accumulation and output.
//
// The GEMV -> GEMM transformation of "Flash-DWC: Making Depthwise Convolution
// Compute-Efficient on GPUs", §4.2 (Fig. 7), restated for the warp-level MMA of sm_103a
// (mma.sync m16n8k16, 16-bit inputs, fp32 accumulators):
//
//   for one channel and one filter row fh, the outputs of a group of 8 consecutive output
//   columns are D[g, n] = sum_k A[g, k] * B[k, n]   (output column 8*gc(g) + n)
//   A[g, k] = x[row(g) + fh, 8*gc(g) + k]            (Hankel: groups overlap by K - 8 inputs)
//   B[k, n] = w[fh, k - n] if 0 <= k - n < FW else 0 (Toeplitz of the filter row)
//
// with K = 16 * KC >= FW + 7 (KC K-steps of 16; the density of B is FW / K, e.g. 31/48).
// Summing over fh gives the 2-D convolution.  One M-tile is 16 groups; the groups of a tile
// may lie in different output rows because every lane supplies its own ldmatrix row address,
// so a band of output rows is covered without padding the row width to a tile multiple.
//
// Data flow per work unit (image n, band of RB output rows, block of 8 channels):
//  * all threads load the band's RB+FH-1 input rows (16-byte loads of 8 channels per pixel)
//    and store them transposed, channel-major, into shared memory (one row of a channel is
//    contiguous along width, which is what the Hankel rows of A need); out-of-image pixels
//    are stored as zeros (the padding);
//  * each warp owns two channels and keeps 7 M-tiles x 4 fp32 accumulators per channel; for
//    every (fh, K-step) it builds the two B registers of each channel from the filter tile
//    and issues ldmatrix.x4 (A) + mma per tile and channel;
//  * the accumulators go through shared memory to 16-byte coalesced fp32 stores.
// Backward data uses the same kernel with the filter read rotated by 180 degrees.
#pragma once

#include <type_traits>

#include <algorithm>

#include "dwc_rows.cuh"

namespace dwc {

constexpr int kMmaCB = 8;       // channels per work unit
constexpr int kMmaWarps = 4;    // two channels per warp
constexpr int kMmaTiles = 7;    // M-tiles of 16 groups per channel and warp (112 groups)
constexpr int kMmaMaxKC = 4;    // K <= 64, i.e. FW <= 57

struct MmaArgs {
    const void* x;
    const void* w;
    void* y;            // OutT elements
    int N, H, W, C, OH, OW, FH, FW, pad_h, pad_w;
    int G;       // groups of 8 output columns per row
    int RB;      // output rows per band
    int KC;      // K-steps of 16
    int XR, XC;  // rows / columns of one channel's transposed input block
    uint32_t cblocks, bands, units;
    uint32_t w_off;  // byte offset of the filter tile in shared memory
};

template <typename T>
struct MmaOp;

template <>
struct MmaOp<__nv_bfloat16> {
    __device__ static __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        // volatile: a skipped tile must not be executed speculatively
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

template <>
struct MmaOp<__half> {
    __device__ static __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

// Four 8x8 16-bit matrices from shared memory; lane L gives the address of row L%8 of
// matrix L/8 (16 contiguous bytes).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

template <typename T, bool FLIP, class OutT = float>
__global__ void __launch_bounds__(kMmaWarps * 32, 2) mma_rows_kernel(const MmaArgs a) {
    // a programmatic dependent of the kernel before it: nothing in global memory is touched
    // before that grid has finished
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(128) unsigned char smem[];
    uint16_t* xb = reinterpret_cast<uint16_t*>(smem);                 // [8][XR][XC]
    float* ob = reinterpret_cast<float*>(smem);                        // [RB][OW][8], after compute
    uint16_t* wb = reinterpret_cast<uint16_t*>(smem + a.w_off);        // [FH*FW][8]
    const uint32_t xb_s = smem_addr(xb);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const uint16_t* X = static_cast<const uint16_t*>(a.x);
    const uint16_t* Wg = static_cast<const uint16_t*>(a.w);
    const size_t plane = static_cast<size_t>(a.XR) * a.XC;

    // each CTA takes a contiguous range of units (channel block slowest), so the filter
    // tile in shared memory changes only when the channel block does
    const uint32_t per_cta = (a.units + gridDim.x - 1) / gridDim.x;
    const uint32_t u_begin = blockIdx.x * per_cta;
    const uint32_t u_end = min(a.units, u_begin + per_cta);
    int loaded_cb = -1;
    for (uint32_t u = u_begin; u < u_end; ++u) {
        uint32_t q = u;
        const int band = static_cast<int>(q % a.bands); q /= a.bands;
        const int n = static_cast<int>(q % a.N); q /= a.N;
        const int cb = static_cast<int>(q);
        const int oh0 = band * a.RB;
        const int c0 = cb * kMmaCB;
        const int rows = min(a.RB, a.OH - oh0);
        const int xrows = rows + a.FH - 1;

        // filter tile: 8 channels of every tap (16 bytes per tap)
        if (cb != loaded_cb) {
            for (int i = tid; i < a.FH * a.FW; i += blockDim.x)
                *reinterpret_cast<uint4*>(wb + i * kMmaCB) =
                    __ldg(reinterpret_cast<const uint4*>(Wg + static_cast<size_t>(i) * a.C + c0));
            loaded_cb = cb;
        }
        // input block, transposed to channel-major, zeros outside the image.  Eight
        // independent 16-byte loads are in flight per thread before their stores.
        constexpr int kBatch = 8;
        const int npx = xrows * a.XC;
        for (int base = tid; base < npx; base += kBatch * blockDim.x) {
            uint4 v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = base + j * blockDim.x;
                v[j] = make_uint4(0u, 0u, 0u, 0u);
                if (i < npx) {
                    const int xr = i / a.XC, xc = i - xr * a.XC;
                    const int ih = oh0 - a.pad_h + xr, iw = xc - a.pad_w;
                    if (ih >= 0 && ih < a.H && iw >= 0 && iw < a.W)
                        v[j] = __ldg(reinterpret_cast<const uint4*>(
                            X + ((static_cast<size_t>(n) * a.H + ih) * a.W + iw) * a.C + c0));
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = base + j * blockDim.x;
                if (i < npx) {
                    const uint32_t e[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                    uint16_t* dst = xb + i;  // (xr, xc) -> xr * XC + xc == i
#pragma unroll
                    for (int cc = 0; cc < kMmaCB; ++cc)
                        dst[cc * plane] = static_cast<uint16_t>(e[cc >> 1] >> ((cc & 1) * 16));
                }
            }
        }
        __syncthreads();

        const int ngroups = rows * a.G;
        const int ntiles = (ngroups + 15) >> 4;
        const int cl0 = 2 * warp;  // this warp's two channels
        float acc[2][kMmaTiles][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int t = 0; t < kMmaTiles; ++t)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[h][t][j] = 0.f;

        // ldmatrix row address of each tile for fh = 0, K-step 0 (channel cl0), and the
        // filter rows / K-steps for which some group of the tile reads inside the image:
        // the rest multiply only zero padding and are skipped (§4.4 trims shared zero rows).
        uint32_t arow[kMmaTiles];
        int fh_lo[kMmaTiles], fh_hi[kMmaTiles], kc_lo[kMmaTiles], kc_hi[kMmaTiles];
#pragma unroll
        for (int t = 0; t < kMmaTiles; ++t) {
            int qg = 16 * t + (lane & 7) + 8 * ((lane >> 3) & 1);
            if (qg >= ngroups) qg = 0;  // tile padding: any valid row, result discarded
            const int r = qg / a.G, gc = qg - r * a.G;
            arow[t] = xb_s + static_cast<uint32_t>(((cl0 * a.XR + r) * a.XC + 8 * gc + 8 * (lane >> 4)) * 2);
            const int q0 = 16 * t, q1 = min(16 * t + 15, ngroups - 1);
            const int r0 = q0 / a.G, r1 = q1 / a.G;          // rows spanned by the tile
            const int g0 = (r0 == r1) ? q0 - r0 * a.G : 0;     // group columns spanned
            const int g1 = (r0 == r1) ? q1 - r1 * a.G : a.G - 1;
            // input row oh0 - pad_h + r + fh inside [0, H) for some r in [r0, r1]
            fh_lo[t] = max(0, a.pad_h - oh0 - r1);
            fh_hi[t] = min(a.FH, a.H + a.pad_h - oh0 - r0);
            // K-step kc of group gc reads block columns 8*gc + 16*kc + [0, 16), i.e. input
            // columns minus pad_w; it is needed iff that range meets [pad_w, pad_w + W) for
            // some gc in [g0, g1]: kc in [ceil((pad_w - 15 - 8*g1) / 16),
            //                             floor((pad_w + W - 1 - 8*g0) / 16)]
            const int lo_num = a.pad_w - 15 - 8 * g1;
            const int hi_num = a.pad_w + a.W - 1 - 8 * g0;
            kc_lo[t] = lo_num <= 0 ? 0 : (lo_num + 15) / 16;
            kc_hi[t] = hi_num < 0 ? 0 : min(a.KC, hi_num / 16 + 1);
        }
        const uint32_t plane_b = static_cast<uint32_t>(plane * 2);
        int fh_begin = a.FH, fh_end = 0, kc_begin = a.KC, kc_end = 0;
#pragma unroll
        for (int t = 0; t < kMmaTiles; ++t)
            if (t < ntiles) {
                fh_begin = min(fh_begin, fh_lo[t]);
                fh_end = max(fh_end, fh_hi[t]);
                kc_begin = min(kc_begin, kc_lo[t]);
                kc_end = max(kc_end, kc_hi[t]);
            }

        for (int fh = fh_begin; fh < fh_end; ++fh) {
            const int fhe = FLIP ? a.FH - 1 - fh : fh;
            const uint16_t* wrow = wb + fhe * a.FW * kMmaCB;
            for (int kc = kc_begin; kc < kc_end; ++kc) {
                // B[k][n] = w[fh][16*kc + k - n]; this lane holds k = 2tq, 2tq+1 (b0) and
                // k = 2tq+8, 2tq+9 (b1) of column n = g, for both of its channels
                uint32_t b[2][2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int k = 2 * tq + (j & 1) + 8 * (j >> 1);
                        const int fw = 16 * kc + k - g;
                        const int fwe = FLIP ? a.FW - 1 - fw : fw;
                        v[j] = (fw >= 0 && fw < a.FW) ? wrow[fwe * kMmaCB + cl0 + h] : 0u;
                    }
                    b[h][0] = v[0] | (v[1] << 16);
                    b[h][1] = v[2] | (v[3] << 16);
                }
                const uint32_t off = static_cast<uint32_t>((fh * a.XC + 16 * kc) * 2);
#pragma unroll
                for (int t = 0; t < kMmaTiles; ++t) {
                    if (t < ntiles && fh >= fh_lo[t] && fh < fh_hi[t] && kc >= kc_lo[t] &&
                        kc < kc_hi[t]) {
                        uint32_t af[4], ag[4];
                        ldsm_x4(af, arow[t] + off);
                        ldsm_x4(ag, arow[t] + off + plane_b);
                        MmaOp<T>::mma(acc[0][t], af, b[0][0], b[0][1]);
                        MmaOp<T>::mma(acc[1][t], ag, b[1][0], b[1][1]);
                    }
                }
            }
        }
        __syncthreads();  // every warp is done with the input block: reuse it for outputs

        // D[g][n] of tile t -> group 16t + g (+8), output column 8*gc + n
#pragma unroll
        for (int t = 0; t < kMmaTiles; ++t) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int qg = 16 * t + g + 8 * hh;
                if (qg < ngroups) {
                    const int r = qg / a.G, gc = qg - r * a.G;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int ow = 8 * gc + 2 * tq + j;
                        if (ow < a.OW) {
                            float* o = ob + (static_cast<size_t>(r) * a.OW + ow) * kMmaCB + cl0;
                            o[0] = acc[0][t][2 * hh + j];
                            o[1] = acc[1][t][2 * hh + j];
                        }
                    }
                }
            }
        }
        __syncthreads();
        // 16-byte coalesced fp32 stores: two per pixel (8 channels)
        for (int i = tid; i < rows * a.OW * 2; i += blockDim.x) {
            const int px = i >> 1, half = i & 1;
            const int r = px / a.OW, ow = px - r * a.OW;
            const float4 v = *reinterpret_cast<const float4*>(ob + static_cast<size_t>(px) * kMmaCB + 4 * half);
            OutT* dst = static_cast<OutT*>(a.y) + ((static_cast<size_t>(n) * a.OH + oh0 + r) * a.OW + ow) * a.C + c0 + 4 * half;
            if constexpr (std::is_same<OutT, float>::value) {
                __stcs(reinterpret_cast<float4*>(dst), v);
            } else {
                store_out_pair(dst, make_float2(v.x, v.y));
                store_out_pair(dst + 2, make_float2(v.z, v.w));
            }
        }
        __syncthreads();  // the block is overwritten by the next unit's loads
    }
}

// Launch plan; false if the shape does not fit the kernel's limits.
inline bool mma_plan(const RowConv& p, MmaArgs& a, size_t& smem) {
    if (p.FW + 7 > 16 * kMmaMaxKC || p.FH < 1 || p.C % kMmaCB != 0) return false;
    a.G = (p.OW + 7) / 8;
    if (a.G > 16 * kMmaTiles) return false;
    a.RB = std::max(1, std::min(p.OH, (16 * kMmaTiles) / a.G));
    a.KC = (p.FW + 7 + 15) / 16;
    a.XR = a.RB + p.FH - 1;
    // Row pitch in 16-byte chunks congruent to G mod 8: the Hankel rows of consecutive
    // groups (q = r*G + gc) then start in consecutive 16-byte bank groups even across image
    // rows, so each 8-row ldmatrix phase is conflict-free.
    {
        const int need = a.G + 2 * a.KC - 1;  // chunks read per row
        const int p16 = a.G + 8 * ((need - a.G + 7) / 8);
        a.XC = 8 * p16;
    }
    const size_t xbytes = static_cast<size_t>(kMmaCB) * a.XR * a.XC * 2;
    const size_t obytes = static_cast<size_t>(a.RB) * p.OW * kMmaCB * 4;
    const size_t wbytes = static_cast<size_t>(p.FH) * p.FW * kMmaCB * 2;
    a.w_off = static_cast<uint32_t>((std::max(xbytes, obytes) + 127) & ~size_t(127));
    smem = a.w_off + wbytes;
    if (smem > static_cast<size_t>(device_info().max_smem_optin)) return false;
    a.cblocks = static_cast<uint32_t>(p.C / kMmaCB);
    a.bands = static_cast<uint32_t>((p.OH + a.RB - 1) / a.RB);
    const long long units = static_cast<long long>(p.N) * a.bands * a.cblocks;  // band fastest
    if (units >= (1LL << 31)) return false;
    a.units = static_cast<uint32_t>(units);
    return true;
}

template <typename T, bool FLIP, class OutT = float>
cudaError_t launch_mma_inst(const RowConv& p) {
    MmaArgs a;
    size_t smem = 0;
    if (!mma_plan(p, a, smem)) return cudaErrorNotSupported;
    a.x = p.in; a.w = p.w; a.y = p.out;
    a.N = p.N; a.H = p.H; a.W = p.W; a.C = p.C; a.OH = p.OH; a.OW = p.OW;
    a.FH = p.FH; a.FW = p.FW; a.pad_h = p.pad_h; a.pad_w = p.pad_w;
    if (a.units == 0) return cudaSuccess;
    auto kern = mma_rows_kernel<T, FLIP, OutT>;
    static DeviceOnce smem_opt_in;
    {
        const cudaError_t err = opt_in_smem(kern, smem_opt_in, device_info().max_smem_optin);
        if (err != cudaSuccess) return err;
    }
    const int ctas = smem * 2 + 2048 <= 233472u ? 2 : 1;
    const long long grid = std::min<long long>(a.units, static_cast<long long>(device_info().sm_count) * ctas);
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kMmaWarps * 32), smem, p.stream, a);
}

// Where the tensor-core kernel beats the row-streaming kernel for 16-bit inputs (timed on
// the stage shapes: from 15-tap filters on rows of at least 24 outputs -- at 13 taps the
// row kernel was 4-10 % faster, at 17 the tensor-core kernel 8-26 %; on narrower maps most
// of each tile's K-steps fall into the padding).
constexpr int kMmaMinFilter = 15;
constexpr int kMmaMinWidth = 24;

inline bool mma_rows_wanted(const RowConv& p) {
    return p.FW >= kMmaMinFilter && p.OW >= kMmaMinWidth;
}

// 16-bit forward / backward data: the tcgen05 kernel, the warp-level MMA kernel or the row
// kernel, in that order of preference where each serves the shape (a family preference set
// for tests and kernel comparisons picks one of them where it can run).
template <typename T, class OutT = float>
cudaError_t launch_rows_or_mma(const RowConv& p) {
    const int pref = family_preference();
    if ((pref == 0 && tc_rows_wanted(p)) || pref == kFamilyTcgen05) {
        const cudaError_t err = std::is_same<T, __nv_bfloat16>::value ? launch_tc_rows_bf16(p)
                                                                      : launch_tc_rows_f16(p);
        if (err != cudaErrorNotSupported) return err;
        (void)cudaGetLastError();
    }
    if ((pref == 0 && mma_rows_wanted(p)) || pref == kFamilyMmaSync) {
        const cudaError_t err = p.flip ? launch_mma_inst<T, true, OutT>(p) : launch_mma_inst<T, false, OutT>(p);
        if (err != cudaErrorNotSupported) return err;
        (void)cudaGetLastError();
    }
    return launch_rows_dispatch<T, OutT>(p);
}

}  // namespace dwc
