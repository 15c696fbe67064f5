// dwc_mma_fgrad.cuh -- tensor-core filter gradient for 16-bit inputs (bf16, fp16), fp32
// accumulation.
//
//   dw[fh, fw, c] = sum_{n, oh, ow} x[n, oh + fh - pad, ow + fw - pad, c] * dy[n, oh, ow, c]
//
// ("Flash-DWC: Making Depthwise Convolution Compute-Efficient on GPUs", §5.1, backward
// filter convolution.)  The pages run this pass on CUDA cores; here it becomes a GEMM with
// the same Hankel x Toeplitz structure as their §4.2 transformation, but with the roles of
// filter and data exchanged: for one channel and one output row (n, oh), the filter taps
// fw = 8*fg + nn of filter row fh receive
//   D[(fh, fg), nn] = sum_k A[(fh, fg), k] * B[k, nn]
//   A[(fh, fg), k]  = xp[oh + fh, 8*fg + k]    (x row oh + fh - pad, left-padded by pad)
//   B[k, nn]        = dy[oh, k - nn] if 0 <= k - nn < OW else 0   (Toeplitz of the dy row)
// with K = 16 * KC >= OW + 7, i.e. the density of B is OW / K (56/64 on 56-wide rows).
// An M-tile is 16 (fh, fg) pairs; all (n, oh) of a slice accumulate into the same tiles.
//
// Work: CTA (channel block of 8, slice z of the bands (n, band of RB output rows)).  Per
// band the x rows (RB + FH - 1) and dy rows (RB) are loaded transposed to channel-major in
// shared memory; each warp owns two channels.  At the end each CTA writes its partial
// gradient to workspace slot z, summed in a fixed order by reduce_slices_kernel.
#pragma once

#include "dwc_mma.cuh"

namespace dwc {

constexpr int kFgMaxTiles = 8;  // up to 128 (fh, fg) pairs: 31 x ceil(31/8) = 124

struct MmaFgArgs {
    const void* x;
    const void* dy;
    float* part;  // [Z][FH][FW][C]
    int N, H, W, C, OH, OW, FH, FW, pad;
    int NFG;      // filter-column groups of 8
    int ntiles;   // M-tiles of 16 (fh, fg) pairs
    int KC;       // K-steps of 16
    int RB;       // output rows per band
    int XR, XC;   // transposed x block: rows, pitch (elements)
    int DC;       // transposed dy block pitch (elements), dy column j stored at j + 8
    int bands, Z, bands_per_slice;
    uint32_t dy_off;  // byte offset of the dy block
};

template <typename T>
__global__ void __launch_bounds__(kMmaWarps * 32, 2) mma_fgrad_kernel(const MmaFgArgs a) {
    pdl_trigger();   // the slice sum may be scheduled now (it waits for this grid)
    pdl_wait();      // (a programmatic dependent itself: the grid before it has finished)
    extern __shared__ __align__(128) unsigned char smem[];
    uint16_t* xb = reinterpret_cast<uint16_t*>(smem);               // [8][XR][XC]
    uint16_t* db = reinterpret_cast<uint16_t*>(smem + a.dy_off);    // [8][RB][DC]
    const uint32_t xb_s = smem_addr(xb);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const uint16_t* X = static_cast<const uint16_t*>(a.x);
    const uint16_t* DY = static_cast<const uint16_t*>(a.dy);
    const size_t xplane = static_cast<size_t>(a.XR) * a.XC;
    const size_t dplane = static_cast<size_t>(a.RB) * a.DC;
    const int cb = blockIdx.x % (a.C / kMmaCB);
    const int z = blockIdx.x / (a.C / kMmaCB);
    const int c0 = cb * kMmaCB;
    const int cl0 = 2 * warp;
    const int total_bands = a.N * a.bands;
    const int b_begin = z * a.bands_per_slice;
    const int b_end = min(total_bands, b_begin + a.bands_per_slice);

    // M-tile rows: lane's ldmatrix row m = 16t + (lane & 7) + 8*((lane >> 3) & 1) is the pair
    // (fh, fg) = (m / NFG, m % NFG); k offset 8*(lane >> 4)
    int mrow_fh[kFgMaxTiles], mrow_fg[kFgMaxTiles], t_fh0[kFgMaxTiles], t_fh1[kFgMaxTiles];
#pragma unroll
    for (int t = 0; t < kFgMaxTiles; ++t) {
        int m = 16 * t + (lane & 7) + 8 * ((lane >> 3) & 1);
        if (m >= a.FH * a.NFG) m = 0;  // tile padding: a valid row, result discarded
        mrow_fh[t] = m / a.NFG;
        mrow_fg[t] = m - mrow_fh[t] * a.NFG;
        t_fh0[t] = (16 * t) / a.NFG;                                   // filter rows of the tile
        t_fh1[t] = min(a.FH - 1, (16 * t + 15) / a.NFG);
    }

    float acc[2][kFgMaxTiles][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int t = 0; t < kFgMaxTiles; ++t)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[h][t][j] = 0.f;

    for (int bi = b_begin; bi < b_end; ++bi) {
        const int n = bi / a.bands, band = bi - n * a.bands;
        const int oh0 = band * a.RB;
        const int rows = min(a.RB, a.OH - oh0);
        const int xrows = rows + a.FH - 1;

        // x rows oh0 - pad + [0, xrows), columns -pad + [0, XC), transposed; zeros outside
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
                    const int ih = oh0 - a.pad + xr, iw = xc - a.pad;
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
#pragma unroll
                    for (int cc = 0; cc < kMmaCB; ++cc)
                        xb[cc * xplane + i] = static_cast<uint16_t>(e[cc >> 1] >> ((cc & 1) * 16));
                }
            }
        }
        // dy rows oh0 + [0, rows); dy column j stored at j + 8, zeros around
        const int nd = rows * a.DC;
        for (int base = tid; base < nd; base += kBatch * blockDim.x) {
            uint4 v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = base + j * blockDim.x;
                v[j] = make_uint4(0u, 0u, 0u, 0u);
                if (i < nd) {
                    const int r = i / a.DC, col = i - r * a.DC - 8;
                    if (col >= 0 && col < a.OW)
                        v[j] = __ldg(reinterpret_cast<const uint4*>(
                            DY + ((static_cast<size_t>(n) * a.OH + oh0 + r) * a.OW + col) * a.C + c0));
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = base + j * blockDim.x;
                if (i < nd) {
                    const uint32_t e[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                    for (int cc = 0; cc < kMmaCB; ++cc)
                        db[cc * dplane + i] = static_cast<uint16_t>(e[cc >> 1] >> ((cc & 1) * 16));
                }
            }
        }
        __syncthreads();

        for (int r = 0; r < rows; ++r) {
            // x rows of this output row: oh0 + r + fh - pad; a tile whose filter rows all
            // land in the padding contributes nothing
            const int fh_ok0 = a.pad - oh0 - r, fh_ok1 = a.H + a.pad - oh0 - r;  // [fh_ok0, fh_ok1)
            const uint16_t* drow0 = db + static_cast<size_t>(cl0) * dplane + static_cast<size_t>(r) * a.DC;
            for (int kc = 0; kc < a.KC; ++kc) {
                // B[k][nn] = dy[16*kc + k - nn]: k = 2tq (+1), 2tq+8 (+1); nn = g
                uint32_t b[2][2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint16_t* d = drow0 + h * dplane + 16 * kc - g + 8;
                    b[h][0] = static_cast<uint32_t>(d[2 * tq]) | (static_cast<uint32_t>(d[2 * tq + 1]) << 16);
                    b[h][1] = static_cast<uint32_t>(d[2 * tq + 8]) | (static_cast<uint32_t>(d[2 * tq + 9]) << 16);
                }
#pragma unroll
                for (int t = 0; t < kFgMaxTiles; ++t) {
                    if (t < a.ntiles && t_fh1[t] >= fh_ok0 && t_fh0[t] < fh_ok1) {
                        const uint32_t addr = xb_s + static_cast<uint32_t>(
                            (((cl0 * a.XR) + r + mrow_fh[t]) * a.XC + 8 * mrow_fg[t] + 16 * kc +
                             8 * (lane >> 4)) * 2);
                        uint32_t af[4], ag[4];
                        ldsm_x4(af, addr);
                        ldsm_x4(ag, addr + static_cast<uint32_t>(xplane * 2));
                        MmaOp<T>::mma(acc[0][t], af, b[0][0], b[0][1]);
                        MmaOp<T>::mma(acc[1][t], ag, b[1][0], b[1][1]);
                    }
                }
            }
        }
        __syncthreads();  // the blocks are reloaded for the next band
    }

    // partial gradient of this slice: D[(fh, fg)][nn] -> dw[fh][8*fg + nn]
    float* out = a.part + static_cast<size_t>(z) * a.FH * a.FW * a.C + c0 + cl0;
#pragma unroll
    for (int t = 0; t < kFgMaxTiles; ++t) {
        if (t >= a.ntiles) continue;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int m = 16 * t + g + 8 * hh;
            if (m >= a.FH * a.NFG) continue;
            const int fh = m / a.NFG, fg = m - (m / a.NFG) * a.NFG;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int fw = 8 * fg + 2 * tq + j;
                if (fw < a.FW) {
                    float* o = out + (static_cast<size_t>(fh) * a.FW + fw) * a.C;
                    o[0] = acc[0][t][2 * hh + j];
                    o[1] = acc[1][t][2 * hh + j];
                }
            }
        }
    }
}

// Plan of the tensor-core filter gradient; false if the shape is outside its limits.
inline bool mma_fgrad_plan(int N, int C, int OH, int OW, int FH, int FW, MmaFgArgs& a,
                           size_t& smem) {
    if (C % kMmaCB != 0) return false;
    a.NFG = (FW + 7) / 8;
    a.ntiles = (FH * a.NFG + 15) / 16;
    if (a.ntiles > kFgMaxTiles) return false;
    a.KC = (OW + 7 + 15) / 16;
    if (a.KC > 8) return false;  // rows up to 121 outputs
    a.RB = std::max(1, std::min(OH, 16));
    a.XR = a.RB + FH - 1;
    // pitch in 16-byte chunks congruent to NFG mod 8: consecutive (fh, fg) rows of a tile
    // start in consecutive bank groups (conflict-free ldmatrix)
    // (the rows read span 8*NFG + 16*KC - 8 columns, NFG + 2*KC - 1 chunks)
    const int p16 = a.NFG + 8 * ((2 * a.KC - 1 + 7) / 8);
    a.XC = 8 * p16;
    a.DC = 16 * a.KC + 8;
    const size_t xbytes = static_cast<size_t>(kMmaCB) * a.XR * a.XC * 2;
    const size_t dbytes = static_cast<size_t>(kMmaCB) * a.RB * a.DC * 2;
    a.dy_off = static_cast<uint32_t>((xbytes + 127) & ~size_t(127));
    smem = a.dy_off + dbytes;
    if (smem > static_cast<size_t>(device_info().max_smem_optin)) return false;
    a.bands = (OH + a.RB - 1) / a.RB;
    const int cblocks = C / kMmaCB;
    const int ctas = smem * 2 + 2048 <= 233472u ? 2 : 1;
    const long long total_bands = static_cast<long long>(N) * a.bands;
    // one wave of equal CTAs (rounding up would leave a few CTAs for a second wave)
    long long Z = static_cast<long long>(device_info().sm_count) * ctas / cblocks;
    Z = std::max<long long>(1, std::min<long long>(Z, total_bands));
    a.bands_per_slice = static_cast<int>((total_bands + Z - 1) / Z);
    a.Z = static_cast<int>((total_bands + a.bands_per_slice - 1) / a.bands_per_slice);
    if (static_cast<long long>(a.Z) * cblocks >= (1LL << 31)) return false;
    return true;
}

// Where the tensor-core filter gradient beats the CUDA-core one for 16-bit inputs (timed on
// the stage shapes: from 27 taps, and from 17 taps on rows of at least 48 outputs; below,
// the fewer MMAs per staged band do not pay for the transposed staging).
inline bool mma_fgrad_wanted(int FW, int OW) {
    return OW >= 14 && (FW >= 27 || (FW >= 17 && OW >= 48));
}

template <typename T>
cudaError_t launch_mma_fgrad(const FilterGrad& p) {
    MmaFgArgs a;
    size_t smem = 0;
    if (!mma_fgrad_wanted(p.FW, p.OW) ||
        !mma_fgrad_plan(p.N, p.C, p.OH, p.OW, p.FH, p.FW, a, smem))
        return cudaErrorNotSupported;
    const size_t count = static_cast<size_t>(p.FH) * p.FW * p.C;
    if (p.workspace == nullptr || p.workspace_floats < count * a.Z) return cudaErrorInvalidValue;
    a.x = p.x; a.dy = p.dy; a.part = p.workspace;
    a.N = p.N; a.H = p.H; a.W = p.W; a.C = p.C; a.OH = p.OH; a.OW = p.OW;
    a.FH = p.FH; a.FW = p.FW; a.pad = p.pad;
    auto kern = mma_fgrad_kernel<T>;
    static DeviceOnce smem_opt_in;
    {
        const cudaError_t err = opt_in_smem(kern, smem_opt_in, device_info().max_smem_optin);
        if (err != cudaSuccess) return err;
    }
    const unsigned grid = static_cast<unsigned>(a.Z) * static_cast<unsigned>(p.C / kMmaCB);
    const cudaError_t err = launch_pdl(kern, dim3(grid), dim3(kMmaWarps * 32), smem, p.stream, a);
    if (err != cudaSuccess) return err;
    return launch_reduce_slices(p.workspace, a.Z, count, p.dw, p.stream);
}

// Workspace floats of the tensor-core filter gradient (0 if it does not serve the shape).
inline size_t mma_fgrad_workspace_floats(int N, int C, int OH, int OW, int FH, int FW) {
    MmaFgArgs a;
    size_t smem = 0;
    if (!mma_fgrad_wanted(FW, OW) || !mma_fgrad_plan(N, C, OH, OW, FH, FW, a, smem))
        return 0;
    return static_cast<size_t>(a.Z) * FH * FW * C;
}

}  // namespace dwc
