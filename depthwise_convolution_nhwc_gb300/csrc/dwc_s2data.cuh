// dwc_s2data.cuh -- backward data ("input gradient") at stride 2 for square filters of 3, 5
// or 7 taps.
//
//   dx[n, ih, iw, c] = sum over (oh, ow, fh, fw) with ih = 2*oh + fh - pad and
//                      iw = 2*ow + fw - pad of dy[n, oh, ow, c] * w[fh, fw, c]
//
// ("Flash-DWC: Making Depthwise Convolution Compute-Efficient on GPUs", §5.1: the input
// gradient is a convolution of dy with the rotated filter; at stride 2 only the taps of the
// matching parity meet a given input pixel.)
//
// GB300 restatement.  Shifted by the padding, the input plane splits into 2x2 cells: cell
// (a, b) holds the pixels ih = 2a + r - pad, iw = 2b + q - pad (r, q in {0, 1}).  Pixel
// (r, q) of the cell receives exactly the taps fh = r + 2k, fw = q + 2j, from dy[a - k, b - j],
// so the whole cell needs only the K x K dy values dy[a - k, b - j] (K = (F + 1) / 2) and
// every tap of the filter once.  A thread owns two channels (one fp32x2 lane pair) of one
// cell row a and a strip of consecutive cells b: the F x F filter taps stay in registers,
// the dy values sit in a circular register window of K columns that advances by one column
// per cell, and each cell costs K dy loads, F*F packed FMAs and four 8-byte stores.  The
// kernel is bound by HBM (the dx writes and the dy reads); consecutive threads take
// consecutive channel pairs, so every warp load and store is contiguous.
#pragma once

#include "dwc_device.cuh"
#include "dwc_host.h"

namespace dwc {

struct S2DataArgs {
    float* dx;
    int N, H, W, C, OH, OW, pad;
    int ncp;            // channel pairs (C / 2)
    int na, a_lo;       // cell rows a_lo .. a_lo + na - 1
    int nb, b_lo;       // cell columns b_lo .. b_lo + nb - 1
    int nstrips, strip; // strips per cell row, cells per strip (a multiple of K)
};

template <typename T, int F>
__global__ void __launch_bounds__(128, F <= 5 ? 4 : 3)
s2_bwd_data_kernel(const T* __restrict__ dy, const T* __restrict__ w, const S2DataArgs a) {
    using P = Pair64;
    using V = P::V;
    constexpr int K = (F + 1) / 2;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int cp = static_cast<int>(tid % a.ncp);
    long long rest = tid / a.ncp;
    const int st = static_cast<int>(rest % a.nstrips);
    rest /= a.nstrips;
    const int ai = static_cast<int>(rest % a.na);
    const long long n = rest / a.na;
    if (n >= a.N) return;
    const int c = 2 * cp;
    const int cell_a = a.a_lo + ai;
    const int b0 = a.b_lo + st * a.strip;
    const int b1 = min(b0 + a.strip, a.b_lo + a.nb);

    V wr[F][F];
#pragma unroll
    for (int fh = 0; fh < F; ++fh)
#pragma unroll
        for (int fw = 0; fw < F; ++fw) wr[fh][fw] = P::load(w + (fh * F + fw) * a.C + c);

    // dy rows a - k; a row outside the map contributes nothing
    const T* yrow[K];
    bool yok[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int oh = cell_a - k;
        yok[k] = oh >= 0 && oh < a.OH;
        yrow[k] = dy + ((n * a.OH + (yok[k] ? oh : 0)) * a.OW) * a.C + c;
    }
    auto load_col = [&](int ow, int k) -> V {
        return (yok[k] && ow >= 0 && ow < a.OW) ? P::load(yrow[k] + static_cast<size_t>(ow) * a.C)
                                                : P::zero();
    };

    // circular window: dy column b sits in slot (b - b0) mod K
    V win[K][K];
#pragma unroll
    for (int j = 1; j < K; ++j)
#pragma unroll
        for (int k = 0; k < K; ++k) win[k][K - j] = load_col(b0 - j, k);

    const int ih0 = 2 * cell_a - a.pad;
    float* xrow0 = a.dx + ((n * a.H + ih0) * a.W) * a.C + c;
    const bool row_ok[2] = {ih0 >= 0 && ih0 < a.H, ih0 + 1 >= 0 && ih0 + 1 < a.H};

#pragma unroll 1
    for (int bb = b0; bb < b1; bb += K) {
#pragma unroll
        for (int u = 0; u < K; ++u) {
            const int b = bb + u;
            if (b >= b1) break;
#pragma unroll
            for (int k = 0; k < K; ++k) win[k][u] = load_col(b, k);
            const int iw0 = 2 * b - a.pad;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    V acc = P::zero();
#pragma unroll
                    for (int k = 0; k < K; ++k) {
                        if (r + 2 * k >= F) continue;
#pragma unroll
                        for (int j = 0; j < K; ++j) {
                            if (q + 2 * j >= F) continue;
                            P::fma(acc, win[k][(u - j + K) % K], wr[r + 2 * k][q + 2 * j]);
                        }
                    }
                    const int iw = iw0 + q;
                    if (row_ok[r] && iw >= 0 && iw < a.W)
                        store_pair_streaming(xrow0 + (static_cast<long long>(r) * a.W + iw) * a.C,
                                             P::unpack(acc));
                }
            }
        }
    }
}

template <typename T, int F>
cudaError_t launch_s2_bwd_data_inst(const GeneralConv& p) {
    S2DataArgs a;
    a.dx = p.out;
    a.N = p.N; a.H = p.H; a.W = p.W; a.C = p.C; a.OH = p.OH; a.OW = p.OW; a.pad = p.pad;
    a.ncp = p.C / 2;
    // cells that hold at least one pixel of the map
    a.a_lo = p.pad >> 1;
    a.na = ((p.H - 1 + p.pad) >> 1) - a.a_lo + 1;
    a.b_lo = p.pad >> 1;
    a.nb = ((p.W - 1 + p.pad) >> 1) - a.b_lo + 1;
    constexpr int K = (F + 1) / 2;
    // about eight cells per strip, a multiple of the window period
    a.strip = (8 + K - 1) / K * K;
    a.nstrips = (a.nb + a.strip - 1) / a.strip;
    const long long threads = static_cast<long long>(p.N) * a.na * a.nstrips * a.ncp;
    if (threads == 0) return cudaSuccess;
    const long long blocks = (threads + 127) / 128;
    if (blocks > 0x7fffffffLL) return cudaErrorNotSupported;
    s2_bwd_data_kernel<T, F><<<static_cast<unsigned>(blocks), 128, 0, p.stream>>>(
        static_cast<const T*>(p.a), static_cast<const T*>(p.b), a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_s2_bwd_data_dispatch(const GeneralConv& p) {
    if (p.FH != p.FW || p.stride != 2 || (p.C & 1)) return cudaErrorNotSupported;
    switch (p.FH) {
        case 3: return launch_s2_bwd_data_inst<T, 3>(p);
        case 5: return launch_s2_bwd_data_inst<T, 5>(p);
        case 7: return launch_s2_bwd_data_inst<T, 7>(p);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
