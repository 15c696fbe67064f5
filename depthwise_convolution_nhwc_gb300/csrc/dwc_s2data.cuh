// dwc_s2data.cuh -- backward data ("input gradient") at stride 2 for square filters of 3 to
// 13 taps.
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
// cell row a and a strip of S consecutive cells b: the F x F filter taps and the strip's
// K x (S + K - 1) dy values sit in registers (7x7: a circular window of K dy columns, see
// s2_bwd_data_stream_kernel), and each cell costs F*F packed FMAs and four 8-byte stores.  The kernel is bound by HBM (the dx writes and the dy reads); consecutive
// threads take consecutive channel pairs, so every warp load and store is contiguous.
#pragma once

#include "dwc_device.cuh"
#include "dwc_host.h"

namespace dwc {

struct S2DataArgs {
    void* dx;           // OutT elements
    int N, H, W, C, OH, OW, pad;
    int ncp;            // channel pairs (C / 2)
    int na, a_lo;       // cell rows a_lo .. a_lo + na - 1
    int nb, b_lo;       // cell columns b_lo .. b_lo + nb - 1
    int nstrips, strip; // strips per cell row, cells per strip
};

// Cells per thread strip: the strip's whole dy window (K rows x S + K - 1 columns) is loaded
// before any FMA, so that every load of the strip is in flight at once (loading one column
// per cell left the kernel waiting on L2/HBM latency: ncu showed long-scoreboard stalls of
// 12 cycles per issued instruction and DRAM half busy; 3x3 on 64x112x112x96 went from 85
// to 64 us).  Used for 3x3 and 5x5.
template <int F>
struct S2DataTile {
    static constexpr int K = (F + 1) / 2;
    static constexpr int S = 8;
};

template <typename T, int F, class OutT = float>
__global__ void __launch_bounds__(128, 4)
s2_bwd_data_kernel(const T* __restrict__ dy, const T* __restrict__ w, const S2DataArgs a) {
    using P = Pair64;
    using V = P::V;
    constexpr int K = S2DataTile<F>::K;
    constexpr int S = S2DataTile<F>::S;
    constexpr int NC = S + K - 1;   // dy columns of a strip
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
    const int b0 = a.b_lo + st * S;

    // dy[a - k, b0 - (K - 1) + m] for m < NC; a row or column outside the map reads zero
    V win[K][NC];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int oh = cell_a - k;
        const bool rok = oh >= 0 && oh < a.OH;
        const T* yrow = dy + ((n * a.OH + (rok ? oh : 0)) * a.OW) * a.C + c;
#pragma unroll
        for (int m = 0; m < NC; ++m) {
            const int ow = b0 - (K - 1) + m;
            win[k][m] = (rok && ow >= 0 && ow < a.OW) ? P::load(yrow + static_cast<size_t>(ow) * a.C)
                                                      : P::zero();
        }
    }
    V wr[F][F];
#pragma unroll
    for (int fh = 0; fh < F; ++fh)
#pragma unroll
        for (int fw = 0; fw < F; ++fw) wr[fh][fw] = P::load(w + (fh * F + fw) * a.C + c);

    const int ih0 = 2 * cell_a - a.pad;
    OutT* xrow0 = static_cast<OutT*>(a.dx) + ((n * a.H + ih0) * a.W) * a.C + c;
    const bool row_ok[2] = {ih0 >= 0 && ih0 < a.H, ih0 + 1 >= 0 && ih0 + 1 < a.H};
    // cell b0 + s: pixel (r, q) takes tap (r + 2k, q + 2j) from dy column b0 + s - j; cells
    // past the row's last one have no pixel inside the map and store nothing
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int iw0 = 2 * (b0 + s) - a.pad;
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
                        P::fma(acc, win[k][s - j + K - 1], wr[r + 2 * k][q + 2 * j]);
                    }
                }
                const int iw = iw0 + q;
                if (row_ok[r] && iw >= 0 && iw < a.W)
                    store_out_pair(xrow0 + (static_cast<long long>(r) * a.W + iw) * a.C,
                                         P::unpack(acc));
            }
        }
    }
}

// The same cells for 7x7, streamed: the dy values sit in a circular register window of K
// columns that advances by one column per cell (K loads per cell).  Holding a whole strip's
// dy values next to the 49 taps would take ~190 registers and halve the resident warps,
// which measured slower (7x7 on 64x56x56x144: 77.5 -> 85.8 us fp32, 90 -> 147 us bf16).
template <typename T, int F, class OutT = float>
__global__ void __launch_bounds__(128, 3)
s2_bwd_data_stream_kernel(const T* __restrict__ dy, const T* __restrict__ w, const S2DataArgs a) {
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
    OutT* xrow0 = static_cast<OutT*>(a.dx) + ((n * a.H + ih0) * a.W) * a.C + c;
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
                        store_out_pair(xrow0 + (static_cast<long long>(r) * a.W + iw) * a.C,
                                             P::unpack(acc));
                }
            }
        }
    }
}

// 9 to 13 taps: a cell's F x F taps no longer fit in registers, so a thread takes one pixel
// class (r, q) of its cells -- the sub-filter w[r + 2k][q + 2j], KR x KQ <= 7 x 7 taps -- in
// a circular window of KQ dy columns (KR loads per cell); the class is the launch's
// blockIdx.y.  Two accumulators split each pixel's chain of up to 49 dependent FMAs.
template <typename T, int F, int R, int Q, class OutT>
__device__ __forceinline__ void s2_data_class(const T* __restrict__ dy, const T* __restrict__ w,
                                              const S2DataArgs& a, int c, long long n, int cell_a,
                                              int b0, int b1) {
    using P = Pair64;
    using V = P::V;
    constexpr int KR = (F - R + 1) / 2, KQ = (F - Q + 1) / 2;
    V tp[KR][KQ];
#pragma unroll
    for (int k = 0; k < KR; ++k)
#pragma unroll
        for (int j = 0; j < KQ; ++j) tp[k][j] = P::load(w + ((R + 2 * k) * F + Q + 2 * j) * a.C + c);
    const T* yrow[KR];
    bool yok[KR];
#pragma unroll
    for (int k = 0; k < KR; ++k) {
        const int oh = cell_a - k;
        yok[k] = oh >= 0 && oh < a.OH;
        yrow[k] = dy + ((n * a.OH + (yok[k] ? oh : 0)) * a.OW) * a.C + c;
    }
    auto load_col = [&](int ow, int k) -> V {
        return (yok[k] && ow >= 0 && ow < a.OW) ? P::load(yrow[k] + static_cast<size_t>(ow) * a.C)
                                                : P::zero();
    };
    // circular window: dy column b sits in slot (b - b0) mod KQ
    V win[KR][KQ];
#pragma unroll
    for (int j = 1; j < KQ; ++j)
#pragma unroll
        for (int k = 0; k < KR; ++k) win[k][KQ - j] = load_col(b0 - j, k);
    const int ih = 2 * cell_a - a.pad + R;
    const bool row_ok = ih >= 0 && ih < a.H;
    OutT* xrow = static_cast<OutT*>(a.dx) + ((n * a.H + (row_ok ? ih : 0)) * a.W) * a.C + c;
#pragma unroll 1
    for (int bb = b0; bb < b1; bb += KQ) {
#pragma unroll
        for (int u = 0; u < KQ; ++u) {
            const int b = bb + u;
            if (b >= b1) break;
#pragma unroll
            for (int k = 0; k < KR; ++k) win[k][u] = load_col(b, k);
            V acc0 = P::zero(), acc1 = P::zero();
#pragma unroll
            for (int k = 0; k < KR; ++k)
#pragma unroll
                for (int j = 0; j < KQ; ++j) {
                    if (k & 1) P::fma(acc1, win[k][(u - j + KQ) % KQ], tp[k][j]);
                    else P::fma(acc0, win[k][(u - j + KQ) % KQ], tp[k][j]);
                }
            const int iw = 2 * b - a.pad + Q;
            if (row_ok && iw >= 0 && iw < a.W) {
                const float2 s0 = P::unpack(acc0), s1 = P::unpack(acc1);
                store_out_pair(xrow + static_cast<size_t>(iw) * a.C, make_float2(s0.x + s1.x, s0.y + s1.y));
            }
        }
    }
}

template <typename T, int F, class OutT = float>
__global__ void __launch_bounds__(128)
s2_bwd_data_class_kernel(const T* __restrict__ dy, const T* __restrict__ w, const S2DataArgs a) {
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int cp = static_cast<int>(tid % a.ncp);
    long long rest = tid / a.ncp;
    const int st = static_cast<int>(rest % a.nstrips);
    rest /= a.nstrips;
    const int ai = static_cast<int>(rest % a.na);
    const long long n = rest / a.na;
    if (n >= a.N) return;
    const int cell_a = a.a_lo + ai;
    const int b0 = a.b_lo + st * a.strip;
    const int b1 = min(b0 + a.strip, a.b_lo + a.nb);
    switch (blockIdx.y) {
        case 0: s2_data_class<T, F, 0, 0, OutT>(dy, w, a, 2 * cp, n, cell_a, b0, b1); break;
        case 1: s2_data_class<T, F, 0, 1, OutT>(dy, w, a, 2 * cp, n, cell_a, b0, b1); break;
        case 2: s2_data_class<T, F, 1, 0, OutT>(dy, w, a, 2 * cp, n, cell_a, b0, b1); break;
        default: s2_data_class<T, F, 1, 1, OutT>(dy, w, a, 2 * cp, n, cell_a, b0, b1); break;
    }
}

template <typename T, int F, class OutT = float>
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
    // whole-strip kernel: S cells per strip; streamed kernels (7 taps and up): about eight
    // cells, a multiple of the window period K (of the class's KQ = K or K - 1 ... close
    // enough: the strip only bounds the cells of a thread)
    constexpr int K = (F + 1) / 2;
    a.strip = F >= 7 ? (8 + K - 1) / K * K : S2DataTile<F>::S;
    a.nstrips = (a.nb + a.strip - 1) / a.strip;
    const long long threads = static_cast<long long>(p.N) * a.na * a.nstrips * a.ncp;
    if (threads == 0) return cudaSuccess;
    const long long blocks = (threads + 127) / 128;
    if (blocks > 0x7fffffffLL) return cudaErrorNotSupported;
    if constexpr (F > 7)
        s2_bwd_data_class_kernel<T, F, OutT><<<dim3(static_cast<unsigned>(blocks), 4), 128, 0, p.stream>>>(
            static_cast<const T*>(p.a), static_cast<const T*>(p.b), a);
    else if constexpr (F == 7)
        s2_bwd_data_stream_kernel<T, F, OutT><<<static_cast<unsigned>(blocks), 128, 0, p.stream>>>(
            static_cast<const T*>(p.a), static_cast<const T*>(p.b), a);
    else
        s2_bwd_data_kernel<T, F, OutT><<<static_cast<unsigned>(blocks), 128, 0, p.stream>>>(
            static_cast<const T*>(p.a), static_cast<const T*>(p.b), a);
    return cudaGetLastError();
}

template <typename T, class OutT = float>
cudaError_t launch_s2_bwd_data_dispatch(const GeneralConv& p) {
    if (p.FH != p.FW || p.stride != 2 || (p.C & 1)) return cudaErrorNotSupported;
    switch (p.FH) {
        case 3: return launch_s2_bwd_data_inst<T, 3, OutT>(p);
        case 5: return launch_s2_bwd_data_inst<T, 5, OutT>(p);
        case 7: return launch_s2_bwd_data_inst<T, 7, OutT>(p);
        case 9: return launch_s2_bwd_data_inst<T, 9, OutT>(p);
        case 11: return launch_s2_bwd_data_inst<T, 11, OutT>(p);
        case 13: return launch_s2_bwd_data_inst<T, 13, OutT>(p);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
