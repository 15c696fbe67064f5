// dwc_small.cuh -- small feature maps (W, OW, H, OH <= 16): direct kernels that run only
// the filter taps that can meet the image.
//
// On a small map most taps of a large filter land in the zero padding for every output
// (a 7x7 map under a 31x31 filter: at most 49 of 961 taps are real), and the row-streaming
// kernels, which run every tap of a row tile, spend most of their FMAs on zeros.  The pages'
// trimming of padding rows ("Flash-DWC: Making Depthwise Convolution Compute-Efficient on
// GPUs", §4.4) is taken here to its end for maps that fit in shared memory whole:
//
//  * A CTA owns a block of 32 channels (one per lane) and stages whole images of it
//    (cp.async, 16-byte chunks) through a ring of up to 8 work units, so that the copies of
//    the units ahead are in flight while one is computed (a 7x7 map's unit is a few KB: two
//    buffers left every unit waiting for its copy).
//  * Forward / backward data: on maps of at most 8 x 8 outputs each warp computes a whole
//    image (all its output rows in registers, every input row loaded once and applied to
//    each output row it meets); otherwise one output row oh of one image.  For every input row ih that
//    meets a filter row (fh = ih - oh + pad_h), the input row is held in registers as two
//    sets of column pairs, {x[2k], x[2k+1]} and {x[2k-1], x[2k]}, so that the packed FMA of
//    tap offset d = fw - pad_w updates the output pair (2k, 2k+1) with the input pair
//    starting at 2k + d.  Offsets run over [-DR, DR], the taps that can meet a
//    map of this width; the window of filter rows that meet the image, 2*DR+1 taps each,
//    is copied once per channel block (cp.async, zero fill for taps outside the filter).
//  * Filter gradient: each warp owns two window rows fh (half a window apart, so that the
//    warps' work is even) and accumulates dw[fh][d + pad_w] for d in [-DR, DR],
//    two taps per packed sum of x[ow + d] * dy[ow]; slices of images are summed afterwards
//    in a fixed order.
//
// MAXW (8 or 16) bounds the map width; DR (3, 7, 11, 15) bounds the tap offsets.
#pragma once

#include <type_traits>

#include <algorithm>

#include "dwc_device.cuh"
#include "dwc_host.h"

namespace dwc {

constexpr int kSmCh = 32;        // channels per CTA (one per lane)
constexpr int kSmMaxWarps = 16;
constexpr int kSmMaxMap = 16;    // largest H, W, OH, OW served

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
// 16-byte copy, or 16 zero bytes when `valid` is false (nothing is read then)
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int K>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory");
}
// cp_async_wait<k> for a run-time k in [0, 7]
__device__ __forceinline__ void cp_async_wait_n(int k) {
    switch (k) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        default: cp_async_wait<7>(); break;
    }
}

// Pair of adjacent columns (x[i], x[i+1]) of a register row for i in [-1, MAXW - 1], with
// zeros outside [0, MAXW): even i from `xe`, odd i from `xo` (xo[j] = (x[2j-1], x[2j])).
template <int MAXW>
__device__ __forceinline__ float2 col_pair(const float2 (&xe)[MAXW / 2], const float2 (&xo)[MAXW / 2 + 1],
                                           int i) {
    return (i & 1) == 0 ? xe[i >> 1] : xo[(i + 1) >> 1];
}

template <typename T, int MAXW>
__device__ __forceinline__ void load_row_pairs(const T* row, int lane, float2 (&xe)[MAXW / 2],
                                               float2 (&xo)[MAXW / 2 + 1]) {
    float v[MAXW];
#pragma unroll
    for (int i = 0; i < MAXW; ++i) v[i] = to_f32(row[i * kSmCh + lane]);
#pragma unroll
    for (int k = 0; k < MAXW / 2; ++k) xe[k] = make_float2(v[2 * k], v[2 * k + 1]);
    xo[0] = make_float2(0.f, v[0]);
#pragma unroll
    for (int k = 1; k < MAXW / 2; ++k) xo[k] = make_float2(v[2 * k - 1], v[2 * k]);
    xo[MAXW / 2] = make_float2(v[MAXW - 1], 0.f);
}

// Stages one image block [rows][MAXW][32] of channels c0.. (columns [0, cols) copied; the
// columns [cols, MAXW) are zeroed once at kernel start and never written by the copies).
template <typename T, int MAXW>
__device__ __forceinline__ void stage_image(T* dst, const T* src_img, int rows, int cols, int C,
                                            int c0, int tid, int nthreads) {
    constexpr int kPerChunk = 16 / static_cast<int>(sizeof(T));
    constexpr int kChunks = kSmCh / kPerChunk;  // 16-byte chunks per pixel
    const int cvalid = min(kSmCh, C - c0);      // a multiple of kPerChunk (host check)
    const int total = rows * cols * kChunks;
    for (int i = tid; i < total; i += nthreads) {
        const int q = i % kChunks;
        const int px = i / kChunks;
        const int r = px / cols, col = px - r * cols;
        if (q * kPerChunk < cvalid)
            cp_async16(dst + (r * MAXW + col) * kSmCh + q * kPerChunk,
                       src_img + (static_cast<size_t>(r) * cols + col) * C + c0 + q * kPerChunk);
    }
}

struct SmallArgs {
    const void* in;
    const void* w;
    void* out;          // OutT elements
    int N, H, W, C, OH, OW, FH, FW, pad_h, pad_w;
    int flip;           // filter rotated by 180 degrees (backward data)
    int fh_lo, nfh;     // filter rows that meet the image for some output row
    int G;              // images per work unit
    int groups;         // work units per channel block
    int ns;             // staged work units in the ring (2..8, at most groups + 1)
    uint32_t units;     // cblocks * groups, channel block slowest
    uint32_t buf_elems; // elements of one staged buffer (G images)
    uint32_t win_off;   // byte offset of the filter-window slots
    uint32_t win_elems; // elements of one filter-window slot
    int win_slots;      // 2: windows staged ahead with their block's first unit; 1: staged
                        // when the block starts (large windows)
};

template <typename T, int MAXW, int DR, class OutT = float>
__global__ void __launch_bounds__(kSmMaxWarps * 32, 1) small_rows_kernel(const SmallArgs a) {
    // a programmatic dependent of the kernel before it: nothing in global memory is touched
    // before that grid has finished
    pdl_trigger();
    pdl_wait();
    constexpr int NJ = 2 * DR + 1;
    extern __shared__ __align__(128) unsigned char smem[];
    T* xbuf = reinterpret_cast<T*>(smem);                          // [ns][G][H][MAXW][32]
    T* wins = reinterpret_cast<T*>(smem + a.win_off);              // [win_slots][nfh][NJ][32]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;
    const T* X = static_cast<const T*>(a.in);
    const T* Wt = static_cast<const T*>(a.w);
    const int img = a.H * MAXW * kSmCh;

    const uint32_t per_cta = (a.units + gridDim.x - 1) / gridDim.x;
    const uint32_t u_begin = blockIdx.x * per_cta;
    const uint32_t u_end = min(a.units, u_begin + per_cta);
    if (u_begin >= u_end) return;
    const uint32_t ns = static_cast<uint32_t>(a.ns);

    if (a.W < MAXW) {
        const int zc = MAXW - a.W;
        for (int i = tid; i < a.ns * a.G * a.H * zc * kSmCh; i += nthreads) {
            const int ch = i % kSmCh, px = i / kSmCh;
            const int col = a.W + px % zc, rr = px / zc;  // rr runs over [ns][G][H]
            xbuf[(rr * MAXW + col) * kSmCh + ch] = T(0.f);
        }
    }
    // Filter window of channel block cb into its slot: win[r][j] = filt(fh_lo + r,
    // j - DR + pad_w), zero where the tap lies outside the filter (whole 16-byte chunks of
    // channels).
    auto stage_window = [&](int cb) {
        constexpr int kPerChunk = 16 / static_cast<int>(sizeof(T));
        constexpr int kChunks = kSmCh / kPerChunk;
        const int c0 = cb * kSmCh;
        const int cvalid = min(kSmCh, a.C - c0);
        T* win = wins + (a.win_slots == 2 ? (cb & 1) : 0) * a.win_elems;
        for (int i = tid; i < a.nfh * NJ * kChunks; i += nthreads) {
            const int q = i % kChunks, rj = i / kChunks;
            const int fh = a.fh_lo + rj / NJ, fw = rj % NJ - DR + a.pad_w;
            const bool valid = fw >= 0 && fw < a.FW && q * kPerChunk < cvalid;
            const int sh = a.flip ? a.FH - 1 - fh : fh;
            const int sw = a.flip ? a.FW - 1 - fw : fw;
            const T* src = valid ? Wt + (static_cast<size_t>(sh) * a.FW + sw) * a.C + c0 + q * kPerChunk
                                 : Wt;
            cp_async16_zfill(win + rj * kSmCh + q * kPerChunk, src, valid);
        }
    };
    auto block_starts = [&](uint32_t u) { return u == u_begin || u % a.groups == 0; };
    // One copy group per unit u, in unit order: the images of u into ring slot
    // (u - u_begin) % ns and, with two window slots, where u is the CTA's first unit of a
    // channel block, the block's window into slot cb % 2 (the ring holds at most groups + 1
    // units, so a window slot is refilled only after every unit of the block that used it
    // has been computed).  With one window slot the window is copied when its block's first
    // unit comes up (every earlier unit is done then), as a group of its own.
    auto stage = [&](uint32_t u) {
        const int cb = static_cast<int>(u / a.groups);
        const int n0 = static_cast<int>(u % a.groups) * a.G;
        if (a.win_slots == 2 && block_starts(u)) stage_window(cb);
        const int slot = static_cast<int>((u - u_begin) % ns);
        for (int g = 0; g < a.G && n0 + g < a.N; ++g)
            stage_image<T, MAXW>(xbuf + slot * a.buf_elems + g * img,
                                 X + static_cast<size_t>(n0 + g) * a.H * a.W * a.C, a.H, a.W, a.C,
                                 cb * kSmCh, tid, nthreads);
        cp_async_commit();
    };

    // groups u_begin .. u_begin + ns - 2 ahead; per unit one more, so that waiting for all
    // but the newest ns - 1 groups covers unit u (empty groups past the end keep the count)
    for (uint32_t k = 0; k + 1 < ns; ++k) {
        if (u_begin + k < u_end) stage(u_begin + k);
        else cp_async_commit();
    }
    for (uint32_t u = u_begin; u < u_end; ++u) {
        const int slot = static_cast<int>((u - u_begin) % ns);
        const int cb = static_cast<int>(u / a.groups);
        const int c0 = cb * kSmCh;
        const T* win = wins + (a.win_slots == 2 ? (cb & 1) : 0) * a.win_elems;
        const bool win_now = a.win_slots == 1 && block_starts(u);
        if (win_now) {
            stage_window(cb);
            cp_async_commit();
        }
        if (u + ns - 1 < u_end) stage(u + ns - 1);
        else cp_async_commit();
        // all but the newest ns - 1 groups (over-waiting where a window group sits among
        // them is harmless); a window copied now is second newest
        cp_async_wait_n(win_now ? 1 : a.ns - 1);
        __syncthreads();

        const int n0 = static_cast<int>(u % a.groups) * a.G;
        const bool lane_ok = c0 + lane < a.C;
        // packed FMAs of input row xe/xo into the output-row accumulators acc through window
        // row wrow (tap offsets -DR..DR)
        auto row_taps = [&](float2 (&acc)[MAXW / 2], const float2 (&xe)[MAXW / 2],
                            const float2 (&xo)[MAXW / 2 + 1], const T* wr) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const float wv = to_f32(wr[j * kSmCh]);
                const float2 w2 = make_float2(wv, wv);
#pragma unroll
                for (int k = 0; k < MAXW / 2; ++k) {
                    const int i = 2 * k + j - DR;  // first input column of the pair
                    if (i < -1 || i > MAXW - 1) continue;
                    fma2(acc[k], col_pair<MAXW>(xe, xo, i), w2);
                }
            }
        };
        auto store_row = [&](const float2 (&acc)[MAXW / 2], int n, int oh) {
            if (!lane_ok) return;
            OutT* o = static_cast<OutT*>(a.out) + (static_cast<size_t>(n) * a.OH + oh) * a.OW * a.C + c0 + lane;
#pragma unroll
            for (int k = 0; k < MAXW / 2; ++k) {
                if constexpr (std::is_same<OutT, float>::value) {
                    if (2 * k < a.OW) __stcs(o + static_cast<size_t>(2 * k) * a.C, acc[k].x);
                    if (2 * k + 1 < a.OW) __stcs(o + static_cast<size_t>(2 * k + 1) * a.C, acc[k].y);
                } else {
                    if (2 * k < a.OW) store_out(o + static_cast<size_t>(2 * k) * a.C, acc[k].x);
                    if (2 * k + 1 < a.OW) store_out(o + static_cast<size_t>(2 * k + 1) * a.C, acc[k].y);
                }
            }
        };
        auto per_row = [&]() {
            for (int q = warp; q < a.G * a.OH; q += nwarps) {
                const int g = q / a.OH, oh = q - g * a.OH;
                const int n = n0 + g;
                if (n >= a.N) break;
                const T* xg = xbuf + slot * a.buf_elems + g * img;
                float2 acc[MAXW / 2];
#pragma unroll
                for (int k = 0; k < MAXW / 2; ++k) acc[k] = make_float2(0.f, 0.f);
                const int ih_lo = max(0, oh - a.pad_h), ih_hi = min(a.H, oh - a.pad_h + a.FH);
                for (int ih = ih_lo; ih < ih_hi; ++ih) {
                    float2 xe[MAXW / 2], xo[MAXW / 2 + 1];
                    load_row_pairs<T, MAXW>(xg + ih * MAXW * kSmCh, lane, xe, xo);
                    row_taps(acc, xe, xo, win + (ih - oh + a.pad_h - a.fh_lo) * NJ * kSmCh + lane);
                }
                store_row(acc, n, oh);
            }
        };
        if constexpr (MAXW == 8) {
          if (a.OH > MAXW) {
            per_row();
          } else {
            // a warp per image: the output rows' accumulators stay in registers while each
            // input row is loaded once (OH <= 8)
            for (int g = warp; g < a.G; g += nwarps) {
                const int n = n0 + g;
                if (n >= a.N) break;
                const T* xg = xbuf + slot * a.buf_elems + g * img;
                float2 acc[MAXW][MAXW / 2];
#pragma unroll
                for (int r = 0; r < MAXW; ++r) {
#pragma unroll
                    for (int k = 0; k < MAXW / 2; ++k) acc[r][k] = make_float2(0.f, 0.f);
                }
                for (int ih = 0; ih < a.H; ++ih) {
                    float2 xe[MAXW / 2], xo[MAXW / 2 + 1];
                    load_row_pairs<T, MAXW>(xg + ih * MAXW * kSmCh, lane, xe, xo);
#pragma unroll
                    for (int oh = 0; oh < MAXW; ++oh) {
                        const int wrow = ih - oh + a.pad_h - a.fh_lo;   // window row (fh - fh_lo)
                        if (oh >= a.OH || wrow < 0 || wrow >= a.nfh) continue;
                        row_taps(acc[oh], xe, xo, win + wrow * NJ * kSmCh + lane);
                    }
                }
#pragma unroll
                for (int oh = 0; oh < MAXW; ++oh)
                    if (oh < a.OH) store_row(acc[oh], n, oh);
            }
          }
        } else {
            per_row();
        }
        __syncthreads();  // the slot is re-staged, and the other window slot may be refilled
    }
    cp_async_wait<0>();
}

struct SmallFgArgs {
    const void* x;
    const void* dy;
    float* part;        // [Z][nfh][FW][C]
    int N, H, W, C, OH, OW, FH, FW, pad_h, pad_w;
    int fh_lo, nfh;
    int cblocks;
    int G, ipc;                   // images per staged group, images per slice
    uint32_t xb_elems, db_elems;  // elements of one staged x / dy buffer (G images)
    uint32_t d_off;               // byte offset of the dy buffers
};

// Filter gradient of one window row held by a warp: two taps per packed accumulator,
// acc[p] = (tap d, tap d + 1) with d = 2p - DR, so DR + 1 pairs cover [-DR, DR] (the second
// tap of the last pair, DR + 1, is dropped).  For output column ow the pair starting at input
// column ow + d multiplies (dy[ow], dy[ow]).
template <int MAXW, int DR>
__device__ __forceinline__ void fgrad_row(float2 (&acc)[DR + 1], const float2 (&xe)[MAXW / 2],
                                          const float2 (&xo)[MAXW / 2 + 1], const float (&dv)[MAXW]) {
#pragma unroll
    for (int ow = 0; ow < MAXW; ++ow) {
        const float2 g2 = make_float2(dv[ow], dv[ow]);
#pragma unroll
        for (int p = 0; p <= DR; ++p) {
            const int i = ow + 2 * p - DR;
            if (i < -1 || i > MAXW - 1) continue;
            fma2(acc[p], col_pair<MAXW>(xe, xo, i), g2);
        }
    }
}

template <typename T, int MAXW, int DR>
__global__ void __launch_bounds__(kSmMaxWarps * 32, 1) small_fgrad_kernel(const SmallFgArgs a) {
    pdl_trigger();   // the slice sum may be scheduled now (it waits for this grid)
    pdl_wait();      // (a programmatic dependent itself: the grid before it has finished)
    constexpr int NP = DR + 1;
    extern __shared__ __align__(128) unsigned char smem[];
    T* xbuf = reinterpret_cast<T*>(smem);                       // [2][G][H][MAXW][32]
    T* dbuf = reinterpret_cast<T*>(smem + a.d_off);             // [2][G][OH][MAXW][32]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x;
    const T* X = static_cast<const T*>(a.x);
    const T* DY = static_cast<const T*>(a.dy);
    const int ximg = a.H * MAXW * kSmCh, dimg = a.OH * MAXW * kSmCh;

    const int cb = blockIdx.x % a.cblocks;
    const int z = blockIdx.x / a.cblocks;
    const int c0 = cb * kSmCh;
    // Warp w owns window rows w and w + ceil(nfh / 2).  The number of output rows a window
    // row meets rises and then falls symmetrically across the window, so a row of the
    // rising half paired with the row half a window later (falling half) gives every warp
    // about the same work.
    const int half = (a.nfh + 1) / 2;
    const int ra = warp, rb = warp + half;
    const bool has_b = rb < a.nfh;
    const int fa = a.fh_lo + ra, fb = a.fh_lo + rb;
    const int nb = z * a.ipc, ne = min(a.N, nb + a.ipc);

    if (a.W < MAXW) {
        const int zc = MAXW - a.W;
        for (int i = tid; i < 2 * a.G * a.H * zc * kSmCh; i += nthreads) {
            const int ch = i % kSmCh, px = i / kSmCh;
            xbuf[((px / zc) * MAXW + a.W + px % zc) * kSmCh + ch] = T(0.f);
        }
    }
    if (a.OW < MAXW) {
        const int zc = MAXW - a.OW;
        for (int i = tid; i < 2 * a.G * a.OH * zc * kSmCh; i += nthreads) {
            const int ch = i % kSmCh, px = i / kSmCh;
            dbuf[((px / zc) * MAXW + a.OW + px % zc) * kSmCh + ch] = T(0.f);
        }
    }
    auto stage = [&](int n0, int buf) {
        for (int g = 0; g < a.G && n0 + g < ne; ++g) {
            stage_image<T, MAXW>(xbuf + buf * a.xb_elems + g * ximg,
                                 X + static_cast<size_t>(n0 + g) * a.H * a.W * a.C, a.H, a.W, a.C,
                                 c0, tid, nthreads);
            stage_image<T, MAXW>(dbuf + buf * a.db_elems + g * dimg,
                                 DY + static_cast<size_t>(n0 + g) * a.OH * a.OW * a.C, a.OH, a.OW,
                                 a.C, c0, tid, nthreads);
        }
        cp_async_commit();
    };

    float2 acc_a[NP], acc_b[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) acc_a[p] = acc_b[p] = make_float2(0.f, 0.f);

    if (nb < ne) stage(nb, 0);
    for (int n0 = nb, it = 0; n0 < ne; n0 += a.G, ++it) {
        const int buf = it & 1;
        if (n0 + a.G < ne) stage(n0 + a.G, buf ^ 1);
        else cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        for (int g = 0; g < a.G && n0 + g < ne; ++g) {
            const T* xg = xbuf + buf * a.xb_elems + g * ximg;
            const T* dg = dbuf + buf * a.db_elems + g * dimg;
            for (int oh = 0; oh < a.OH; ++oh) {
                // input rows of this output row under the warp's two filter rows
                const int iha = oh + fa - a.pad_h, ihb = oh + fb - a.pad_h;
                const bool va = iha >= 0 && iha < a.H;
                const bool vb = has_b && ihb >= 0 && ihb < a.H;
                if (!va && !vb) continue;
                float dv[MAXW];
#pragma unroll
                for (int i = 0; i < MAXW; ++i) dv[i] = to_f32(dg[(oh * MAXW + i) * kSmCh + lane]);
                if (va) {
                    float2 xe[MAXW / 2], xo[MAXW / 2 + 1];
                    load_row_pairs<T, MAXW>(xg + iha * MAXW * kSmCh, lane, xe, xo);
                    fgrad_row<MAXW, DR>(acc_a, xe, xo, dv);
                }
                if (vb) {
                    float2 xe[MAXW / 2], xo[MAXW / 2 + 1];
                    load_row_pairs<T, MAXW>(xg + ihb * MAXW * kSmCh, lane, xe, xo);
                    fgrad_row<MAXW, DR>(acc_b, xe, xo, dv);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    if (c0 + lane < a.C) {
        auto write_row = [&](int r, const float2 (&acc)[NP]) {
            float* dst = a.part + ((static_cast<size_t>(z) * a.nfh + r) * a.FW) * a.C + c0 + lane;
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                const int fw = 2 * p - DR + a.pad_w;
                if (fw >= 0 && fw < a.FW) dst[static_cast<size_t>(fw) * a.C] = acc[p].x;
                if (2 * p + 1 <= 2 * DR && fw + 1 >= 0 && fw + 1 < a.FW)
                    dst[static_cast<size_t>(fw + 1) * a.C] = acc[p].y;
            }
            // taps whose offset lies beyond DR never meet the map
            for (int fw = 0; fw < a.FW; ++fw)
                if (fw - a.pad_w < -DR || fw - a.pad_w > DR) dst[static_cast<size_t>(fw) * a.C] = 0.f;
        };
        if (ra < a.nfh) write_row(ra, acc_a);
        if (has_b) write_row(rb, acc_b);
    }
}

// ------------------------------------------------------------------------------ host side

// Map-size class and tap-offset bound; false if the small kernels do not serve the map.
inline bool small_shape(int H, int W, int OH, int OW, int FW, int pad_w, int& maxw, int& dr) {
    if (H > kSmMaxMap || W > kSmMaxMap || OH > kSmMaxMap || OW > kSmMaxMap) return false;
    maxw = (W <= 8 && OW <= 8) ? 8 : 16;
    // offsets d = fw - pad_w that pair an output column with an input column
    const int dlo = std::max(-pad_w, -(OW - 1));
    const int dhi = std::min(FW - 1 - pad_w, W - 1);
    const int need = std::max(std::max(-dlo, dhi), 0);
    dr = need <= 3 ? 3 : (need <= 7 ? 7 : (need <= 11 ? 11 : 15));
    return dr <= maxw - 1;
}

// Resident CTAs per SM of a small-map launch.
inline int small_ctas_per_sm(size_t smem, int nwarps, int regs) {
    return resident_ctas(smem, nwarps * 32, regs);
}

// Where the small-map kernels beat the row-streaming / filter-gradient kernels (timed on the
// 14x14 and 7x7 stage shapes): larger filters, whose taps mostly miss such maps, and every
// filter from 5 taps on maps of at most 8 columns.
inline bool small_rows_wanted(int W, int OW, int FW) {
    return FW >= 13 || (std::max(W, OW) <= 8 && FW >= 5);
}
inline bool small_fgrad_wanted(int W, int OW, int FW) {
    return FW >= 9 || (std::max(W, OW) <= 8 && FW >= 5);
}

// Filter rows fh = ih - oh + pad that meet the image for some output row.
inline void small_window_rows(int H, int OH, int FH, int pad_h, int& fh_lo, int& nfh) {
    fh_lo = std::max(0, pad_h - (OH - 1));
    const int fh_hi = std::min(FH - 1, H - 1 + pad_h);
    nfh = std::max(0, fh_hi - fh_lo + 1);
}

template <typename T, int MAXW, int DR, class OutT = float>
cudaError_t launch_small_rows_inst(const RowConv& p) {
    constexpr int NJ = 2 * DR + 1;
    SmallArgs a;
    a.in = p.in; a.w = p.w; a.out = p.out;
    a.N = p.N; a.H = p.H; a.W = p.W; a.C = p.C; a.OH = p.OH; a.OW = p.OW;
    a.FH = p.FH; a.FW = p.FW; a.pad_h = p.pad_h; a.pad_w = p.pad_w; a.flip = p.flip ? 1 : 0;
    small_window_rows(p.H, p.OH, p.FH, p.pad_h, a.fh_lo, a.nfh);
    const size_t img_bytes = static_cast<size_t>(p.H) * MAXW * kSmCh * sizeof(T);
    const size_t win_bytes = static_cast<size_t>(std::max(a.nfh, 1)) * NJ * kSmCh * sizeof(T);
    const size_t cap = static_cast<size_t>(device_info().max_smem_optin);
    // images per unit: maps of at most 8 x 8 outputs, one per warp (8); others, enough output rows
    // for the warps; within shared memory
    const bool per_image = MAXW == 8 && p.OH <= MAXW;   // the kernel's warp-per-image path
    int G = per_image ? std::min(8, std::max(p.N, 1))
                      : std::max(1, std::min(4, (kSmMaxWarps + p.OH - 1) / std::max(p.OH, 1)));
    while (G > 1 && 2 * G * img_bytes + win_bytes + 128 > cap) --G;
    if (2 * G * img_bytes + win_bytes + 128 > cap) return cudaErrorNotSupported;
    a.G = G;
    a.buf_elems = static_cast<uint32_t>(G * p.H * MAXW * kSmCh);
    const int cblocks = (p.C + kSmCh - 1) / kSmCh;
    a.groups = (p.N + G - 1) / G;
    const long long units = static_cast<long long>(cblocks) * a.groups;
    if (units == 0) return cudaSuccess;
    if (units >= (1LL << 31)) return cudaErrorNotSupported;
    a.units = static_cast<uint32_t>(units);
    // ring depth: the CTA's units up to 8, at most groups + 1 (a filter-window slot is
    // refilled only after its block's units are done), within shared memory
    const long long grid0 = std::min<long long>(units, static_cast<long long>(device_info().sm_count));
    const long long per_cta = (units + grid0 - 1) / grid0;
    int ns = static_cast<int>(std::min<long long>({8LL, std::max(2LL, per_cta), a.groups + 1LL}));
    a.win_slots = 2 * G * img_bytes + 2 * win_bytes + 128 <= cap ? 2 : 1;
    while (ns > 2 && ns * G * img_bytes + a.win_slots * win_bytes + 128 > cap) --ns;
    a.ns = ns;
    a.win_elems = static_cast<uint32_t>(std::max(a.nfh, 1) * NJ * kSmCh);
    a.win_off = static_cast<uint32_t>((ns * G * img_bytes + 127) & ~size_t(127));
    const size_t smem = a.win_off + a.win_slots * win_bytes;
    // warps: the unit's images (maps up to 8 wide) or output rows, spread evenly
    const int pairs = per_image ? G : G * p.OH;
    const int rounds = (pairs + kSmMaxWarps - 1) / kSmMaxWarps;
    const int nwarps = (pairs + rounds - 1) / rounds;
    auto kern = small_rows_kernel<T, MAXW, DR, OutT>;
    // one CTA per SM: a CTA stages the filter window of each channel block it meets, so
    // fewer CTAs with more units each was faster on the stage shapes than two per SM
    const int per_sm = 1;
    const long long grid = std::min<long long>(units, static_cast<long long>(device_info().sm_count) * per_sm);
    static DeviceOnce smem_opt_in;
    {
        const cudaError_t err = opt_in_smem(kern, smem_opt_in, device_info().max_smem_optin);
        if (err != cudaSuccess) return err;
    }
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(nwarps * 32), smem, p.stream, a);
}

// Launch plan of the small-map filter gradient (shared by the workspace query and launch).
template <typename T, int MAXW, int DR>
bool small_fgrad_plan(int N, int H, int W, int C, int OH, int OW, int FH, int pad_h,
                      SmallFgArgs& a, size_t& smem, int& nwarps) {
    small_window_rows(H, OH, FH, pad_h, a.fh_lo, a.nfh);
    if (a.nfh <= 0 || N <= 0) return false;
    nwarps = (a.nfh + 1) / 2;  // two window rows per warp
    if (nwarps > kSmMaxWarps) return false;
    a.cblocks = (C + kSmCh - 1) / kSmCh;
    const size_t ximg = static_cast<size_t>(H) * MAXW * kSmCh * sizeof(T);
    const size_t dimg = static_cast<size_t>(OH) * MAXW * kSmCh * sizeof(T);
    const size_t cap = static_cast<size_t>(device_info().max_smem_optin);
    int G = 8;
    while (G > 1 && 2 * G * (ximg + dimg) > 114688) G >>= 1;  // two CTAs per SM where possible
    if (2 * G * (ximg + dimg) > cap) return false;
    a.G = G;
    a.xb_elems = static_cast<uint32_t>(G * H * MAXW * kSmCh);
    a.db_elems = static_cast<uint32_t>(G * OH * MAXW * kSmCh);
    a.d_off = static_cast<uint32_t>((2 * G * ximg + 127) & ~size_t(127));
    smem = a.d_off + 2 * G * dimg;
    static const int regs = kernel_regs(small_fgrad_kernel<T, MAXW, DR>, 128);
    const int per_sm = std::min(2, small_ctas_per_sm(smem, nwarps, regs));
    long long Z = static_cast<long long>(device_info().sm_count) * per_sm / a.cblocks;
    Z = std::max<long long>(1, std::min<long long>(Z, N));
    a.ipc = static_cast<int>((N + Z - 1) / Z);
    if (a.ipc > G) a.ipc = (a.ipc + G - 1) / G * G;  // whole groups per slice
    Z = (N + a.ipc - 1) / a.ipc;
    if (Z * a.cblocks >= (1LL << 31)) return false;
    a.part = nullptr;
    return true;
}

template <typename T, int MAXW, int DR>
cudaError_t launch_small_fgrad_inst(const FilterGrad& p) {
    SmallFgArgs a;
    size_t smem = 0;
    int nwarps = 0;
    if (!small_fgrad_plan<T, MAXW, DR>(p.N, p.H, p.W, p.C, p.OH, p.OW, p.FH, p.pad, a, smem, nwarps))
        return cudaErrorNotSupported;
    const int Z = (p.N + a.ipc - 1) / a.ipc;
    const size_t count = static_cast<size_t>(a.nfh) * p.FW * p.C;
    if (p.workspace == nullptr || p.workspace_floats < count * Z) return cudaErrorInvalidValue;
    a.x = p.x; a.dy = p.dy; a.part = p.workspace;
    a.N = p.N; a.H = p.H; a.W = p.W; a.C = p.C; a.OH = p.OH; a.OW = p.OW;
    a.FH = p.FH; a.FW = p.FW; a.pad_h = p.pad; a.pad_w = p.pad;
    auto kern = small_fgrad_kernel<T, MAXW, DR>;
    static DeviceOnce smem_opt_in;
    {
        const cudaError_t err = opt_in_smem(kern, smem_opt_in, device_info().max_smem_optin);
        if (err != cudaSuccess) return err;
    }
    const unsigned grid = static_cast<unsigned>(Z) * a.cblocks;
    cudaError_t err = launch_pdl(kern, dim3(grid), dim3(nwarps * 32), smem, p.stream, a);
    if (err != cudaSuccess) return err;
    // rows of dw outside the window never meet the image
    const size_t row = static_cast<size_t>(p.FW) * p.C;
    if (a.fh_lo > 0) {
        err = cudaMemsetAsync(p.dw, 0, a.fh_lo * row * sizeof(float), p.stream);
        if (err != cudaSuccess) return err;
    }
    const int tail = p.FH - a.fh_lo - a.nfh;
    if (tail > 0) {
        err = cudaMemsetAsync(p.dw + (a.fh_lo + a.nfh) * row, 0, tail * row * sizeof(float), p.stream);
        if (err != cudaSuccess) return err;
    }
    return launch_reduce_slices(p.workspace, Z, count, p.dw + a.fh_lo * row, p.stream);
}


// ------------------------------------------------------------------ 7 x 7 maps, 3 to 7 taps
// The last stage of the networks the pages evaluate ("Flash-DWC", §6.3: 7 x 7 maps, "same"
// padding) has little independent work: one 49-pixel plane per (image, channel).  A warp per
// image and lane per channel (the kernels above) leaves 8 warps on an SM and spends most of its
// instructions assembling column pairs.  Here a thread owns a channel PAIR of one image
// (consecutive lanes, consecutive pairs: 8-byte loads and stores coalesce across the warp),
// every packed FMA takes both channels at once (no pair assembly), and every loop is
// unrolled for the fixed map and filter, so only the taps that meet the image are issued:
// 37 x 37 of the 49 x 49 products per pixel plane at 7 taps.
//  * forward / backward data: the thread's 49 input pairs sit in registers (loaded at once:
//    one memory latency), the filter rows come from L1; the two warps of a CTA take the even
//    and the odd output rows of the same 32 channel pairs of an image;
//  * filter gradient: the two warps of a CTA take the even and the odd filter rows; each
//    thread accumulates its dw rows in registers over a range of images (the input image in
//    registers, one output-gradient row at a time) and writes them to a slice of the
//    workspace; the slices are summed afterwards in a fixed order.
constexpr int kTinyMap = 7;
constexpr int kTinyPairs = 32;   // channel pairs per CTA (one per lane)

inline bool tiny_shape(int H, int W, int OH, int OW, int FH, int FW, int pad_h, int pad_w) {
    return H == kTinyMap && W == kTinyMap && OH == kTinyMap && OW == kTinyMap && FH == FW &&
           (FH == 3 || FH == 5 || FH == 7) && pad_h == (FH - 1) / 2 && pad_w == (FW - 1) / 2;
}

struct TinyArgs {
    const void* in;     // N x 7 x 7 x C
    const void* w;      // F x F x C
    void* out;          // N x 7 x 7 x C, OutT
    int N, C, flip;
    int cblocks;        // blocks of 32 channel pairs
};

// Output rows oh = PART, PART + 2, ... of one image and channel pair.
template <typename T, int F, class OutT, int PART>
__device__ __forceinline__ void tiny_rows_part(const T* __restrict__ X, const T* __restrict__ Wt,
                                               OutT* __restrict__ O, int C, bool flip) {
    constexpr int M = kTinyMap, P = (F - 1) / 2;
    float2 x[M][M];
#pragma unroll
    for (int i = 0; i < M; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) x[i][j] = Elem<T>::load_pair(X + static_cast<size_t>(i * M + j) * C);
#pragma unroll
    for (int oh = PART; oh < M; oh += 2) {
        float2 acc[M];
#pragma unroll
        for (int ow = 0; ow < M; ++ow) acc[ow] = make_float2(0.f, 0.f);
#pragma unroll
        for (int fh = 0; fh < F; ++fh) {
            const int ih = oh + fh - P;
            if (ih < 0 || ih >= M) continue;
            const int sh = flip ? F - 1 - fh : fh;   // backward data: the filter rotated by 180
            float2 wr[F];
#pragma unroll
            for (int fw = 0; fw < F; ++fw)
                wr[fw] = Elem<T>::load_pair(Wt + static_cast<size_t>(sh * F + (flip ? F - 1 - fw : fw)) * C);
#pragma unroll
            for (int fw = 0; fw < F; ++fw)
#pragma unroll
                for (int ow = 0; ow < M; ++ow) {
                    const int iw = ow + fw - P;
                    if (iw < 0 || iw >= M) continue;
                    fma2(acc[ow], x[ih][iw], wr[fw]);
                }
        }
#pragma unroll
        for (int ow = 0; ow < M; ++ow) store_out_pair(O + static_cast<size_t>(oh * M + ow) * C, acc[ow]);
    }
}

// Grid: cblocks x N CTAs of 2 warps (even / odd output rows).
template <typename T, int F, class OutT>
__global__ void __launch_bounds__(64) tiny_rows_kernel(const TinyArgs a) {
    // a programmatic dependent of the kernel before it: nothing in global memory is touched
    // before that grid has finished
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, part = threadIdx.x >> 5;
    const int cb = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.cblocks));
    const int n = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.cblocks));
    const int c = 2 * (cb * kTinyPairs + lane);
    if (n >= a.N || c >= a.C) return;
    const size_t img = static_cast<size_t>(n) * kTinyMap * kTinyMap * a.C + c;
    const T* X = static_cast<const T*>(a.in) + img;
    const T* Wt = static_cast<const T*>(a.w) + c;
    OutT* O = static_cast<OutT*>(a.out) + img;
    if (part == 0) tiny_rows_part<T, F, OutT, 0>(X, Wt, O, a.C, a.flip != 0);
    else tiny_rows_part<T, F, OutT, 1>(X, Wt, O, a.C, a.flip != 0);
}

template <typename T, class OutT>
cudaError_t launch_tiny_rows(const RowConv& p) {
    TinyArgs a;
    a.in = p.in; a.w = p.w; a.out = p.out;
    a.N = p.N; a.C = p.C; a.flip = p.flip ? 1 : 0;
    a.cblocks = (p.C / 2 + kTinyPairs - 1) / kTinyPairs;
    const long long grid = static_cast<long long>(a.cblocks) * p.N;
    if (grid == 0) return cudaSuccess;
    if (grid >= (1LL << 31) || p.C % 2 != 0) return cudaErrorNotSupported;
    const unsigned g = static_cast<unsigned>(grid);
    switch (p.FH) {
        case 3: return launch_pdl(tiny_rows_kernel<T, 3, OutT>, dim3(g), dim3(64), 0, p.stream, a);
        case 5: return launch_pdl(tiny_rows_kernel<T, 5, OutT>, dim3(g), dim3(64), 0, p.stream, a);
        case 7: return launch_pdl(tiny_rows_kernel<T, 7, OutT>, dim3(g), dim3(64), 0, p.stream, a);
        default: return cudaErrorNotSupported;
    }
}

struct TinyFgArgs {
    const void* x;      // N x 7 x 7 x C
    const void* dy;     // N x 7 x 7 x C
    float* ws;          // Z slices of F x F x C
    int N, C;
    int ipb;            // images per CTA (slice)
    int cblocks;
};

// Filter rows fh = PART, PART + 2, ... of one channel pair, summed over images [n0, n1).
template <typename T, int F, int PART>
__device__ __forceinline__ void tiny_fgrad_part(const T* __restrict__ X, const T* __restrict__ D,
                                                float* __restrict__ out, int C, int n0, int n1) {
    constexpr int M = kTinyMap, P = (F - 1) / 2, NR = (F - PART + 1) / 2;
    float2 acc[NR][F];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int fw = 0; fw < F; ++fw) acc[r][fw] = make_float2(0.f, 0.f);
    const size_t img = static_cast<size_t>(M) * M * C;
    for (int n = n0; n < n1; ++n) {
        const T* Xn = X + static_cast<size_t>(n) * img;
        const T* Dn = D + static_cast<size_t>(n) * img;
        float2 x[M][M];
#pragma unroll
        for (int i = 0; i < M; ++i)
#pragma unroll
            for (int j = 0; j < M; ++j) x[i][j] = Elem<T>::load_pair(Xn + static_cast<size_t>(i * M + j) * C);
#pragma unroll
        for (int oh = 0; oh < M; ++oh) {
            float2 d[M];
#pragma unroll
            for (int ow = 0; ow < M; ++ow) d[ow] = Elem<T>::load_pair(Dn + static_cast<size_t>(oh * M + ow) * C);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const int ih = oh + PART + 2 * r - P;
                if (ih < 0 || ih >= M) continue;
#pragma unroll
                for (int fw = 0; fw < F; ++fw)
#pragma unroll
                    for (int ow = 0; ow < M; ++ow) {
                        const int iw = ow + fw - P;
                        if (iw < 0 || iw >= M) continue;
                        fma2(acc[r][fw], x[ih][iw], d[ow]);
                    }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int fw = 0; fw < F; ++fw)
            *reinterpret_cast<float2*>(out + static_cast<size_t>((PART + 2 * r) * F + fw) * C) = acc[r][fw];
}

// Grid: cblocks x Z CTAs of 2 warps (even / odd filter rows); slice z covers images
// [z * ipb, (z + 1) * ipb).
template <typename T, int F>
__global__ void __launch_bounds__(64) tiny_fgrad_kernel(const TinyFgArgs a) {
    pdl_trigger();   // the slice sum may be scheduled now (it waits for this grid)
    pdl_wait();      // (a programmatic dependent itself: the grid before it has finished)
    const int lane = threadIdx.x & 31, part = threadIdx.x >> 5;
    const int cb = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.cblocks));
    const int z = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.cblocks));
    const int c = 2 * (cb * kTinyPairs + lane);
    if (c >= a.C) return;
    const int n0 = z * a.ipb, n1 = min(a.N, n0 + a.ipb);
    const T* X = static_cast<const T*>(a.x) + c;
    const T* D = static_cast<const T*>(a.dy) + c;
    float* out = a.ws + static_cast<size_t>(z) * F * F * a.C + c;
    if (part == 0) tiny_fgrad_part<T, F, 0>(X, D, out, a.C, n0, n1);
    else tiny_fgrad_part<T, F, 1>(X, D, out, a.C, n0, n1);
}

// Images per slice: CTAs for about 8 (up to 5 taps) or 4 (7 taps) per SM.  fp32 64x7x7x1024
// at 5 taps: one image per CTA (64 slices) 16.9 -> 14.9 us; at 7 taps (254 registers, 4 CTAs
// per SM) two images per CTA stay faster (17.2 against 18.7 us), and fewer slices were slower
// for both (3 images 18.7 / 18.8 us, 4 images 22.1 / 19.9 us).
inline int tiny_fgrad_ipb(int N, int C, int F) {
    const long long cblocks = (C / 2 + kTinyPairs - 1) / kTinyPairs;
    const long long want = (F <= 5 ? 8LL : 4LL) * device_info().sm_count;
    const long long z = std::max(1LL, std::min<long long>(N, want / std::max(1LL, cblocks)));
    return static_cast<int>((N + z - 1) / z);
}

inline size_t tiny_fgrad_workspace_floats(int N, int C, int F) {
    if (N <= 0) return 0;
    const int ipb = tiny_fgrad_ipb(N, C, F);
    return static_cast<size_t>((N + ipb - 1) / ipb) * F * F * C;
}

template <typename T, int F>
cudaError_t launch_tiny_fgrad_cluster(const FilterGrad& p);

template <typename T>
cudaError_t launch_tiny_fgrad(const FilterGrad& p) {
    if (p.FH == 3) {
        const cudaError_t err = launch_tiny_fgrad_cluster<T, 3>(p);
        if (err != cudaErrorNotSupported) return err;
    }
    TinyFgArgs a;
    a.x = p.x; a.dy = p.dy;
    a.N = p.N; a.C = p.C;
    a.ipb = tiny_fgrad_ipb(p.N, p.C, p.FH);
    a.cblocks = (p.C / 2 + kTinyPairs - 1) / kTinyPairs;
    const int Z = (p.N + a.ipb - 1) / a.ipb;
    const size_t count = static_cast<size_t>(p.FH) * p.FW * p.C;
    if (p.workspace == nullptr || p.workspace_floats < static_cast<size_t>(Z) * count) return cudaErrorInvalidValue;
    a.ws = p.workspace;
    const long long grid = static_cast<long long>(a.cblocks) * Z;
    if (grid >= (1LL << 31) || p.C % 2 != 0) return cudaErrorNotSupported;
    const unsigned g = static_cast<unsigned>(grid);
    cudaError_t err = cudaErrorNotSupported;
    switch (p.FH) {
        case 3: err = launch_pdl(tiny_fgrad_kernel<T, 3>, dim3(g), dim3(64), 0, p.stream, a); break;
        case 5: err = launch_pdl(tiny_fgrad_kernel<T, 5>, dim3(g), dim3(64), 0, p.stream, a); break;
        case 7: err = launch_pdl(tiny_fgrad_kernel<T, 7>, dim3(g), dim3(64), 0, p.stream, a); break;
        default: break;
    }
    if (err != cudaSuccess) return err;
    return launch_reduce_slices(p.workspace, Z, count, p.dw, p.stream);
}


// ---- 7x7 maps, filter gradient in one launch (thread-block clusters) -----------------
//
// The two-launch form above reads its images straight from global memory into registers
// (one thread per channel pair holds a whole image) and sums its slices in a second kernel.
// Here a CTA owns one 64-channel block and a range of images, and a producer warp stages
// those images (x and dy, 49 pixels x 64 channels each) into a ring of shared-memory slots
// with tensor copies.  The work of one image is its NP (filter row fh, output row oh) pairs
// that meet the map (37 at 7 taps: filter row fh meets 7 - |fh - P| output rows); compute
// warp w takes pairs 3w .. 3w + 2 of every image, loads the pair's dy row and the x row fh
// away (7 channel pairs each) from shared memory and adds their products into its own
// F accumulators per pair, so the warps carry equal work.  After the last image the pair
// partials go to shared memory, the CTA sums each filter row's pairs in list order, and the
// Z CTAs of a channel block, one cluster along the image axis, sum their CTA partials in
// rank order by reading each other's shared memory.  The result is bit-reproducible and
// needs no workspace or second launch.  It serves 3 taps: fp32 64x7x7x1024 20.4 -> 14.6 us
// (bf16 16.7 -> 14.7 us, CUDA events).  At 5 and 7 taps it measured 19.1 / 24.6 us against
// 19.0 / 19.4 us for the two-launch form: a CTA works through its 8 images one ring slot at
// a time (ncu: 33 % issue, fixed-latency and barrier stalls), and the cluster scheduler
// places two CTAs on some SMs while others get none (busiest SM 37 k cycles against 22 k on
// average), so the form is kept for 3 taps only.
constexpr int kTfcMaxZ = 8;     // CTAs per cluster (images split Z ways)
constexpr int kTfcBarBytes = 256;
constexpr int kTfcPairsPerWarp = 3;
// Shared memory per CTA: at most half an SM's, so that two CTAs fit on an SM and every
// cluster of a launch of 16 channel blocks is resident at once (at one CTA per SM the
// 8-CTA clusters of such a launch ran in two waves).
constexpr size_t kTfcSmemCap = 115712;

template <int F>
struct TinyFgcShape {
    static constexpr int M = kTinyMap, P = (F - 1) / 2;
    // (fh, oh) pairs that meet the map: filter row fh meets M - |fh - P| output rows
    static constexpr int NP = F * M - P * (P + 1);
    static constexpr int NWC = (NP + kTfcPairsPerWarp - 1) / kTfcPairsPerWarp;   // compute warps
    static constexpr int THREADS = (NWC + 1) * 32;
    // pair partials [NWC * 3][F][64] and the CTA partial [F][F][64], fp32, in the ring
    static constexpr int PAIR_FLOATS = NWC * kTfcPairsPerWarp * F * 64;
    static constexpr int RED_BYTES = (PAIR_FLOATS + F * F * 64) * 4;
    static constexpr int RING_OFF = kTfcBarBytes;
};

struct TinyFgcArgs {
    float* dw;                  // F x F x C
    unsigned int* status;
    unsigned long long wait_ns;
    int N, C, ipb, ns;          // images per CTA, ring slots
    uint32_t img_bytes;         // one staged image: 49 pixels x 64 channels
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Two floats at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float2 ld_cluster_f2(const float* local, uint32_t rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(r) : "memory");
    return v;
}

// Pair p of the list (filter rows in order, each with its output rows in order): its
// filter row and output row, or false past the list's end.
template <int F>
__device__ __forceinline__ bool tiny_pair(int p, int& fh, int& oh) {
    constexpr int M = kTinyMap, P = (F - 1) / 2;
#pragma unroll
    for (int f = 0; f < F; ++f) {
        const int lo = f < P ? P - f : 0;              // first output row filter row f meets
        const int n = M - (f < P ? P - f : f - P);     // output rows it meets
        if (p < n) {
            fh = f;
            oh = lo + p;
            return true;
        }
        p -= n;
    }
    return false;
}

// Grid: (channel blocks, Z), clusters of (1, Z, 1): CTA z of a cluster takes the images
// [z * ipb, (z + 1) * ipb).
template <typename T, int F>
__global__ void __launch_bounds__(TinyFgcShape<F>::THREADS, 2)
tiny_fgrad_cluster_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap dmap,
                          const TinyFgcArgs a) {
    using Sh = TinyFgcShape<F>;
    constexpr int M = kTinyMap, P = Sh::P, NWC = Sh::NWC, K = kTfcPairsPerWarp;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + a.ns;
    unsigned char* ring = smem + Sh::RING_OFF;
    float* pairs = reinterpret_cast<float*>(ring);   // after the last image is consumed
    float* part = pairs + Sh::PAIR_FLOATS;            // the CTA partial [F][F][64]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cb = blockIdx.x;
    const uint32_t rank = cluster_ctarank();
    const uint32_t nrank = gridDim.y;
    const int n0 = static_cast<int>(blockIdx.y) * a.ipb;
    const int nimg = max(0, min(a.N, n0 + a.ipb) - n0);
    if (threadIdx.x == 0) {
        for (int k = 0; k < a.ns; ++k) {
            mbar_init(&full[k], 1);
            mbar_init(&empty[k], NWC);   // every compute warp reads every image
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NWC) {
        // ---- producer: image i -> slot i mod ns ----
        if (lane == 0) {
            prefetch_tensormap(&xmap);
            prefetch_tensormap(&dmap);
            bool ok = true;
            for (int i = 0; i < nimg && ok; ++i) {
                const int k = i % a.ns;
                const uint32_t ph = static_cast<uint32_t>(i / a.ns) & 1u;
                if (i >= a.ns && !mbar_wait(&empty[k], ph ^ 1u, a.wait_ns)) {
                    ok = false;
                    break;
                }
                unsigned char* dst = ring + static_cast<size_t>(k) * 2 * a.img_bytes;
                mbar_arrive_expect_tx(&full[k], 2 * a.img_bytes);
                tma_load_4d(dst, &xmap, &full[k], cb * 64, 0, 0, n0 + i);
                tma_load_4d(dst + a.img_bytes, &dmap, &full[k], cb * 64, 0, 0, n0 + i);
            }
            if (!ok) record_status(a.status, DWC_DEVSTAT_TIMEOUT);
            // the copies still in flight land before the ring is reused or the CTA leaves
            for (int i = max(0, nimg - a.ns); i < nimg; ++i)
                if (!mbar_wait(&full[i % a.ns], static_cast<uint32_t>(i / a.ns) & 1u, a.wait_ns)) {
                    record_status(a.status, DWC_DEVSTAT_TIMEOUT);
                    break;
                }
        }
        __syncwarp();
    }
    // ---- compute warp w: pairs K*w .. K*w + K - 1 of every image ----
    int pfh[K], poh[K];
    bool pok[K];
#pragma unroll
    for (int j = 0; j < K; ++j) pok[j] = warp < NWC && tiny_pair<F>(warp * K + j, pfh[j], poh[j]);
    float2 acc[K][F];
#pragma unroll
    for (int j = 0; j < K; ++j)
#pragma unroll
        for (int fw = 0; fw < F; ++fw) acc[j][fw] = make_float2(0.f, 0.f);
    if (warp < NWC) {
        for (int i = 0; i < nimg; ++i) {
            const int k = i % a.ns;
            if (!mbar_wait(&full[k], static_cast<uint32_t>(i / a.ns) & 1u, a.wait_ns)) {
                record_status(a.status, DWC_DEVSTAT_TIMEOUT);
                break;
            }
            const T* X = reinterpret_cast<const T*>(ring + static_cast<size_t>(k) * 2 * a.img_bytes) + 2 * lane;
            const T* D = reinterpret_cast<const T*>(ring + static_cast<size_t>(k) * 2 * a.img_bytes + a.img_bytes) + 2 * lane;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (!pok[j]) continue;
                const int ih = poh[j] + pfh[j] - P;
                float2 d[M], x[M];
#pragma unroll
                for (int c = 0; c < M; ++c) {
                    d[c] = Elem<T>::load_pair(D + (poh[j] * M + c) * 64);
                    x[c] = Elem<T>::load_pair(X + (ih * M + c) * 64);
                }
#pragma unroll
                for (int fw = 0; fw < F; ++fw)
#pragma unroll
                    for (int ow = 0; ow < M; ++ow) {
                        const int iw = ow + fw - P;
                        if (iw < 0 || iw >= M) continue;
                        fma2(acc[j][fw], x[iw], d[ow]);
                    }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[k]);
        }
    }
    // every image consumed and every copy landed (the producer drained): the ring becomes
    // the pair partials, then the CTA partial (filter row fh: its pairs in list order)
    __syncthreads();
    if (warp < NWC) {
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
            for (int fw = 0; fw < F; ++fw)
                *reinterpret_cast<float2*>(pairs + ((warp * K + j) * F + fw) * 64 + 2 * lane) = acc[j][fw];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < F * F * 32; e += blockDim.x) {
        const int fh = e / (F * 32), fw = (e / 32) % F, cp = e % 32;
        int p0 = 0;
        for (int f = 0; f < fh; ++f) p0 += M - (f < P ? P - f : f - P);
        const int n = M - (fh < P ? P - fh : fh - P);
        float2 v = make_float2(0.f, 0.f);
        for (int r = 0; r < n; ++r) {
            const float2 t = *reinterpret_cast<const float2*>(pairs + ((p0 + r) * F + fw) * 64 + 2 * cp);
            v.x += t.x;
            v.y += t.y;
        }
        *reinterpret_cast<float2*>(part + (fh * F + fw) * 64 + 2 * cp) = v;
    }
    // every CTA's partial is in its shared memory
    __syncwarp();
    cluster_sync_all();
    // this CTA's share of the F x F x 64 outputs (channel pairs e), summed over the
    // cluster's CTAs in rank order (all loads issued first)
    constexpr int E2 = F * F * 32;
    for (int e = static_cast<int>(rank * blockDim.x + threadIdx.x); e < E2; e += static_cast<int>(nrank * blockDim.x)) {
        float2 t[kTfcMaxZ];
#pragma unroll
        for (int q = 0; q < kTfcMaxZ; ++q)
            t[q] = static_cast<uint32_t>(q) < nrank ? ld_cluster_f2(part + 2 * e, q) : make_float2(0.f, 0.f);
        float2 v = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kTfcMaxZ; ++q) {
            v.x += t[q].x;
            v.y += t[q].y;
        }
        const int c = cb * 64 + 2 * (e % 32);
        if (c < a.C) *reinterpret_cast<float2*>(a.dw + static_cast<size_t>(e / 32) * a.C + c) = v;
    }
    // no CTA leaves while another still reads its shared memory
    cluster_sync_all();
}

// Plan of the cluster form: Z CTAs per channel block (at most 8, one cluster), ipb images
// each, ring slots a multiple of S that fit in shared memory.  False where the channels
// cannot be copied with tensor copies (rows of C elements must be 16-byte multiples).
template <typename T, int F>
bool tiny_fgrad_cluster_plan(int N, int C, int& Z, int& ipb, int& ns, size_t& smem) {
    using Sh = TinyFgcShape<F>;
    if (N <= 0 || C <= 0 || (static_cast<size_t>(C) * sizeof(T)) % 16 != 0) return false;
    Z = std::min(N, kTfcMaxZ);
    ipb = (N + Z - 1) / Z;
    Z = (N + ipb - 1) / ipb;
    const size_t img = static_cast<size_t>(kTinyMap) * kTinyMap * 64 * sizeof(T);
    const size_t cap = std::min(kTfcSmemCap, static_cast<size_t>(device_info().max_smem_optin));
    const int fit = static_cast<int>((cap - Sh::RING_OFF) / (2 * img));
    ns = std::min(fit, ipb);
    if (ns < std::min(2, ipb) || 2 * ns * sizeof(uint64_t) > static_cast<size_t>(kTfcBarBytes)) return false;
    smem = Sh::RING_OFF + std::max(static_cast<size_t>(ns) * 2 * img, static_cast<size_t>(Sh::RED_BYTES));
    return smem <= cap;
}

template <typename T, int F>
cudaError_t launch_tiny_fgrad_cluster(const FilterGrad& p) {
    using Sh = TinyFgcShape<F>;
    int Z = 0, ipb = 0, ns = 0;
    size_t smem = 0;
    if (!tiny_fgrad_cluster_plan<T, F>(p.N, p.C, Z, ipb, ns, smem)) return cudaErrorNotSupported;
    auto kern = tiny_fgrad_cluster_kernel<T, F>;
    static DeviceOnce smem_opt_in;
    cudaError_t err = opt_in_smem(kern, smem_opt_in, device_info().max_smem_optin);
    if (err != cudaSuccess) return err;
    const int e = static_cast<int>(sizeof(T));
    CUtensorMap xmap, dmap;
    const cuuint64_t dims[4] = {(cuuint64_t)p.C, (cuuint64_t)kTinyMap, (cuuint64_t)kTinyMap, (cuuint64_t)p.N};
    const cuuint64_t strides[3] = {(cuuint64_t)p.C * e, (cuuint64_t)kTinyMap * p.C * e,
                                   (cuuint64_t)kTinyMap * kTinyMap * p.C * e};
    const cuuint32_t box[4] = {64u, (cuuint32_t)kTinyMap, (cuuint32_t)kTinyMap, 1u};
    if (encode_tiled(&xmap, Elem<T>::kTmaType, 4, const_cast<void*>(p.x), dims, strides, box) != CUDA_SUCCESS ||
        encode_tiled(&dmap, Elem<T>::kTmaType, 4, const_cast<void*>(p.dy), dims, strides, box) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    TinyFgcArgs a;
    a.dw = p.dw;
    a.status = p.status;
    a.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    a.N = p.N;
    a.C = p.C;
    a.ipb = ipb;
    a.ns = ns;
    a.img_bytes = static_cast<uint32_t>(kTinyMap * kTinyMap * 64 * e);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((p.C + 63) / 64), static_cast<unsigned>(Z), 1);
    cfg.blockDim = dim3(Sh::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = p.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(Z);
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (err != cudaSuccess || clusters < 1) {
        (void)cudaGetLastError();
        return cudaErrorNotSupported;
    }
    err = cudaLaunchKernelEx(&cfg, kern, xmap, dmap, a);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

// Whether the one-launch cluster form serves a 7x7-map filter gradient of these sizes
// (3 taps only).
template <typename T>
bool tiny_fgrad_cluster_fits(int N, int C, int F) {
    int Z, ipb, ns;
    size_t smem;
    return F == 3 && tiny_fgrad_cluster_plan<T, 3>(N, C, Z, ipb, ns, smem);
}


#define DWC_SMALL_SHAPES(X) X(8, 3) X(8, 7) X(16, 3) X(16, 7) X(16, 11) X(16, 15)

template <typename T>
size_t small_fgrad_workspace_t(int N, int H, int W, int C, int OH, int OW, int FH, int FW, int pad) {
    if (tiny_shape(H, W, OH, OW, FH, FW, pad, pad)) return tiny_fgrad_workspace_floats(N, C, FH);
    int maxw = 0, dr = 0;
    if (!small_fgrad_wanted(W, OW, FW) || !small_shape(H, W, OH, OW, FW, pad, maxw, dr)) return 0;
    SmallFgArgs a;
    size_t smem = 0;
    int nwarps = 0;
    bool ok = false;
#define DWC_SMALL_FG_PLAN(M, D) \
    if (maxw == M && dr == D) ok = small_fgrad_plan<T, M, D>(N, H, W, C, OH, OW, FH, pad, a, smem, nwarps);
    DWC_SMALL_SHAPES(DWC_SMALL_FG_PLAN)
#undef DWC_SMALL_FG_PLAN
    if (!ok) return 0;
    const size_t Z = static_cast<size_t>((N + a.ipc - 1) / a.ipc);
    return Z * a.nfh * FW * static_cast<size_t>(C);
}


template <typename T, class OutT = float>
cudaError_t launch_small_rows_t(const RowConv& p) {
    if (tiny_shape(p.H, p.W, p.OH, p.OW, p.FH, p.FW, p.pad_h, p.pad_w)) return launch_tiny_rows<T, OutT>(p);
    int maxw = 0, dr = 0;
    if (!small_rows_wanted(p.W, p.OW, p.FW) || !small_shape(p.H, p.W, p.OH, p.OW, p.FW, p.pad_w, maxw, dr))
        return cudaErrorNotSupported;
#define DWC_SMALL_ROWS_CASE(M, D) \
    if (maxw == M && dr == D) return launch_small_rows_inst<T, M, D, OutT>(p);
    DWC_SMALL_SHAPES(DWC_SMALL_ROWS_CASE)
#undef DWC_SMALL_ROWS_CASE
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t launch_small_fgrad_t(const FilterGrad& p) {
    if (tiny_shape(p.H, p.W, p.OH, p.OW, p.FH, p.FW, p.pad, p.pad)) return launch_tiny_fgrad<T>(p);
    int maxw = 0, dr = 0;
    if (!small_fgrad_wanted(p.W, p.OW, p.FW) || !small_shape(p.H, p.W, p.OH, p.OW, p.FW, p.pad, maxw, dr))
        return cudaErrorNotSupported;
#define DWC_SMALL_FG_CASE(M, D) \
    if (maxw == M && dr == D) return launch_small_fgrad_inst<T, M, D>(p);
    DWC_SMALL_SHAPES(DWC_SMALL_FG_CASE)
#undef DWC_SMALL_FG_CASE
    return cudaErrorNotSupported;
}

}  // namespace dwc
