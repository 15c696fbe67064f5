// dwc_rows.cuh -- row-streaming depthwise convolution kernel (forward and backward data).
//
// Computes, for stride 1,
//   out[n, oh, ow, c] = sum_{fh < FH, fw < FW} in[n, oh + fh - pad_h, ow + fw - pad_w, c] * filt(fh, fw, c)
// over channels-last tensors ("Flash-DWC: Making Depthwise Convolution Compute-Efficient on
// GPUs", §2.1 / Fig. 1 for the operation, §2.3 for the unified channels-last layout).  For
// backward data, filt(fh, fw, c) = w[FH-1-fh, FW-1-fw, c] (the 180-degree rotation of §5.1),
// folded into the filter index so no rotated copy of w is ever written.
//
// Design (GB300 restatement of the §3 dataflow, not a copy of it):
//  * Work unit = (image n, block of 64 channels, band of R output rows, tile of TW = nwc*TM
//    output columns) -- the output tiling of §3.1 with BN = 64 channels.  A persistent grid
//    walks the units; the band index is fastest so that CTAs running at the same time read
//    overlapping input rows out of L2.
//  * One producer warp streams, per unit, the R + FH - 1 input rows of the band (each a
//    64-channel x (TW + FW - 1)-pixel box) and the filter rows through a ring of shared
//    memory stages with TMA.  Out-of-image rows, columns and channels arrive zero-filled,
//    which is the zero padding (the predicated loads of §4.4 become TMA bounds handling).
//  * Each compute lane owns two adjacent channels (one packed fp32x2 FMA per tap) and a
//    block of R rows x TM columns of outputs in registers.  Input rows are consumed in order;
//    every input element is loaded from shared memory once and used for up to R*FW taps
//    (width-first reuse inside a row, §3.3, plus reuse across the R output rows the lane
//    holds).  The filter rows in use live in registers as a window of R rows that slides
//    by one row per input row (filter reuse across TM*R outputs, §3.2).
//  * 16-bit inputs are widened to fp32 once per shared-memory load, not per FMA (§4.1).
//  * Optional BN + Act fusion (§5.2, forward only): each input value is normalised with the
//    channel's batch statistics and activated right after its shared-memory load, before
//    its taps; values that lie in the padding are replaced by zero (the DWC pads the
//    activated tensor), and input rows outside the image are skipped.
#pragma once

#include <climits>
#include <type_traits>
#include <utility>

#include "dwc_device.cuh"
#include "dwc_host.h"

namespace dwc {

constexpr int kBN = 64;                 // channels per work unit (32 lanes x 2)
constexpr int kMaxComputeWarps = 7;   // + 1 producer warp = 256 threads per CTA
constexpr int kRowsMaxThreads = (kMaxComputeWarps + 1) * 32;

// Register tile per filter size: R output rows x TM output columns per lane.
// R > 1 unrolls all R + FH - 1 input rows of a band (compile-time filter-register slots),
// so it is used for the smaller filters only; large filters take one output row per lane
// and a rolled row loop.
// Chosen by timing candidate tiles on the filter sizes of the benchmark shapes.
template <int FH, int FW>
struct RowsTile {
    static constexpr int R = (FH <= 3) ? 8 : (FH <= 5 ? 4 : (FH <= 15 ? 2 : 1));
    static constexpr int TM = (FH <= 3) ? 4 : (FH <= 15 ? 8 : 14);
    // CTAs per SM for the registers (past 31 taps a filter row alone takes ~100 registers)
    static constexpr int MINB = FH == 7 ? 3 : (FH > 31 ? 1 : 2);
};

struct RowsArgs {
    void* out;            // OutT elements
    unsigned int* status;
    int H, W;             // input rows / columns (rows and columns that lie in the padding)
    int OH, OW, C;
    int pad_h, pad_w;
    int FH;               // filter rows (the kernel's template FH, or any for FH = 0)
    int cbase;            // first channel of channel block 0
    int nwc;              // compute warps per CTA
    int ns;               // pipeline stages
    uint32_t cblocks, bands, ctiles;
    FastDiv fd_bands, fd_ctiles, fd_cblocks;   // the same three, as invariant divisors
    uint32_t units;
    uint32_t x_bytes;     // bytes of one staged input row box
    uint32_t w_off;       // offset of the filter row in a stage (x_bytes rounded up to 128)
    uint32_t w_bytes;     // bytes of one staged filter row box
    uint32_t stage_stride;
    unsigned long long wait_ns;  // limit of every mbarrier wait
    int stall;            // fault injection (tests): CTA 0 issues no copy, so it times out
    // fused BN + Act (ACT >= 0): batch statistics and affine parameters, C floats each
    const float* bn_mean;
    const float* bn_var;
    const float* bn_gamma;
    const float* bn_beta;
    float bn_eps;
};

// Value transform between the shared-memory load and the taps.  NoXform: the plain DWC.
struct NoXform {
    template <class V>
    __device__ __forceinline__ V operator()(V x, int) const { return x; }
};

// BN + Act on a pair of channels: z = act(x * scale + shift) with scale = gamma / sqrt(var +
// eps) and shift = beta - mean * scale; ACT 0 = identity, 1 = ReLU, 2 = ReLU6.  MASKED: bit
// j of colmask says whether staged column j lies inside the image, and a column in the
// padding yields zero.  Every lane of a warp stages the same columns, so a warp whose
// columns all lie inside the image runs the unmasked form.
template <class P, int ACT, bool MASKED>
struct BnActXform {
    typename P::V scale, shift;
    uint32_t colmask;
    __device__ __forceinline__ typename P::V operator()(typename P::V x, int j) const {
        typename P::V z = shift;
        P::fma(z, x, scale);
        if constexpr (ACT >= 1) {
            float2 f = P::unpack(z);
            f.x = fmaxf(f.x, 0.f);
            f.y = fmaxf(f.y, 0.f);
            if constexpr (ACT == 2) {
                f.x = fminf(f.x, 6.f);
                f.y = fminf(f.y, 6.f);
            }
            z = P::pack(f.x, f.y);
        }
        if constexpr (MASKED) return ((colmask >> j) & 1u) ? z : P::zero();
        return z;
    }
};

template <int I>
using IntC = std::integral_constant<int, I>;
template <unsigned U>
using UIntC = std::integral_constant<unsigned, U>;

// Input rows i of a one-row band (output row oh0, input row oh0 - pad + i) that fall
// inside the image: [i_lo, i_hi) intersected with the band's [i_lo, i_hi).  Rows outside
// contribute only zeros (the trimming of shared zero rows described in §4.4).
__device__ __forceinline__ void rows_in_image(int oh0, int pad, int H, int& i_lo, int& i_hi) {
    i_lo = max(i_lo, pad - oh0);
    i_hi = min(i_hi, H + pad - oh0);
    if (i_hi < i_lo) i_hi = i_lo;
}

template <class F, int... Is>
__device__ __forceinline__ void static_for_impl(F&& f, std::integer_sequence<int, Is...>) {
    (f(IntC<Is>{}), ...);
}

template <int N, class F>
__device__ __forceinline__ void static_for(F&& f) {
    static_for_impl(f, std::make_integer_sequence<int, N>{});
}

// Valid output rows r of the lane's band for input row i: 0 <= i - r < FH.
template <int R, int FH>
__host__ __device__ constexpr unsigned valid_rows(int i) {
    unsigned m = 0;
    for (int r = 0; r < R; ++r)
        if (i - r >= 0 && i - r < FH) m |= 1u << r;
    return m;
}

// Accumulate one staged input row i into the lane's R x TM outputs.  Output row r (in
// MASK) takes filter row i - r, held in register slot (i - r) mod R; ISLOT = i mod R.
// With column stride SD, input column j of the lane feeds output t through tap
// fw = j - SD * t.
template <class P, typename T, int FW, int R, int TM, unsigned MASK, int ISLOT, int SD = 1,
          class XF = NoXform, int PITCH = kBN>
__device__ __forceinline__ void consume_rows(const T* __restrict__ xs, typename P::V (&acc)[R][TM],
                                             const typename P::V (&wwin)[R][FW], const XF& xf = XF{}) {
#pragma unroll
    for (int j = 0; j < SD * (TM - 1) + FW; ++j) {
        const typename P::V x = xf(P::load(xs + j * PITCH), j);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (!((MASK >> r) & 1u)) continue;
            const int slot = (ISLOT - r + R) % R;
#pragma unroll
            for (int fw = 0; fw < FW; ++fw) {
                if ((j - fw) % SD != 0) continue;
                const int t = (j - fw) / SD;
                if (j - fw >= 0 && t < TM) P::fma(acc[r][t], x, wwin[slot][fw]);
            }
        }
    }
}

// SD: stride of both spatial axes (1, or 2 with one output row per band).  ACT: -1 plain
// DWC, else BN + Act fused in front (0 identity, 1 ReLU, 2 ReLU6; forward only).  OutT:
// output element type (fp32, or the 16-bit input type).
// G: lane groups (1, or 2 / 4 for a tail block of at most 32 / 16 channels: each group of
// 32 / G lanes covers the block's channels for its own TM columns, so no lane idles).
template <typename T, int FH, int FW, int R, int TM, int MINB, bool FLIP, class P = Pair64, int SD = 1,
          int ACT = -1, class OutT = float, int G = 1>
__global__ void __launch_bounds__(kRowsMaxThreads, MINB)
rows_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
            const RowsArgs a) {
    static_assert(SD == 1 || (R == 1 && !FLIP), "strided bands hold one output row (forward)");
    static_assert(ACT < 0 || !FLIP, "BN + Act fusion precedes the forward pass only");
    static_assert(ACT < 0 || SD * (TM - 1) + FW <= 32, "column mask holds 32 staged columns");
    static_assert(FH > 0 || R == 1, "a filter height chosen at run time needs one-row bands");
    static_assert(G == 1 || G == 2 || G == 4, "lane groups");
    static_assert(G == 1 || ACT < 0, "lane groups run the plain DWC");
    constexpr int PITCH = kBN / G;   // channels per staged pixel
    constexpr int LPG = 32 / G;      // lanes per group
    // filter rows: the template's, or (FH = 0, stripe filters) the launch's
    const int fhn = FH > 0 ? FH : a.FH;
    constexpr int SC = R + FH - 1;  // input rows per band (compile time, R > 1)
    const int S = FH > 0 ? SC : R + fhn - 1;

    extern __shared__ __align__(128) unsigned char smem[];
    // a programmatic dependent of the kernel before it: the next kernel may be scheduled
    // now, and nothing in global memory is touched before the previous grid has finished
    pdl_trigger();
    pdl_wait();
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + a.ns;
    unsigned char* stages = smem + 128;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], a.nwc);
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int TW = a.nwc * G * TM;

    // ---------------- producer warp: TMA streaming of input and filter rows -------------
    if (warp == a.nwc) {
        if (lane != 0) return;
        prefetch_tensormap(&xmap);
        prefetch_tensormap(&wmap);
        Ring ring;
        uint32_t issued = 0;  // stages issued so far (saturating; only compared with ns)
        // fault injection: CTA 0 issues nothing, so no copy is ever in flight while its
        // compute warps run out their wait limit
        bool ok = !(a.stall && blockIdx.x == 0);
        for (uint32_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
            uint32_t r0, r1, r2;
            const uint32_t q = a.fd_cblocks.divmod(a.fd_ctiles.divmod(a.fd_bands.divmod(u, r0), r1), r2);
            const int band = static_cast<int>(r0), ct = static_cast<int>(r1), cb = static_cast<int>(r2);
            const int n = static_cast<int>(q);
            const int oh0 = band * R, ow0 = ct * TW;
            int i_lo = 0, i_hi = S;
            if constexpr (R == 1) rows_in_image(oh0 * SD, a.pad_h, a.H, i_lo, i_hi);
            for (int i = i_lo; i < i_hi; ++i, ring.next(a.ns)) {
                // slot reuse: wait until every compute warp released its previous stage
                if (issued >= static_cast<uint32_t>(a.ns) &&
                    !mbar_wait(&empty[ring.slot], ring.phase ^ 1u, a.wait_ns)) {
                    record_status(a.status, DWC_DEVSTAT_TIMEOUT);
                    ok = false;
                    break;
                }
                if (issued < static_cast<uint32_t>(a.ns)) ++issued;
                unsigned char* st = stages + static_cast<size_t>(ring.slot) * a.stage_stride;
                const bool wrow = i < fhn;
                mbar_arrive_expect_tx(&full[ring.slot], a.x_bytes + (wrow ? a.w_bytes : 0u));
                tma_load_4d(st, &xmap, &full[ring.slot], a.cbase + cb * PITCH, ow0 * SD - a.pad_w,
                            oh0 * SD - a.pad_h + i, n);
                if (wrow)
                    tma_load_3d(st + a.w_off, &wmap, &full[ring.slot], a.cbase + cb * PITCH, 0,
                                FLIP ? fhn - 1 - i : i);
            }
        }
        // Never leave the CTA with copies in flight: wait (bounded) for the stages still
        // outstanding (the last `issued` ones, walking the ring backwards).
        for (uint32_t j = 0; j < issued; ++j) {
            ring.slot = ring.slot == 0 ? a.ns - 1 : ring.slot - 1;
            if (ring.slot == static_cast<uint32_t>(a.ns) - 1) ring.phase ^= 1u;
            if (!mbar_wait(&full[ring.slot], ring.phase, a.wait_ns)) {
                record_status(a.status, DWC_DEVSTAT_TIMEOUT);
                break;
            }
        }
        return;
    }

    // ---------------- compute warps ----------------------------------------------------
    const int wc = warp;
    const int lg = lane / LPG;       // lane group: column sub-tile wc * G + lg
    const int cl = lane % LPG;       // channel pair within the block
    Ring ring;
    for (uint32_t u = blockIdx.x; u < a.units; u += gridDim.x) {
        uint32_t r0, r1, r2;
        const uint32_t q = a.fd_cblocks.divmod(a.fd_ctiles.divmod(a.fd_bands.divmod(u, r0), r1), r2);
        const int band = static_cast<int>(r0), ct = static_cast<int>(r1), cb = static_cast<int>(r2);
        const int n = static_cast<int>(q);
        const int oh0 = band * R;
        const int owl = ct * TW + (wc * G + lg) * TM;  // first output column of this lane
        const int c = a.cbase + cb * PITCH + 2 * cl;

        // BN + Act of this lane's two channels and the staged columns inside the image
        using XFull = typename std::conditional<(ACT >= 0), BnActXform<P, ACT, false>, NoXform>::type;
        using XMask = typename std::conditional<(ACT >= 0), BnActXform<P, ACT, true>, NoXform>::type;
        XMask xf{};
        bool colfull = true;
        if constexpr (ACT >= 0) {
            float sc[2] = {0.f, 0.f}, sh[2] = {0.f, 0.f};
            if (c < a.C) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    sc[k] = a.bn_gamma[c + k] * rsqrtf(a.bn_var[c + k] + a.bn_eps);
                    sh[k] = a.bn_beta[c + k] - a.bn_mean[c + k] * sc[k];
                }
            }
            xf.scale = P::pack(sc[0], sc[1]);
            xf.shift = P::pack(sh[0], sh[1]);
            const int iw0 = ct * TW * SD - a.pad_w + wc * TM * SD;
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < SD * (TM - 1) + FW; ++j)
                if (iw0 + j >= 0 && iw0 + j < a.W) m |= 1u << j;
            xf.colmask = m;
            constexpr int ncols = SD * (TM - 1) + FW;
            colfull = m == (ncols >= 32 ? ~0u : (1u << ncols) - 1u);
        }
        // whether input row i of the band lies inside the image (rows in the padding add
        // nothing to the plain DWC, whose staged copy is zero; with BN + Act they are skipped)
        auto row_in = [&](int i) -> bool {
            if constexpr (ACT < 0) {
                return true;
            } else {
                const int ih = oh0 * SD - a.pad_h + i;
                return ih >= 0 && ih < a.H;
            }
        };

        typename P::V acc[R][TM];
        typename P::V wwin[R][FW];
        // (every filter slot is loaded at its first row before any tap reads it)
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int t = 0; t < TM; ++t) acc[r][t] = P::zero();
        }
        // consume one staged row (output-row mask M, filter slot SL) with the transform the
        // warp's columns need; where the band is unrolled (R > 1) a second copy of the row
        // code costs more in instruction fetch than the mask saves, so those bands always
        // take the masked form
        auto consume = [&](auto mc, auto sc, const T* xs) {
            constexpr unsigned M = decltype(mc)::value;
            constexpr int SL = decltype(sc)::value;
            if constexpr (ACT < 0) {
                consume_rows<P, T, FW, R, TM, M, SL, SD, NoXform, PITCH>(xs, acc, wwin);
            } else if constexpr (R > 1) {
                consume_rows<P, T, FW, R, TM, M, SL, SD>(xs, acc, wwin, xf);
            } else if (colfull) {
                consume_rows<P, T, FW, R, TM, M, SL, SD>(xs, acc, wwin, XFull{xf.scale, xf.shift, 0u});
            } else {
                consume_rows<P, T, FW, R, TM, M, SL, SD>(xs, acc, wwin, xf);
            }
        };

        // Filter row fh lives in register slot fh % R: it enters at input row i = fh and is
        // last used at i = fh + R - 1, when row fh + R (same slot) is not yet needed.
        // Wait for the stage of input row i, load filter row i into its slot (i < FH) and
        // return the row's shared-memory pointer.  The slot index is a compile-time
        // constant wherever the row loop is unrolled, so no register ever moves.
        auto begin_row = [&](auto ic, int i, const T*& xs) -> bool {
            if (!mbar_wait(&full[ring.slot], ring.phase, a.wait_ns)) {
                record_status(a.status, DWC_DEVSTAT_TIMEOUT);
                return false;
            }
            const unsigned char* st = stages + static_cast<size_t>(ring.slot) * a.stage_stride;
            constexpr int slot = decltype(ic)::value % R;
            if (i < fhn) {
                const T* ws = reinterpret_cast<const T*>(st + a.w_off) + 2 * cl;
#pragma unroll
                for (int f = 0; f < FW; ++f)
                    wwin[slot][f] = P::load(ws + (FLIP ? FW - 1 - f : f) * PITCH);
            }
            xs = reinterpret_cast<const T*>(st) + ((wc * G + lg) * TM * SD) * PITCH + 2 * cl;
            return true;
        };
        auto end_row = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[ring.slot]);
            ring.next(a.ns);
        };

        bool ok = true;
        if constexpr (R == 2 && FH >= 9) {
            // Two output rows, rolled in pairs of input rows (the fully unrolled band of
            // FH + 1 rows overflows the instruction cache from 9 taps on): input row 0 feeds
            // output row 0 only, rows 1..FH-1 both, row FH output row 1 only; filter row i
            // goes to register slot i % 2, so the slots stay compile-time constants.
            const T* xs;
            if (!begin_row(IntC<0>{}, 0, xs)) {
                ok = false;
            } else {
                if (row_in(0)) consume(UIntC<1u>{}, IntC<0>{}, xs);
                end_row();
            }
#pragma unroll 1
            for (int i = 1; i < FH && ok; i += 2) {
                if (!begin_row(IntC<1>{}, i, xs)) { ok = false; break; }
                if (row_in(i)) consume(UIntC<3u>{}, IntC<1>{}, xs);
                end_row();
                if (!begin_row(IntC<0>{}, i + 1, xs)) { ok = false; break; }
                if (row_in(i + 1)) consume(UIntC<3u>{}, IntC<0>{}, xs);
                end_row();
            }
            if (ok) {
                if (!begin_row(IntC<1>{}, FH, xs)) {
                    ok = false;
                } else {
                    if (row_in(FH)) consume(UIntC<2u>{}, IntC<1>{}, xs);
                    end_row();
                }
            }
        } else if constexpr (R > 1) {
            // every input row of the band unrolled: output row r takes filter row i - r
            // from slot (i - r) % R
            static_for<SC>([&](auto I) {
                constexpr int i = decltype(I)::value;
                if (!ok) return;
                const T* xs;
                if (!begin_row(I, i, xs)) { ok = false; return; }
                if (row_in(i)) consume(UIntC<valid_rows<R, FH>(i)>{}, IntC<i % R>{}, xs);
                end_row();
            });
        } else {
            // one output row: the filter row for input row i is simply row i; input rows
            // that lie entirely in the zero padding are neither loaded nor computed
            int i_lo = 0, i_hi = S;
            rows_in_image(oh0 * SD, a.pad_h, a.H, i_lo, i_hi);
#pragma unroll 1
            for (int i = i_lo; i < i_hi && ok; ++i) {
                const T* xs;
                if (!begin_row(IntC<0>{}, i, xs)) { ok = false; break; }
                consume(UIntC<1u>{}, IntC<0>{}, xs);
                end_row();
            }
        }
        if (!ok) return;

        if (c < a.C) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int oh = oh0 + r;
                if (oh >= a.OH) break;
                OutT* row = static_cast<OutT*>(a.out) + ((static_cast<size_t>(n) * a.OH + oh) * a.OW + owl) * a.C + c;
                if (owl + TM <= a.OW) {
#pragma unroll
                    for (int t = 0; t < TM; ++t)
                        store_out_pair(row + static_cast<size_t>(t) * a.C, P::unpack(acc[r][t]));
                } else {
#pragma unroll
                    for (int t = 0; t < TM; ++t)
                        if (owl + t < a.OW)
                            store_out_pair(row + static_cast<size_t>(t) * a.C, P::unpack(acc[r][t]));
                }
            }
        }
    }
}

template <typename T, int FH, int FW, int R, int TM, int MINB, bool FLIP, class P = Pair64, int SD = 1,
          int ACT = -1, class OutT = float, int G = 1>
cudaError_t launch_rows_inst(const RowConv& p) {
    const int e = static_cast<int>(sizeof(T));
    const DeviceInfo& dev = device_info();
    constexpr int PITCH = kBN / G;
    // channels [c_lo, c_hi) of the tensor (the tail launch of lane groups covers only the
    // channels past the last multiple of 64)
    const int c_lo = p.c_lo, c_hi = p.c_hi < 0 ? p.C : p.c_hi;
    if (c_hi <= c_lo) return cudaSuccess;

    // compute warps side by side along the row (G column sub-tiles each); the staged box
    // (SD * (TW - 1) + FW pixels) must stay within the TMA box limit of 256
    const int max_nwc = std::min(kMaxComputeWarps, (256 - FW + SD) / (SD * G * TM));
    if (max_nwc < 1) return cudaErrorNotSupported;
    // warps per row tile: fewest computed columns plus half a halo per column tile
    int nwc = 1;
    long long best = LLONG_MAX;
    for (int n = 1; n <= max_nwc; ++n) {
        const int tw = n * G * TM;
        const long long tiles = (p.OW + tw - 1) / tw;
        const long long cost = 2 * tiles * tw + tiles * (FW - 1);
        if (cost <= best) { best = cost; nwc = n; }
    }
    const int TW = nwc * G * TM;
    const int TWH = SD * (TW - 1) + FW;

    CUtensorMap xmap, wmap;
    {
        const cuuint64_t dims[4] = {(cuuint64_t)p.C, (cuuint64_t)p.W, (cuuint64_t)p.H,
                                    (cuuint64_t)p.N};
        const cuuint64_t strides[3] = {(cuuint64_t)p.C * e, (cuuint64_t)p.W * p.C * e,
                                       (cuuint64_t)p.H * p.W * p.C * e};
        const cuuint32_t box[4] = {(cuuint32_t)PITCH, (cuuint32_t)TWH, 1u, 1u};
        if (encode_tiled(&xmap, Elem<T>::kTmaType, 4, const_cast<void*>(p.in), dims, strides,
                         box) != CUDA_SUCCESS)
            return cudaErrorNotSupported;  // the caller falls back to the general kernels
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p.C, (cuuint64_t)FW, (cuuint64_t)p.FH};
        const cuuint64_t strides[2] = {(cuuint64_t)p.C * e, (cuuint64_t)FW * p.C * e};
        const cuuint32_t box[3] = {(cuuint32_t)PITCH, (cuuint32_t)FW, 1u};
        if (encode_tiled(&wmap, Elem<T>::kTmaType, 3, const_cast<void*>(p.w), dims, strides,
                         box) != CUDA_SUCCESS)
            return cudaErrorNotSupported;
    }

    RowsArgs a;
    a.out = p.out;
    a.status = p.status;
    a.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    a.stall = p.stall;
    a.H = p.H;
    a.W = p.W;
    a.FH = p.FH;
    a.bn_mean = p.bn_mean; a.bn_var = p.bn_var; a.bn_gamma = p.bn_gamma; a.bn_beta = p.bn_beta;
    a.bn_eps = p.bn_eps;
    a.OH = p.OH; a.OW = p.OW; a.C = p.C;
    a.pad_h = p.pad_h; a.pad_w = p.pad_w;
    a.nwc = nwc;
    a.cbase = c_lo;
    a.cblocks = static_cast<uint32_t>((c_hi - c_lo + PITCH - 1) / PITCH);
    a.bands = static_cast<uint32_t>((p.OH + R - 1) / R);
    a.ctiles = static_cast<uint32_t>((p.OW + TW - 1) / TW);
    a.fd_bands.init(a.bands);
    a.fd_ctiles.init(a.ctiles);
    a.fd_cblocks.init(a.cblocks);
    const long long units = static_cast<long long>(p.N) * a.cblocks * a.bands * a.ctiles;
    if (units >= (1LL << 31)) return cudaErrorNotSupported;
    a.units = static_cast<uint32_t>(units);
    a.x_bytes = static_cast<uint32_t>(TWH * PITCH * e);
    a.w_bytes = static_cast<uint32_t>(FW * PITCH * e);
    // TMA writes shared memory at 128-byte aligned addresses: a stage and the filter row in
    // it start on 128-byte boundaries (a staged pixel of a lane-group tail block holds only
    // 32 or 64 bytes, so the input row's size need not be a multiple of 128)
    a.w_off = (a.x_bytes + 127u) & ~127u;
    a.stage_stride = (a.w_off + a.w_bytes + 127u) & ~127u;
    if (a.units == 0) return cudaSuccess;

    auto kern = rows_kernel<T, FH, FW, R, TM, MINB, FLIP, P, SD, ACT, OutT, G>;
    const int threads = (nwc + 1) * 32;
    static int regs = -1;  // per instantiation (the same code on every device)
    if (regs < 0) {
        cudaFuncAttributes fa;
        const cudaError_t err = cudaFuncGetAttributes(&fa, kern);
        if (err != cudaSuccess) return err;
        regs = fa.numRegs;
    }
    static DeviceOnce smem_opt_in;
    {
        const cudaError_t err = opt_in_smem(kern, smem_opt_in, dev.max_smem_optin);
        if (err != cudaSuccess) return err;
    }
    // CTAs per SM allowed by registers, then split shared memory between them.
    const int regs_per_cta = ((regs * 32 + 255) / 256) * 256 * (nwc + 1);
    int ctas = std::max(1, std::min(65536 / std::max(regs_per_cta, 1), 2048 / threads));
    int ns = 0;
    for (; ctas >= 1; --ctas) {
        const int budget = std::min(dev.max_smem_optin, 233472 / ctas - 1024) - 128;
        ns = std::min(6, budget / static_cast<int>(a.stage_stride));
        if (ns >= 2) break;
    }
    if (ns < 2) return cudaErrorNotSupported;
    a.ns = ns;
    const size_t smem = 128 + static_cast<size_t>(ns) * a.stage_stride;
    const long long grid = std::min<long long>(units, static_cast<long long>(dev.sm_count) * ctas);
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(threads), smem, p.stream, xmap, wmap, a);
}

// Channel counts that are not a multiple of 64 (3x3, 5x5, 7x7, fp32 or 16-bit outputs): the
// tail of at most 32 channels runs with 2 or 4 lane groups, so that it does not leave half the
// lanes idle; below 64 channels that is the only launch, above it a second one after the
// launch over the channels below the last multiple of 64.
template <typename T, int F, int G, class OutT>
cudaError_t launch_rows_tail(const RowConv& p) {
    using Tl = RowsTile<F, F>;
    RowConv t = p;
    t.c_lo = p.C / kBN * kBN;
    return p.flip ? launch_rows_inst<T, F, F, Tl::R, Tl::TM, Tl::MINB, true, Pair64, 1, -1, OutT, G>(t)
                  : launch_rows_inst<T, F, F, Tl::R, Tl::TM, Tl::MINB, false, Pair64, 1, -1, OutT, G>(t);
}

template <typename T, int F, class OutT>
cudaError_t launch_rows_square(const RowConv& p) {
    using Tl = RowsTile<F, F>;
    if constexpr (F <= 7) {
        // C > 64: a second, serialised launch for the tail pays only where the kernel is
        // near its compute bound (7x7); the HBM-bound 3x3 / 5x5 hide the idle lanes (3x3 at
        // stride 2 on 64x112x112x96 measured 71 us in one launch, 92 us split)
        const int rem = p.C % kBN;
        if (rem != 0 && rem <= 32 && p.c_lo == 0 && p.c_hi < 0 && (p.C < kBN || F == 7)) {
            if (p.C > kBN) {
                RowConv q = p;
                q.c_hi = p.C / kBN * kBN;
                const cudaError_t err = launch_rows_square<T, F, OutT>(q);
                if (err != cudaSuccess) return err;
            }
            return rem <= 16 ? launch_rows_tail<T, F, 4, OutT>(p) : launch_rows_tail<T, F, 2, OutT>(p);
        }
    }
    return p.flip ? launch_rows_inst<T, F, F, Tl::R, Tl::TM, Tl::MINB, true, Pair64, 1, -1, OutT>(p)
                  : launch_rows_inst<T, F, F, Tl::R, Tl::TM, Tl::MINB, false, Pair64, 1, -1, OutT>(p);
}

// Dispatch over the compiled odd square filter sizes.
template <typename T, class OutT = float>
cudaError_t launch_rows_dispatch(const RowConv& p) {
    if (p.FH != p.FW) return cudaErrorNotSupported;
#define DWC_ROWS_CASE(F) \
    case F:              \
        return launch_rows_square<T, F, OutT>(p);
    switch (p.FH) {
        DWC_ROWS_CASE(3)
        DWC_ROWS_CASE(5)
        DWC_ROWS_CASE(7)
        DWC_ROWS_CASE(9)
        DWC_ROWS_CASE(11)
        DWC_ROWS_CASE(13)
        DWC_ROWS_CASE(15)
        DWC_ROWS_CASE(17)
        DWC_ROWS_CASE(19)
        DWC_ROWS_CASE(21)
        DWC_ROWS_CASE(23)
        DWC_ROWS_CASE(25)
        DWC_ROWS_CASE(27)
        DWC_ROWS_CASE(29)
        DWC_ROWS_CASE(31)
        DWC_ROWS_CASE(33)
        DWC_ROWS_CASE(35)
        DWC_ROWS_CASE(37)
        DWC_ROWS_CASE(39)
        DWC_ROWS_CASE(41)
        DWC_ROWS_CASE(43)
        DWC_ROWS_CASE(45)
        DWC_ROWS_CASE(47)
        DWC_ROWS_CASE(49)
        DWC_ROWS_CASE(51)
        default:
            return cudaErrorNotSupported;
    }
#undef DWC_ROWS_CASE
}

// Stride-2 forward: one output row per band, 8 outputs per lane (filters of 3 to 13 taps:
// the down-sampling layers of mobile networks, 3 to 7, and of large-kernel networks).
template <typename T, int F, class OutT>
cudaError_t launch_rows_s2_square(const RowConv& p) {
    if constexpr (F <= 7) {
        // a tail of at most 32 channels past the last multiple of 64: lane groups, under the
        // rule of the stride-1 launch above
        const int rem = p.C % kBN;
        if (rem != 0 && rem <= 32 && p.c_lo == 0 && p.c_hi < 0 && (p.C < kBN || F == 7)) {
            if (p.C > kBN) {
                RowConv q = p;
                q.c_hi = p.C / kBN * kBN;
                const cudaError_t err = launch_rows_inst<T, F, F, 1, 8, 3, false, Pair64, 2, -1, OutT>(q);
                if (err != cudaSuccess) return err;
            }
            RowConv t = p;
            t.c_lo = p.C / kBN * kBN;
            return rem <= 16 ? launch_rows_inst<T, F, F, 1, 8, 3, false, Pair64, 2, -1, OutT, 4>(t)
                             : launch_rows_inst<T, F, F, 1, 8, 3, false, Pair64, 2, -1, OutT, 2>(t);
        }
    }
    return launch_rows_inst<T, F, F, 1, 8, 3, false, Pair64, 2, -1, OutT>(p);
}

template <typename T, class OutT = float>
cudaError_t launch_rows_s2_dispatch(const RowConv& p) {
    if (p.FH != p.FW || p.flip) return cudaErrorNotSupported;
    switch (p.FH) {
        case 3: return launch_rows_s2_square<T, 3, OutT>(p);
        case 5: return launch_rows_s2_square<T, 5, OutT>(p);
        case 7: return launch_rows_s2_square<T, 7, OutT>(p);
        case 9: return launch_rows_s2_square<T, 9, OutT>(p);
        case 11: return launch_rows_s2_square<T, 11, OutT>(p);
        case 13: return launch_rows_s2_square<T, 13, OutT>(p);
        default: return cudaErrorNotSupported;
    }
}

// BN + Act + forward DWC (filters of 3, 5 and 7 taps, stride 1 or 2) on the tiles of the
// plain forward kernels.
template <int F>
struct BnActTile {
    static constexpr int R = RowsTile<F, F>::R;
    static constexpr int TM = RowsTile<F, F>::TM;
    static constexpr int MINB = RowsTile<F, F>::MINB;
};

template <typename T, int SD, int F, int ACT>
cudaError_t launch_rows_bnact_inst(const RowConv& p) {
    if constexpr (SD == 1)
        return launch_rows_inst<T, F, F, BnActTile<F>::R, BnActTile<F>::TM, BnActTile<F>::MINB,
                                false, Pair64, 1, ACT>(p);
    else
        return launch_rows_inst<T, F, F, 1, 8, 3, false, Pair64, 2, ACT>(p);
}

template <typename T, int SD, int F>
cudaError_t launch_rows_bnact_act(const RowConv& p) {
    switch (p.act) {
        case 0: return launch_rows_bnact_inst<T, SD, F, 0>(p);
        case 1: return launch_rows_bnact_inst<T, SD, F, 1>(p);
        case 2: return launch_rows_bnact_inst<T, SD, F, 2>(p);
        default: return cudaErrorNotSupported;
    }
}

template <typename T, int SD>
cudaError_t launch_rows_bnact_dispatch(const RowConv& p) {
    if (p.FH != p.FW || p.flip || p.bn_mean == nullptr) return cudaErrorNotSupported;
    switch (p.FH) {
        case 3: return launch_rows_bnact_act<T, SD, 3>(p);
        case 5: return launch_rows_bnact_act<T, SD, 5>(p);
        case 7: return launch_rows_bnact_act<T, SD, 7>(p);
        default: return cudaErrorNotSupported;
    }
}

// Stripe (non-square) filters: any filter height, odd widths 1..51, one output row per lane
// with the filter height read at run time.  Narrow filters take 16 outputs per lane (more
// taps per staged value), the others the tiles of the large square filters.
template <int FW>
struct StripeTile {
    static constexpr int TM = FW <= 7 ? 16 : 14;
    static constexpr int MINB = FW <= 7 ? 3 : (FW <= 31 ? 2 : 1);
};

template <typename T, int FW>
cudaError_t launch_rows_stripe_inst(const RowConv& p) {
    using St = StripeTile<FW>;
    return p.flip ? launch_rows_inst<T, 0, FW, 1, St::TM, St::MINB, true>(p)
                  : launch_rows_inst<T, 0, FW, 1, St::TM, St::MINB, false>(p);
}

#define DWC_STRIPE_WIDTHS(X) X(1) X(3) X(5) X(7) X(9) X(11) X(13) X(15) X(17) X(19) X(21) X(23) \
    X(25) X(27) X(29) X(31) X(33) X(35) X(37) X(39) X(41) X(43) X(45) X(47) X(49) X(51)

template <typename T>
cudaError_t launch_rows_stripe_dispatch(const RowConv& p) {
    if (p.FH == p.FW || p.FH < 1 || p.out_dtype != kF32) return cudaErrorNotSupported;
    switch (p.FW) {
#define DWC_STRIPE_CASE(F) \
    case F:                \
        return launch_rows_stripe_inst<T, F>(p);
        DWC_STRIPE_WIDTHS(DWC_STRIPE_CASE)
#undef DWC_STRIPE_CASE
        default:
            return cudaErrorNotSupported;
    }
}

}  // namespace dwc
