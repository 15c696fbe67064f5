// dwc_fgrad.cuh -- filter-gradient kernel ("backward filter convolution").
//
//   dw[fh, fw, c] = sum_{n, oh, ow} x[n, S*oh + fh - pad, S*ow + fw - pad, c] * dy[n, oh, ow, c]
//
// with stride S = 1, or S = 2 for square filters of 3, 5 or 7 taps.
// ("Flash-DWC: Making Depthwise Convolution Compute-Efficient on GPUs", §5.1: the output is
// only FH x FW x C and does not grow with batch or resolution, so the work is spread over
// the accumulation axis N*OH*OW.)  GB300 restatement:
//  * The accumulation axis (flattened output rows n*OH + oh) is cut into Z slices; a CTA
//    owns one slice, one block of 64 channels and one chunk of FHC filter rows.  Z is chosen
//    from the SM count so that the grid fills the GPU.
//  * Instead of the pages' fp32 atomics, every CTA writes its partial gradient to its own
//    slot of a workspace [Z][FH][FW][C]; a second kernel sums the Z slots in a fixed order.
//    Within a CTA the column strips of the warps are summed in a fixed order through shared
//    memory.  Results are therefore bit-identical from run to run.
//  * A producer warp streams, with TMA, the dy rows of the slice and the x rows they pair
//    with.  The x rows form a window of FHC rows that slides by S rows per output row, so
//    every x row enters shared memory once per CTA (at S = 2 with a one-row window, the
//    rows between two windows are skipped).
//  * Each compute warp owns RF filter rows and one strip of output columns; a lane owns two
//    channels and keeps RF x FW fp32x2 accumulators plus, per owned row, a circular register
//    window of U >= FW x values (the FW that the current output column multiplies and the
//    next ones).  Each dy element is loaded once and used for RF*FW packed FMAs.  At S = 2
//    the output column ow meets the x columns 2*ow + t: even taps t = 2j read the even
//    column 2*(ow + j), odd taps t = 2j + 1 the odd column 2*(ow + j) + 1, so each row keeps
//    two circular windows (even and odd columns) that advance by one column per output
//    column.
#pragma once

#include <type_traits>

#include "dwc_rows.cuh"

namespace dwc {

// Filter rows per warp (RF: accumulators + x windows take about 4*RF*FW registers), the
// CTAs per SM the shared-memory window is sized for (MINB) and the period U of the circular
// x window (any U >= FW works; output columns are processed in blocks of U, so a U that
// divides the row width leaves no padded columns).
template <int FH, int FW, int RF_ = 0, int MINB_ = 0, int U_ = 0, int NY_ = 0, int SD_ = 1,
          int FWC_ = 0, int MAXCW_ = 0, int ROT_ = 0>
struct FgradTile {
    // convolution stride (1, or 2 for the strided 3x3 / 5x5 / 7x7 filter gradient)
    static constexpr int SD = SD_;
    // taps of a filter row one warp owns (FWC) and the chunks a row is cut into (NFC): past
    // 31 taps a whole row's accumulators and window no longer fit in registers, so each
    // warp takes a chunk of consecutive taps (x read from the chunk's first tap on)
    static constexpr int FWC = FWC_ > 0 ? FWC_ : FW;
    static constexpr int NFC = (FW + FWC - 1) / FWC;
    static_assert(SD == 1 || FWC == FW, "strided tiles keep whole filter rows");
    // x columns one output column of one parity class needs (FWC at stride 1; at stride 2
    // the even taps read the even columns and the odd taps the odd ones)
    static constexpr int KW = (FWC + SD - 1) / SD;
    // dy ring slots, also the x rows staged ahead of the window: deeper for small filters,
    // whose rows are consumed fastest (timed: 4 up to 5 taps, 3 for 7, else 2)
    static constexpr int NY = NY_ > 0 ? NY_ : (FW <= 5 ? 4 : (FW == 7 ? 3 : 2));
    // rows per warp timed fastest on the stage shapes: 2 for 7x7, 1 for 5x5, 9x9 and
    // 11x11, else what about 120 registers hold
    static constexpr int kFit = FH == 7 ? 2 : ((FH == 5 || FH == 9 || FH == 11) ? 1 : 120 / (4 * FWC));
    static constexpr int RF = RF_ > 0 ? RF_ : (kFit < 1 ? 1 : ((FH > 0 && kFit > FH) ? FH : kFit));
    static constexpr int MINB = MINB_ > 0 ? MINB_ : 1;
    static constexpr int U = U_ > 0 ? U_ : (SD == 1 ? FWC : (KW <= 4 ? 4 : KW));
    static_assert(U >= KW, "the window must hold the columns one output column needs");
    // compute warps per CTA where the registers leave room for more (the launch bound caps
    // registers at 128 per thread for 13 warps, 168 for 12), else 8
    // (7x7 at stride 1, two rows per warp: 12 warps timed 2.5 % faster than 8 on 56x56x128)
    static constexpr int MAXCW = MAXCW_ > 0 ? MAXCW_ :
        ((RF == 1 && FWC <= 19) || (FW == 7 && RF == 2 && SD == 1) ? 12 : ((RF == 1 && FWC <= 27) ? 11 : 8));
    // Rotated layout (ROT_ = 1, 7x7 at stride 1): 7 filter rows at two rows per warp make
    // four row groups, the last with one live row (whose warps compute only that row).
    // With 16 compute warps (the four groups x four column strips of equal width) the warps
    // of a strip take the groups in a rotated order, so that each of the SM's four
    // schedulers (warp w issues on scheduler w mod 4) holds one warp of every group and the
    // same number of packed FMAs.
    static constexpr bool ROT = ROT_ != 0 && SD == 1 && RF == 2 && FWC == FW && FH == 7;
    // compute warps the launch bound allows
    static constexpr int MAXW = ROT ? 16 : MAXCW;
};

template <int F>
using FgradRotTile = FgradTile<F, F, 0, 0, 0, 0, 1, 0, 0, 1>;

// A second window period per filter width: a multiple of 7 (the widths of the usual
// 224-pixel pyramids, 112/56/28/14/7, are multiples of 7) at least FW, where the longer
// register window does not spill (none for 15 and 29..31).
template <int FW>
struct FgradAltPeriod {
    static constexpr int U = FW <= 3 ? 4 : (FW <= 7 ? 7 : (FW <= 13 ? 14 :
                             (FW == 15 ? 15 : (FW <= 27 ? 28 : FW))));
};

// (the default tile itself where the second period equals FW, so nothing is built twice)
template <int F>
using FgradAltTile = typename std::conditional<FgradAltPeriod<F>::U == F, FgradTile<F, F>,
                                               FgradTile<F, F, 0, 0, FgradAltPeriod<F>::U>>::type;

// The alternative period runs when it pads the row to fewer columns than blocks of FW do.
template <int FW>
bool fgrad_use_alt_period(int OW) {
    constexpr int UA = FgradAltPeriod<FW>::U;
    if (UA == FW) return false;
    return (OW + UA - 1) / UA * UA < (OW + FW - 1) / FW * FW;
}

struct FgradArgs {
    float* part;           // [Z * ncp][FH][FW][C] partial sums
    unsigned int* status;
    int N, OH, C, pad;
    int c_lo;              // first channel of the launch's channel blocks
    int FH;                // filter rows (the template's, or any for a stripe tile, FH = 0)
    int ncp, owpart;       // column parts of a row, output columns per part
    int nwf, nwc;          // compute warps: filter-row groups x column strips
    int fhc, chunks, cblocks, Z;
    int rows_per_slice;    // flattened output rows per slice
    int nblocks, bps;      // U-wide column blocks per row, blocks per strip
    int nx, ny;            // ring slots for x rows and dy rows
    uint32_t x_bytes, y_bytes;   // ring slot strides (multiples of 128 bytes)
    uint32_t x_tx, y_tx;         // bytes one TMA box writes into a slot
    uint32_t y_off;        // byte offset of the dy ring after the x ring
    unsigned long long wait_ns;  // limit of every mbarrier wait
};

// One output row of a column strip at stride 2: acc[f][t] += x[2*ow + t] * dy[ow] over the
// strip's output columns, for the RF x rows xs[f].  Even taps t = 2j read the even x column
// 2*(ow + j), odd taps t = 2j + 1 the odd column 2*(ow + j) + 1; each class has its own
// circular window (x column 2m or 2m + 1 sits in slot m mod U).
template <typename T, int FW, int RF, int U>
__device__ __forceinline__ void fgrad_row_s2(float2 (&acc)[RF][FW], const T* const (&xs)[RF],
                                             const T* ys, int blk0, int blk1) {
    constexpr int KE = (FW + 1) / 2;  // even taps
    constexpr int KO = FW / 2;        // odd taps
    float2 we[RF][U], wo[RF][U];
    const int c0 = blk0 * U;
#pragma unroll
    for (int f = 0; f < RF; ++f) {
#pragma unroll
        for (int m = 0; m < KE - 1; ++m) we[f][m] = Elem<T>::load_pair(xs[f] + 2 * (c0 + m) * kBN);
#pragma unroll
        for (int m = 0; m < KO - 1; ++m) wo[f][m] = Elem<T>::load_pair(xs[f] + (2 * (c0 + m) + 1) * kBN);
    }
#pragma unroll 1
    for (int blk = blk0; blk < blk1; ++blk) {
        const int cb0 = blk * U;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float2 g = Elem<T>::load_pair(ys + (cb0 + u) * kBN);
#pragma unroll
            for (int f = 0; f < RF; ++f) {
                we[f][(u + KE - 1) % U] = Elem<T>::load_pair(xs[f] + 2 * (cb0 + u + KE - 1) * kBN);
                if constexpr (KO > 0)
                    wo[f][(u + KO - 1) % U] = Elem<T>::load_pair(xs[f] + (2 * (cb0 + u + KO - 1) + 1) * kBN);
#pragma unroll
                for (int j = 0; j < KE; ++j) fma2(acc[f][2 * j], we[f][(u + j) % U], g);
#pragma unroll
                for (int j = 0; j < KO; ++j) fma2(acc[f][2 * j + 1], wo[f][(u + j) % U], g);
            }
        }
    }
}

// One output row of a column strip at stride 1, for the first R of the RF rows xs[f]:
// acc[f][t] += x[ow + t] * dy[ow] over the strip's output columns (ow from blk0 * U to
// blk1 * U).  Column c of the padded x row sits in slot c mod U of a circular register window.
template <typename T, int FC, int RF, int R, int U, int PITCH>
__device__ __forceinline__ void fgrad_row_s1(float2 (&acc)[RF][FC], const T* const (&xs)[RF],
                                             const T* ys, int blk0, int blk1) {
    float2 win[R][U];
    const int c0 = blk0 * U;
#pragma unroll
    for (int f = 0; f < R; ++f)
#pragma unroll
        for (int m = 0; m < FC - 1; ++m) win[f][m] = Elem<T>::load_pair(xs[f] + (c0 + m) * PITCH);
#pragma unroll 1
    for (int blk = blk0; blk < blk1; ++blk) {
        const int cb0 = blk * U;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float2 g = Elem<T>::load_pair(ys + (cb0 + u) * PITCH);
#pragma unroll
            for (int f = 0; f < R; ++f) {
                win[f][(u + FC - 1) % U] = Elem<T>::load_pair(xs[f] + (cb0 + u + FC - 1) * PITCH);
#pragma unroll
                for (int t = 0; t < FC; ++t) fma2(acc[f][t], win[f][(u + t) % U], g);
            }
        }
    }
}

// G: lane groups (1, or 2 / 4 when all channels fit in 32 / 16: each group of 32 / G lanes
// covers them for its own column strip, so no lane idles).
template <typename T, int FH, int FW, class Tile = FgradTile<FH, FW>, int G = 1>
__global__ void __launch_bounds__((Tile::MAXW + 1) * 32, Tile::MINB)
fgrad_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
             const FgradArgs a) {
    constexpr int RF = Tile::RF;
    constexpr int U = Tile::U;
    constexpr int SD = Tile::SD;
    constexpr int FC = Tile::FWC;
    constexpr int NFC = Tile::NFC;
    static_assert(G == 1 || (SD == 1 && (G == 2 || G == 4)), "lane groups at stride 1");
    constexpr int PITCH = kBN / G;   // channels per staged pixel
    constexpr int LPG = 32 / G;      // lanes per group
    extern __shared__ __align__(128) unsigned char smem[];
    // the slice sum may be scheduled now (it waits for this grid); a programmatic dependent
    // of the kernel before it, this grid touches no global memory before that one finished
    pdl_trigger();
    pdl_wait();
    uint64_t* xfull = reinterpret_cast<uint64_t*>(smem);
    uint64_t* xempty = xfull + a.nx;
    uint64_t* yfull = xempty + a.nx;
    uint64_t* yempty = yfull + a.ny;
    unsigned char* xring = smem + 512;
    unsigned char* yring = xring + a.y_off;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ncompute = a.nwf * NFC * a.nwc;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.nx; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], ncompute);
        }
        for (int s = 0; s < a.ny; ++s) {
            mbar_init(&yfull[s], 1);
            mbar_init(&yempty[s], ncompute);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // CTA -> (slice z, channel block cb, filter-row chunk); chunks of one slice are adjacent
    // so that they read the same rows out of L2.
    int b = blockIdx.x;
    const int chunk = b % a.chunks; b /= a.chunks;
    const int cb = b % a.cblocks; b /= a.cblocks;
    const int cp = b % a.ncp; b /= a.ncp;   // column part: output columns cp*owpart + [0, owpart)
    const int z = b;
    const int ow_base = cp * a.owpart;
    const int fh0 = chunk * a.fhc;
    const long long total_rows = static_cast<long long>(a.N) * a.OH;
    const long long q0 = static_cast<long long>(z) * a.rows_per_slice;
    const long long q1 = std::min<long long>(q0 + a.rows_per_slice, total_rows);
    // x rows each output row adds to the window (and drops from it afterwards)
    const int nnew = SD == 1 ? 1 : std::min(SD, a.fhc);

    // ---------------- producer ----------------------------------------------------------
    if (warp == ncompute) {
        if (lane != 0) return;
        prefetch_tensormap(&xmap);
        prefetch_tensormap(&ymap);
        Ring xr, yr;
        uint32_t xissued = 0, yissued = 0;  // saturating counts, compared with the ring sizes
        bool ok = true;
        auto put_x = [&](int n, int ih) -> bool {
            if (xissued >= static_cast<uint32_t>(a.nx) && !mbar_wait(&xempty[xr.slot], xr.phase ^ 1u, a.wait_ns))
                return false;
            if (xissued < static_cast<uint32_t>(a.nx)) ++xissued;
            mbar_arrive_expect_tx(&xfull[xr.slot], a.x_tx);
            tma_load_4d(xring + static_cast<size_t>(xr.slot) * a.x_bytes, &xmap, &xfull[xr.slot],
                        a.c_lo + cb * PITCH, ow_base * SD - a.pad, ih, n);
            xr.next(a.nx);
            return true;
        };
        auto put_y = [&](int n, int oh) -> bool {
            if (yissued >= static_cast<uint32_t>(a.ny) && !mbar_wait(&yempty[yr.slot], yr.phase ^ 1u, a.wait_ns))
                return false;
            if (yissued < static_cast<uint32_t>(a.ny)) ++yissued;
            mbar_arrive_expect_tx(&yfull[yr.slot], a.y_tx);
            tma_load_4d(yring + static_cast<size_t>(yr.slot) * a.y_bytes, &ymap, &yfull[yr.slot],
                        a.c_lo + cb * PITCH, ow_base, oh, n);
            yr.next(a.ny);
            return true;
        };
        for (long long q = q0; q < q1 && ok;) {
            const int n = static_cast<int>(q / a.OH);
            const int oha = static_cast<int>(q % a.OH);
            const int ohb = static_cast<int>(std::min<long long>(q1 - static_cast<long long>(n) * a.OH, a.OH));
            // output row oh reads the x rows ih0 + SD*(oh - oha) + [0, fhc)
            const int ih0 = oha * SD + fh0 - a.pad;
            for (int r = 0; r < a.fhc - nnew && ok; ++r) ok = put_x(n, ih0 + r);
            for (int oh = oha; oh < ohb && ok; ++oh) {
                const int ihn = ih0 + (oh - oha) * SD + a.fhc - nnew;
                for (int r = 0; r < nnew && ok; ++r) ok = put_x(n, ihn + r);
                if (ok) ok = put_y(n, oh);
            }
            q = static_cast<long long>(n) * a.OH + ohb;
        }
        if (!ok) record_status(a.status, DWC_DEVSTAT_TIMEOUT);
        // drain: the copies still outstanding in both rings must land before the CTA exits
        auto drain = [&](Ring r, uint32_t issued, uint32_t n, uint64_t* full) {
            for (uint32_t j = 0; j < issued; ++j) {
                r.slot = r.slot == 0 ? n - 1 : r.slot - 1;
                if (r.slot == n - 1) r.phase ^= 1u;
                if (!mbar_wait(&full[r.slot], r.phase, a.wait_ns)) {
                    record_status(a.status, DWC_DEVSTAT_TIMEOUT);
                    return;
                }
            }
        };
        drain(xr, xissued, a.nx, xfull);
        drain(yr, yissued, a.ny, yfull);
        return;
    }

    // ---------------- compute warps -----------------------------------------------------
    static_assert(!Tile::ROT || G == 1, "the rotated layout has no lane groups");
    // (rotated layout: warp w -> strip w / 4, row group (w + strip) mod 4)
    const int wc = Tile::ROT ? warp >> 2 : warp / (a.nwf * NFC);
    const int wf = Tile::ROT ? (warp + wc) & 3 : warp % a.nwf;
    const int fc = Tile::ROT ? 0 : (warp / a.nwf) % NFC;  // tap chunk: taps fc*FC .. fc*FC + FC - 1
    const int lg = lane / LPG;                     // lane group: column strip wc * G + lg
    const int cl = lane % LPG;                     // channel pair
    const int frow0 = wf * RF;                     // first owned row within the chunk
    const int blk0 = (wc * G + lg) * a.bps;
    const int blk1 = std::min(blk0 + a.bps, a.nblocks);

    float2 acc[RF][FC];
#pragma unroll
    for (int f = 0; f < RF; ++f)
#pragma unroll
        for (int t = 0; t < FC; ++t) acc[f][t] = make_float2(0.f, 0.f);

    const int fhn = FH > 0 ? FH : a.FH;
    bool live[RF];
#pragma unroll
    for (int f = 0; f < RF; ++f) live[f] = (frow0 + f < a.fhc) && (fh0 + frow0 + f < fhn);

    Ring xbase, yr;  // oldest x row of the current window; current dy row
    bool ok = true;
    // slot and parity of the x row `d` rows after the window base (d < nx)
    auto xslot = [&](uint32_t d, uint32_t& phase) -> uint32_t {
        uint32_t s = xbase.slot + d;
        phase = xbase.phase;
        if (s >= static_cast<uint32_t>(a.nx)) {
            s -= a.nx;
            phase ^= 1u;
        }
        return s;
    };
    for (long long q = q0; q < q1 && ok;) {
        const int n = static_cast<int>(q / a.OH);
        const int oha = static_cast<int>(q % a.OH);
        const int ohb = static_cast<int>(std::min<long long>(q1 - static_cast<long long>(n) * a.OH, a.OH));
        const int L = ohb - oha;
        for (int row = 0; row < L && ok; ++row) {
            // wait for the x rows this output row needs (the whole window at the segment start)
            for (int d = (row == 0 ? 0 : a.fhc - nnew); d < a.fhc; ++d) {
                uint32_t ph;
                const uint32_t sl = xslot(static_cast<uint32_t>(d), ph);
                if (!mbar_wait(&xfull[sl], ph, a.wait_ns)) {
                    ok = false;
                    break;
                }
            }
            if (ok && !mbar_wait(&yfull[yr.slot], yr.phase, a.wait_ns)) ok = false;
            if (!ok) break;

            const T* ys = reinterpret_cast<const T*>(yring + static_cast<size_t>(yr.slot) * a.y_bytes) + 2 * cl;
            const T* xs[RF];
#pragma unroll
            for (int f = 0; f < RF; ++f) {
                uint32_t ph;
                const uint32_t sl = xslot(static_cast<uint32_t>(frow0 + f), ph);
                xs[f] = reinterpret_cast<const T*>(xring + static_cast<size_t>(sl) * a.x_bytes) +
                        2 * cl + fc * FC * PITCH;
            }
            if constexpr (SD == 2) {
                if (blk0 < blk1) fgrad_row_s2<T, FC, RF, U>(acc, xs, ys, blk0, blk1);
            } else if constexpr (Tile::ROT) {
                // the last group (one live row of two) computes its live row only
                if (!live[RF - 1])
                    fgrad_row_s1<T, FC, RF, 1, U, PITCH>(acc, xs, ys, blk0, blk1);
                else
                    fgrad_row_s1<T, FC, RF, RF, U, PITCH>(acc, xs, ys, blk0, blk1);
            } else if (blk0 < blk1) {
                // circular window: column c of the padded x row sits in slot c mod U
                float2 win[RF][U];
                const int c0 = blk0 * U;
#pragma unroll
                for (int f = 0; f < RF; ++f)
#pragma unroll
                    for (int m = 0; m < FC - 1; ++m)
                        win[f][m] = Elem<T>::load_pair(xs[f] + (c0 + m) * PITCH);
#pragma unroll 1
                for (int blk = blk0; blk < blk1; ++blk) {
                    const int cb0 = blk * U;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const float2 g = Elem<T>::load_pair(ys + (cb0 + u) * PITCH);
#pragma unroll
                        for (int f = 0; f < RF; ++f) {
                            // a row past the filter's last row (last chunk) computes from its
                            // staged window row like the others and is never written: no
                            // branch in this loop
                            win[f][(u + FC - 1) % U] = Elem<T>::load_pair(xs[f] + (cb0 + u + FC - 1) * PITCH);
#pragma unroll
                            for (int t = 0; t < FC; ++t) fma2(acc[f][t], win[f][(u + t) % U], g);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&yempty[yr.slot]);
            yr.next(a.ny);
            // the nnew oldest rows have no later use
            for (int d = 0; d < nnew; ++d) {
                if (lane == 0) mbar_arrive(&xempty[xbase.slot]);
                xbase.next(a.nx);
            }
        }
        if (!ok) break;
        // the last fhc-nnew rows of the window are not needed by later output rows
        __syncwarp();
        for (int d = 0; d < a.fhc - nnew; ++d) {
            if (lane == 0) mbar_arrive(&xempty[xbase.slot]);
            xbase.next(a.nx);
        }
        q = static_cast<long long>(n) * a.OH + ohb;
    }
    // A warp that gave up still goes through the two CTA barriers below, so that no
    // compute warp can wait on them forever; the status word reports the failure.
    if (!ok) record_status(a.status, DWC_DEVSTAT_TIMEOUT);

    // ---- fixed-order sum over the column strips, through shared memory ----------------
    // All ring copies have landed (every stage was waited on), so the ring is reused.
    asm volatile("bar.sync 1, %0;" ::"r"(ncompute * 32) : "memory");
    float2* red = reinterpret_cast<float2*>(xring);
    // layout: [wc][wf][fc][f][t][lane]
    const size_t per_warp = static_cast<size_t>(RF) * FC * 32;
    const size_t wslot = static_cast<size_t>(a.nwf) * NFC;   // warps of one column strip
    float2* mine = red + (static_cast<size_t>(wc) * wslot + wf * NFC + fc) * per_warp;
#pragma unroll
    for (int f = 0; f < RF; ++f)
#pragma unroll
        for (int t = 0; t < FC; ++t) mine[(f * FC + t) * 32 + lane] = acc[f][t];
    asm volatile("bar.sync 1, %0;" ::"r"(ncompute * 32) : "memory");
    if (wc == 0 && lg == 0) {
        const int c = a.c_lo + cb * PITCH + 2 * cl;
        for (int f = 0; f < RF; ++f) {
            const int fh = fh0 + frow0 + f;
            if (!live[f] || c >= a.C) continue;
            for (int t = 0; t < FC; ++t) {
                const int fw = fc * FC + t;
                if (fw >= FW) break;
                // column strips in a fixed order: warp strips k, lane groups g within
                const size_t off = static_cast<size_t>(wf * NFC + fc) * per_warp + (f * FC + t) * 32 + cl;
                float2 s = make_float2(0.f, 0.f);
                for (int k = 0; k < a.nwc; ++k) {
                    for (int g = 0; g < G; ++g) {
                        const float2 v = red[static_cast<size_t>(k) * wslot * per_warp + off + g * LPG];
                        s.x += v.x;
                        s.y += v.y;
                    }
                }
                float* dst = a.part + ((static_cast<size_t>(z * a.ncp + cp) * fhn + fh) * FW + fw) * a.C + c;
                *reinterpret_cast<float2*>(dst) = s;
            }
        }
    }
}

template <int FH, int FW, class Tile = FgradTile<FH, FW>>
struct FgradPlan {
    int nwf, nwc, fhc, chunks, cblocks, Z, rows_per_slice, nblocks, bps, nx, ny;
    uint32_t x_bytes, y_bytes, y_off;
    uint32_t x_tx, y_tx;   // bytes of one x / dy TMA box (the slots are these rounded to 128)
    size_t smem;
    int pwx, owp;
    int ncp, owpart;   // column parts per row and output columns per part
};

// One candidate launch shape: the row cut into ncp column parts (one CTA each), with the
// deepest lookahead between min_la output rows and the tile's that fits.
template <typename T, int FH, int FW, class Tile, int G = 1>
bool fgrad_plan_parts(int N, int OH, int OW, int C, int ncp, int min_la,
                      FgradPlan<FH, FW, Tile>& P, int fhr) {
    constexpr int PITCH = kBN / G;
    const int e = static_cast<int>(sizeof(T));
    constexpr int RF = Tile::RF;
    const DeviceInfo& dev = device_info();
    const size_t smem_cap = std::min<size_t>(dev.max_smem_optin, 233472 / Tile::MINB - 1024);
    P.ncp = ncp;
    P.owpart = (OW + ncp - 1) / ncp;
    P.nblocks = (P.owpart + Tile::U - 1) / Tile::U;
    P.owpart = P.nblocks * Tile::U;
    P.owp = P.nblocks * Tile::U;
    // (the last tap chunk may run past the filter's last tap: its x columns are staged too)
    P.pwx = Tile::SD * (P.owp - 1) + Tile::NFC * Tile::FWC;
    if (P.pwx > 256) return false;
    // TMA writes shared memory at 128-byte aligned addresses: ring slots are rounded up
    P.x_tx = static_cast<uint32_t>(P.pwx * PITCH * e);
    P.y_tx = static_cast<uint32_t>(P.owp * PITCH * e);
    P.x_bytes = (P.x_tx + 127u) & ~127u;
    P.y_bytes = (P.y_tx + 127u) & ~127u;
    // Filter-row groups per CTA (nwf, one warp each) and column strips (nwc): the x window of
    // nwf*RF rows must fit in shared memory; among the fitting choices take the one with the
    // most useful warp slots, counting warps up to 12 (about what hides the latencies of one
    // CTA per SM), discounted by the chunk count (each chunk streams every x and dy row of
    // its slice again); the weights were fitted to timings of the stage shapes.
    const int groups = (fhr + RF - 1) / RF;  // RF-row groups needed to cover the filter
    // The lookahead (dy slots, and the x rows staged ahead of the window) is Tile::NY
    // output rows, or the deepest down to min_la that fits.
    double best = -1.0;
    P.nwf = 0;
    int best_la = 0;
    constexpr int NFC = Tile::NFC;
    if constexpr (Tile::ROT) {
        // The rotated layout, or no plan: the whole filter in one chunk of four groups and
        // the row's blocks in four equal strips of at least two blocks (strips of one block,
        // 28-wide rows, timed slower than the default tile's eight warps of two blocks).
        static_assert(G == 1, "the rotated layout has no lane groups");
        if (fhr != FH || ncp != 1 || P.nblocks % 4 != 0 || P.nblocks < 8) return false;
        if (512 + static_cast<size_t>(16) * RF * Tile::FWC * 32 * sizeof(float2) > smem_cap) return false;
        int la = Tile::NY;
        auto need = [&](int l) {
            return 512 + static_cast<size_t>(4 * RF + l) * P.x_bytes + static_cast<size_t>(l) * P.y_bytes;
        };
        while (la > min_la && need(la) > smem_cap) --la;
        if (need(la) > smem_cap) return false;
        P.nwf = 4;
        P.nwc = 4;
        P.bps = P.nblocks / 4;
        best_la = la;
    }
    for (int nwf = Tile::ROT ? 0 : std::min(groups, Tile::MAXCW / NFC); nwf >= 1; --nwf) {
        int la = Tile::NY;
        auto need = [&](int l) {
            return 512 + static_cast<size_t>(nwf * RF + l * Tile::SD) * P.x_bytes +
                   static_cast<size_t>(l) * P.y_bytes;
        };
        while (la > min_la && need(la) > smem_cap) --la;
        if (need(la) > smem_cap) continue;
        const int chunks = (groups + nwf - 1) / nwf;
        if ((groups + chunks - 1) / chunks != nwf) continue;  // same chunks, fewer warps: seen
        // column strips: G per warp (lane groups)
        const int nwc0 = std::max(1, std::min(Tile::MAXCW / (nwf * NFC), (P.nblocks + G - 1) / G));
        const int bps = (P.nblocks + nwc0 * G - 1) / (nwc0 * G);
        const int nwc = (P.nblocks + bps * G - 1) / (bps * G);
        // the strip sums at the end reuse the ring: [nwc][nwf][NFC][RF][FWC][32] float2
        if (512 + static_cast<size_t>(nwc) * nwf * NFC * RF * Tile::FWC * 32 * sizeof(float2) > smem_cap)
            continue;
        const double useful = static_cast<double>(groups) / (chunks * nwf) *
                              static_cast<double>(P.nblocks) / (nwc * G * bps);
        const double score = useful * std::min(nwf * NFC * nwc, 12) / (1.0 + 0.2 * chunks);
        if (score > best * (1.0 + 1e-9)) {
            best = score;
            P.nwf = nwf;
            P.nwc = nwc;
            P.bps = bps;
            best_la = la;
        }
    }
    if (P.nwf < 1) return false;
    P.fhc = P.nwf * RF;
    P.ny = best_la;
    P.nx = P.fhc + best_la * Tile::SD;
    P.smem = 512 + static_cast<size_t>(P.nx) * P.x_bytes + static_cast<size_t>(P.ny) * P.y_bytes;
    P.chunks = (fhr + P.fhc - 1) / P.fhc;
    // strip reduction buffer reuses the ring
    const size_t red = static_cast<size_t>(P.nwc) * P.nwf * NFC * RF * Tile::FWC * 32 * sizeof(float2);
    if (red > P.smem - 512) P.smem = 512 + red;
    P.y_off = static_cast<uint32_t>(P.nx) * P.x_bytes;
    P.cblocks = (C + PITCH - 1) / PITCH;
    const long long rows = static_cast<long long>(N) * OH;
    const long long per_z = static_cast<long long>(P.cblocks) * P.chunks * P.ncp;
    // One wave: every CTA runs the same number of rows, so a grid a few CTAs larger than
    // the resident capacity would take a second wave for those few; round down.  For
    // filters up to 5 taps the capacity counts every CTA that shared memory, threads and
    // registers let an SM hold (measured faster there); larger filters keep one CTA per SM
    // (more, shorter slices measured slower from 7 taps on).
    static const int regs = kernel_regs(fgrad_kernel<T, FH, FW, Tile, G>, 224);
    const int ctas_per_sm = FW <= 5 ? std::max(Tile::MINB, resident_ctas(P.smem, (P.nwf * NFC * P.nwc + 1) * 32, regs))
                                    : Tile::MINB;
    long long Z = static_cast<long long>(dev.sm_count) * ctas_per_sm / per_z;
    Z = std::max<long long>(1, std::min<long long>(Z, rows));
    P.rows_per_slice = static_cast<int>((rows + Z - 1) / Z);
    P.Z = static_cast<int>((rows + P.rows_per_slice - 1) / P.rows_per_slice);
    return true;
}

// Shapes of the launch for one problem (shared by the workspace query and the launch).  A
// whole row per CTA with the tile's lookahead where it fits (stride 2: the deepest lookahead
// that fits); otherwise a lookahead of at least two rows, then of one (two rows with fewer
// filter rows per CTA timed faster than one row with more: 7x7 on 64x112x112x64, 177 against
// 233 us), then the row cut into 2, 3 or 4 column parts (rows too wide for shared memory or
// for one 256-column TMA box), each part a CTA of its own with its own partial-sum slot.
template <typename T, int FH, int FW, class Tile = FgradTile<FH, FW>, int G = 1>
bool fgrad_plan(int N, int OH, int OW, int C, FgradPlan<FH, FW, Tile>& P, int fhr = FH) {
    if (fhr < 1) return false;
    for (int ncp = 1; ncp <= 4; ++ncp) {
        if (ncp > 1 && (OW + ncp - 1) / ncp < Tile::U) break;
        if constexpr (Tile::SD > 1) {
            if (fgrad_plan_parts<T, FH, FW, Tile, G>(N, OH, OW, C, ncp, 1, P, fhr)) return true;
        } else {
            for (int min_la : {Tile::NY, 2, 1})
                if (min_la <= Tile::NY &&
                    fgrad_plan_parts<T, FH, FW, Tile, G>(N, OH, OW, C, ncp, min_la, P, fhr))
                    return true;
        }
    }
    return false;
}

// The kernel launch of plan P over the channel blocks from channel c_lo (its partial sums go
// to the workspace slices; the caller sums them).
template <typename T, int FH, int FW, class Tile, int G>
cudaError_t fgrad_enqueue(const FilterGrad& p, const FgradPlan<FH, FW, Tile>& P, int fhr, int c_lo) {
    const int e = static_cast<int>(sizeof(T));
    constexpr int PITCH = kBN / G;
    CUtensorMap xmap, ymap;
    {
        const cuuint64_t dims[4] = {(cuuint64_t)p.C, (cuuint64_t)p.W, (cuuint64_t)p.H, (cuuint64_t)p.N};
        const cuuint64_t strides[3] = {(cuuint64_t)p.C * e, (cuuint64_t)p.W * p.C * e,
                                       (cuuint64_t)p.H * p.W * p.C * e};
        const cuuint32_t box[4] = {(cuuint32_t)PITCH, (cuuint32_t)P.pwx, 1u, 1u};
        if (encode_tiled(&xmap, Elem<T>::kTmaType, 4, const_cast<void*>(p.x), dims, strides, box) !=
            CUDA_SUCCESS)
            return cudaErrorNotSupported;
    }
    {
        const cuuint64_t dims[4] = {(cuuint64_t)p.C, (cuuint64_t)p.OW, (cuuint64_t)p.OH, (cuuint64_t)p.N};
        const cuuint64_t strides[3] = {(cuuint64_t)p.C * e, (cuuint64_t)p.OW * p.C * e,
                                       (cuuint64_t)p.OH * p.OW * p.C * e};
        const cuuint32_t box[4] = {(cuuint32_t)PITCH, (cuuint32_t)P.owp, 1u, 1u};
        if (encode_tiled(&ymap, Elem<T>::kTmaType, 4, const_cast<void*>(p.dy), dims, strides, box) !=
            CUDA_SUCCESS)
            return cudaErrorNotSupported;
    }
    FgradArgs a;
    a.part = p.workspace;
    a.status = p.status;
    a.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    a.N = p.N; a.OH = p.OH; a.C = p.C; a.pad = p.pad;
    a.c_lo = c_lo;
    a.ncp = P.ncp; a.owpart = P.owpart;
    a.FH = fhr;
    a.nwf = P.nwf; a.nwc = P.nwc; a.fhc = P.fhc; a.chunks = P.chunks; a.cblocks = P.cblocks;
    a.Z = P.Z; a.rows_per_slice = P.rows_per_slice; a.nblocks = P.nblocks; a.bps = P.bps;
    a.nx = P.nx; a.ny = P.ny; a.x_bytes = P.x_bytes; a.y_bytes = P.y_bytes; a.y_off = P.y_off;
    a.x_tx = P.x_tx; a.y_tx = P.y_tx;

    auto kern = fgrad_kernel<T, FH, FW, Tile, G>;
    static DeviceOnce smem_opt_in;
    {
        const cudaError_t err = opt_in_smem(kern, smem_opt_in, device_info().max_smem_optin);
        if (err != cudaSuccess) return err;
    }
    const int threads = (P.nwf * Tile::NFC * P.nwc + 1) * 32;
    const unsigned grid = static_cast<unsigned>(P.Z) * P.ncp * P.cblocks * P.chunks;
    return launch_pdl(kern, dim3(grid), dim3(threads), P.smem, p.stream, xmap, ymap, a);
}

template <typename T, int FH, int FW, class Tile = FgradTile<FH, FW>, int G = 1>
cudaError_t launch_fgrad_inst(const FilterGrad& p) {
    FgradPlan<FH, FW, Tile> P;
    const int fhr = FH > 0 ? FH : p.FH;
    if (!fgrad_plan<T, FH, FW, Tile, G>(p.N, p.OH, p.OW, p.C, P, fhr)) return cudaErrorNotSupported;
    if (p.N == 0 || p.OH == 0 || p.OW == 0) {
        return cudaMemsetAsync(p.dw, 0, sizeof(float) * fhr * FW * p.C, p.stream);
    }
    const size_t need = static_cast<size_t>(P.Z) * P.ncp * fhr * FW * p.C;
    if (p.workspace_floats < need || p.workspace == nullptr) return cudaErrorInvalidValue;
    const cudaError_t err = fgrad_enqueue<T, FH, FW, Tile, G>(p, P, fhr, 0);
    if (err != cudaSuccess) return err;
    return launch_reduce_slices(p.workspace, P.Z * P.ncp, static_cast<size_t>(fhr) * FW * p.C, p.dw,
                                p.stream);
}

template <typename T, int FH, int FW, class Tile = FgradTile<FH, FW>, int G = 1>
size_t fgrad_workspace_inst(int N, int OH, int OW, int C, int fhr = FH) {
    FgradPlan<FH, FW, Tile> P;
    if (!fgrad_plan<T, FH, FW, Tile, G>(N, OH, OW, C, P, fhr)) return 0;
    return static_cast<size_t>(P.Z) * P.ncp * fhr * FW * static_cast<size_t>(C);
}

// 3x3, 5x5 and 7x7 with at most 32 (16) channels: 2 (4) lane groups, so that the single
// partial channel block does not leave half the lanes idle.  (A tail of at most 32 channels
// past a multiple of 64 as a second launch on lane groups, sharing the first launch's slices,
// was slower at 7x7 -- 64x56x56: 96 channels 88 against 84 us for 128, 160 channels 131
// against 115 for 192 -- since every launch pays the kernel's fixed costs: the blocks of a
// tail stay in the one launch.)
// 7x7 takes the rotated layout wherever it has a plan.
template <typename T, int F, class Tile>
cudaError_t launch_fgrad_grouped(const FilterGrad& p) {
    if constexpr (F <= 7) {
        if (p.C <= 16) return launch_fgrad_inst<T, F, F, Tile, 4>(p);
        if (p.C <= 32) return launch_fgrad_inst<T, F, F, Tile, 2>(p);
    }
    if constexpr (FgradRotTile<F>::ROT) {
        FgradPlan<F, F, FgradRotTile<F>> P;
        if (fgrad_plan<T, F, F, FgradRotTile<F>>(p.N, p.OH, p.OW, p.C, P))
            return launch_fgrad_inst<T, F, F, FgradRotTile<F>>(p);
    }
    return launch_fgrad_inst<T, F, F, Tile>(p);
}

template <typename T, int F, class Tile>
size_t fgrad_workspace_grouped(int N, int OH, int OW, int C) {
    if constexpr (F <= 7) {
        if (C <= 16) return fgrad_workspace_inst<T, F, F, Tile, 4>(N, OH, OW, C);
        if (C <= 32) return fgrad_workspace_inst<T, F, F, Tile, 2>(N, OH, OW, C);
    }
    if constexpr (FgradRotTile<F>::ROT) {
        const size_t rot = fgrad_workspace_inst<T, F, F, FgradRotTile<F>>(N, OH, OW, C);
        if (rot > 0) return rot;
    }
    return fgrad_workspace_inst<T, F, F, Tile>(N, OH, OW, C);
}

// Workspace of the launch that launch_fgrad_dispatch makes for this problem.
template <typename T, int F>
size_t fgrad_workspace_dispatch(int N, int OH, int OW, int C) {
    return fgrad_use_alt_period<F>(OW) ? fgrad_workspace_grouped<T, F, FgradAltTile<F>>(N, OH, OW, C)
                                       : fgrad_workspace_grouped<T, F, FgradTile<F, F>>(N, OH, OW, C);
}

#define DWC_FGRAD_FILTERS(X) X(3) X(5) X(7) X(9) X(11) X(13) X(15) X(17) X(19) X(21) X(23) X(25) X(27) X(29) X(31)
#define DWC_FGRAD_BIG_FILTERS(X) X(33) X(35) X(37) X(39) X(41) X(43) X(45) X(47) X(49) X(51)

// 33..51 taps: each filter row in two chunks of (F + 1) / 2 taps, one warp each; window
// period the chunk width, or 28 (a multiple of 7) where that pads the row less.
template <int F>
using FgradBigTile = FgradTile<F, F, 0, 0, 0, 0, 1, (F + 1) / 2>;
template <int F>
using FgradBigAltTile = FgradTile<F, F, 0, 0, 28, 0, 1, (F + 1) / 2>;

template <int F>
bool fgrad_big_use_alt(int OW) {
    constexpr int UD = (F + 1) / 2;
    return (OW + 27) / 28 * 28 < (OW + UD - 1) / UD * UD;
}

// Workspace floats of the CUDA-core filter gradient for inputs of type T.
template <typename T>
size_t fgrad_workspace_t(int N, int OH, int OW, int C, int FH, int FW) {
    if (FH != FW) return 0;
    switch (FH) {
#define DWC_FGRAD_WS(F) \
    case F:             \
        return fgrad_workspace_dispatch<T, F>(N, OH, OW, C);
        DWC_FGRAD_FILTERS(DWC_FGRAD_WS)
#undef DWC_FGRAD_WS
#define DWC_FGRAD_BIG_WS(F)                                                              \
    case F:                                                                              \
        return fgrad_big_use_alt<F>(OW) ? fgrad_workspace_inst<T, F, F, FgradBigAltTile<F>>(N, OH, OW, C) \
                                        : fgrad_workspace_inst<T, F, F, FgradBigTile<F>>(N, OH, OW, C);
        DWC_FGRAD_BIG_FILTERS(DWC_FGRAD_BIG_WS)
#undef DWC_FGRAD_BIG_WS
        default:
            return 0;
    }
}


// Stride-2 filter gradient: square filters of 3 to 13 taps.
template <int F>
using FgradS2Tile = FgradTile<F, F, 0, 0, 0, 0, 2>;

template <typename T>
cudaError_t launch_fgrad_s2_dispatch(const FilterGrad& p) {
    if (p.FH != p.FW) return cudaErrorNotSupported;
    switch (p.FH) {
        case 3: return launch_fgrad_inst<T, 3, 3, FgradS2Tile<3>>(p);
        case 5: return launch_fgrad_inst<T, 5, 5, FgradS2Tile<5>>(p);
        case 7: return launch_fgrad_inst<T, 7, 7, FgradS2Tile<7>>(p);
        case 9: return launch_fgrad_inst<T, 9, 9, FgradS2Tile<9>>(p);
        case 11: return launch_fgrad_inst<T, 11, 11, FgradS2Tile<11>>(p);
        case 13: return launch_fgrad_inst<T, 13, 13, FgradS2Tile<13>>(p);
        default: return cudaErrorNotSupported;
    }
}

template <typename T>
size_t fgrad_s2_workspace_t(int N, int OH, int OW, int C, int FH, int FW) {
    if (FH != FW) return 0;
    switch (FH) {
        case 3: return fgrad_workspace_inst<T, 3, 3, FgradS2Tile<3>>(N, OH, OW, C);
        case 5: return fgrad_workspace_inst<T, 5, 5, FgradS2Tile<5>>(N, OH, OW, C);
        case 7: return fgrad_workspace_inst<T, 7, 7, FgradS2Tile<7>>(N, OH, OW, C);
        case 9: return fgrad_workspace_inst<T, 9, 9, FgradS2Tile<9>>(N, OH, OW, C);
        case 11: return fgrad_workspace_inst<T, 11, 11, FgradS2Tile<11>>(N, OH, OW, C);
        case 13: return fgrad_workspace_inst<T, 13, 13, FgradS2Tile<13>>(N, OH, OW, C);
        default: return 0;
    }
}

template <typename T>
cudaError_t launch_fgrad_dispatch(const FilterGrad& p) {
    if (p.FH != p.FW) return cudaErrorNotSupported;
    switch (p.FH) {
#define DWC_FGRAD_CASE(F)                                          \
    case F:                                                        \
        return fgrad_use_alt_period<F>(p.OW)                       \
                   ? launch_fgrad_grouped<T, F, FgradAltTile<F>>(p) \
                   : launch_fgrad_grouped<T, F, FgradTile<F, F>>(p);
        DWC_FGRAD_FILTERS(DWC_FGRAD_CASE)
#undef DWC_FGRAD_CASE
#define DWC_FGRAD_BIG_CASE(F)                                             \
    case F:                                                               \
        return fgrad_big_use_alt<F>(p.OW)                                 \
                   ? launch_fgrad_inst<T, F, F, FgradBigAltTile<F>>(p)     \
                   : launch_fgrad_inst<T, F, F, FgradBigTile<F>>(p);
        DWC_FGRAD_BIG_FILTERS(DWC_FGRAD_BIG_CASE)
#undef DWC_FGRAD_BIG_CASE
        default:
            return cudaErrorNotSupported;
    }
}

// Stripe (non-square) filters: the filter height read at run time, one filter row per warp,
// odd widths 1..51 (past 31 taps in two chunks), window period a multiple of 7 of at least 4.
template <int FW>
struct FgradStripe {
    static constexpr int FWC = FW > 31 ? (FW + 1) / 2 : FW;
    static constexpr int U = FWC <= 3 ? 4 : (FWC <= 7 ? 7 : (FWC <= 14 ? 14 : (FWC <= 28 ? 28 : FWC)));
    using Tile = FgradTile<0, FW, 1, 0, U, 0, 1, (FW > 31 ? FWC : 0)>;
};

template <typename T>
cudaError_t launch_fgrad_stripe_dispatch(const FilterGrad& p) {
    if (p.FH == p.FW) return cudaErrorNotSupported;
    switch (p.FW) {
#define DWC_FGRAD_STRIPE_CASE(F) \
    case F:                      \
        return launch_fgrad_inst<T, 0, F, typename FgradStripe<F>::Tile>(p);
        DWC_STRIPE_WIDTHS(DWC_FGRAD_STRIPE_CASE)
#undef DWC_FGRAD_STRIPE_CASE
        default:
            return cudaErrorNotSupported;
    }
}

template <typename T>
size_t fgrad_stripe_workspace_t(int N, int OH, int OW, int C, int FH, int FW) {
    if (FH == FW || FH < 1 || FH > 255) return 0;
    switch (FW) {
#define DWC_FGRAD_STRIPE_WS(F) \
    case F:                    \
        return fgrad_workspace_inst<T, 0, F, typename FgradStripe<F>::Tile>(N, OH, OW, C, FH);
        DWC_STRIPE_WIDTHS(DWC_FGRAD_STRIPE_WS)
#undef DWC_FGRAD_STRIPE_WS
        default:
            return 0;
    }
}

}  // namespace dwc
