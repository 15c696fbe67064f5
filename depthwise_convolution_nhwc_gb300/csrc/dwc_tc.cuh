// dwc_tc.cuh -- forward / backward-data kernel on the 5th-generation tensor cores (tcgen05
// MMA, accumulators in tensor memory) for 16-bit inputs (bf16, fp16), fp32 accumulation.
//
// The GEMV -> GEMM transformation of "Flash-DWC: Making Depthwise Convolution
// Compute-Efficient on GPUs", §4.2-§4.4, re-derived for a 128-row MMA whose operands come
// straight from shared memory through matrix descriptors:
//
//   for one channel and one filter row fh, a tile of 128 output rows x N output columns is
//     D[m, n] += sum_k A_fh[m, k] * T_fh[k, n]
//   A_fh[m, k] = x[row(m) + fh, col0 + k]        (the staged input rows, shifted by fh)
//   T_fh[k, n] = filt(fh, k - n) if 0 <= k - n < FW else 0   (Toeplitz of the filter row)
//   with K = N + FW - 1 rounded up to 16; summing over fh gives the 2-D convolution.
//
// Both operands are stored once and read through descriptors, without duplication:
//  * A: one channel's input rows in the K-major core-matrix layout without swizzle, i.e.
//    "planes" of 8 input columns, each plane a column of 16-byte rows.  Consecutive output
//    rows are 16 bytes apart, so the shift by fh is just a start address 16*fh bytes later.
//  * T: a Toeplitz matrix is constant along its diagonals.  With the output columns taken in
//    reverse order (n' = N-1-n) every 8x8 core matrix depends only on the sum of its block
//    indices, so the whole matrix is N/8 + K/8 - 1 distinct core matrices laid end to end
//    (a "run"), and a descriptor with both strides 128 bytes reads every block of the K x N
//    matrix.  The epilogue undoes the reversal.
//  * Rows of the tile run through several images: image n occupies the S rows starting at
//    virtual row n*S (S = image rows + padding shared with the next image), so one 128-row
//    MMA covers, for example, two 56-row images; rows in the gaps are computed and dropped.
//
// Paired filter rows.  An MMA's time is set by reading its operands from shared memory (A's
// 4 KB and T's N x 32 bytes at 128 bytes a clock) and a floor of ~46 cycles, so narrow MMAs
// cost nearly as much as wide ones.  One MMA of N = 2 N' takes the Toeplitz matrices of filter
// rows 2p and 2p+1 side by side against the same A (input rows shifted by 2p):
//    D[m, (0, n)] = sum_p A_2p[m] T_2p    the even filter rows of output row m,
//    D[m, (1, n)] = sum_p A_2p[m] T_2p+1  the odd filter rows of output row m - 1,
// so output row m is D[m, (0, .)] + D[m+1, (1, .)]: A is read once for two filter rows (for
// N' = 32, one N=64 MMA of 48 cycles instead of two N=32 ones of 46).  A tile then owns 127
// rows; the epilogue takes the odd part from the next lane (a shuffle, and at the three
// warp boundaries of the tile the next warp's first lane through shared memory).  The two
// runs are interleaved core matrix by core matrix, so a descriptor with a K-direction stride
// of 256 bytes and an N-direction stride of 128 reads both halves.  An odd last filter row is
// paired with zeros.  Column tiles of up to 32 outputs keep a unit's 4 channels in 256
// accumulator columns (two buffers).
//
// Two launches.  A preparation kernel writes, into scratch memory of the call,
//  * the input as per-channel planes in the layout above, plane-major: for each channel and
//    8-column plane all the virtual rows (the images' rows stacked, zero rows between
//    images) lie contiguously, and the columns are padded so that every tile's first column
//    falls on an 8-column boundary -- one bulk copy of a contiguous band then fills one
//    8-column plane of a unit, with no gather and no transposition in the main kernel (a
//    row-major copy read by tensor-map boxes of 16-byte rows moved one row per clock);
//  * every Toeplitz run (channel, filter row), rotated by 180 degrees for backward data.
// The main kernel then only moves data with the copy engines: bulk copies for the planes
// and for the runs.  Gathering and transposing inside it (one cache line per
// pixel and channel group, and shuffles to build the runs) tied up the load/store and
// shared-memory pipes that the MMA issuers and their barriers also go through.
//
// Warp roles per CTA (one CTA per SM, persistent over units of (row tile, column tile, group
// of CG = 2 or 4 channels)):
//  * 4 epilogue warps -- warp w reads the 32-lane quadrant w of the accumulators
//    (tcgen05.ld) and writes the CG channels of a pixel with 16-byte stores;
//  * 4 MMA warps: one lane each issues the MMAs of every fourth channel of the group, or,
//    in groups of 2 channels, of one channel's even or odd filter rows into a partial sum of
//    its own (a single thread issues an MMA only every ~100 cycles, an M=128 N=64 MMA takes
//    48); the first also allocates the tensor memory;
//  * 4 run feeders: one lane each copies, in order, the runs of its issuer's items into
//    that issuer's ring;
//  * 1 plane feeder: lane b copies plane b of each of the units' channels into the plane ring.
// Stages pass through mbarrier rings; every wait has a time limit and a shared abort flag,
// so a lost arrival ends the kernel (status word set) instead of hanging it.
#pragma once

#include <algorithm>
#include <type_traits>

#include "dwc_device.cuh"
#include "dwc_host.h"

namespace dwc {

constexpr int kTcM = 128;           // MMA rows (tensor-memory lanes)
// Roles (13 warps; warp w runs on sub-partition w % 4):
//   0-3   epilogue, warp w reading the 32-lane quadrant w of tensor memory
//   4-7   MMA issuers, one lane each: issuer i takes the channels c with c % 4 == i, every
//         filter row of them (groups of 2 channels: channel i / 2, the filter rows of
//         parity i % 2); warp 4 also allocates the tensor memory
//   8-11  run feeders, feeder i filling issuer i's ring
//   12    plane feeder
constexpr int kTcEpiWarps = 4;
constexpr int kTcMmaWarp = 4;       // first MMA warp
constexpr int kTcIssuers = 4;       // MMA-issuing threads (one per MMA warp)
constexpr int kTcFeed0 = kTcMmaWarp + kTcIssuers;
constexpr int kTcPlaneWarp = kTcFeed0 + kTcIssuers;
constexpr int kTcWarps = kTcPlaneWarp + 1;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcRingSlots = 4;     // most run slots per issuer ring (a power of two)
constexpr int kTcRunsPerSlot = 4;   // most filter rows per ring item (runs per slot)
constexpr int kTcTmemCols = 512;
constexpr int kTcDCols = 256;       // columns of one accumulator buffer (two buffers)
constexpr int kTcMaxPlanes = 16;
constexpr int kTcMaxToep = kTcIssuers * kTcRingSlots;
constexpr int kTcMaxBox = 256;      // most staged rows per plane
// barriers (plane and run rings, two accumulator buffers, the final MMA barriers, the
// epilogue warps' exchange of paired rows), the tensor-memory address and the abort flag
constexpr int kTcBarBytes =
    ((2 * kTcMaxPlanes + 2 * kTcMaxToep + 2 * 2 + kTcIssuers + 2 * kTcEpiWarps * 2) * 8 + 8 + 127) /
    128 * 128;
// paired rows: per epilogue warp and accumulator buffer, its first lane's odd-row sums of 4
// channels x up to 32 columns
constexpr int kTcXFloats = 128;
constexpr int kTcXBytes = kTcEpiWarps * 2 * kTcXFloats * 4;

struct TcArgs {
    const unsigned char* planes; // plane-major stacked copy [C][np][vp rows][8 columns], 16-bit
    const unsigned char* zeros;  // MR * 16 zero bytes (planes outside the copy)
    const unsigned char* runs;   // Toeplitz runs [C][FHI][(pair + 1) * NCM core matrices], 16-bit
    void* out;          // N x OH x OW x C, OutT
    unsigned int* status;
    unsigned long long wait_ns;
    int N, C, OH, OW, FH;
    int pair;           // 1: filter rows in pairs (N = 2 NN per MMA), 0: one row per MMA
    int FHI;            // MMA rows of filters per channel: FH, or ceil(FH / 2) in pairs
    int mrows;          // output rows a row tile owns: 128, or 127 in pairs
    int S;              // virtual rows per image
    int kimg;           // images per row tile (0: tiles are 128-row bands of one image)
    int bands;          // row tiles per image when kimg == 0
    int NN;             // output columns of a column tile's accumulator (multiple of 16; in
                        // pairs a multiple of 8 up to 32, the MMA's N being 2 NN)
    int TWc;            // output columns a column tile owns (<= NN, multiple of 8)
    int KS;             // K-steps of 16
    int MR;             // staged rows per plane (>= FH + 127, multiple of 8, <= 256)
    int NCM;            // core matrices of one run: NN/8 + 2*KS - 1
    int x0;             // column of the stacked copy holding input column -pad_w (<= 0)
    int cbase;          // first channel of the launch's groups
    int ncg;            // channel groups of the launch
    int ps;             // plane ring slots
    int rps;            // filter rows per ring item (1 .. kTcRunsPerSlot)
    int rslots, rshift; // slots per run ring (4, or 2 for items of 3 or 4 rows) and its log2
    uint32_t units, col_tiles;
    int np;             // planes of the stacked copy
    uint32_t vp;        // rows of a plane (the V virtual rows, then zero rows)
    FastDiv fd_S;
    uint32_t plane_bytes, toep_bytes;   // one plane; one run (a pair of runs in pairs)
    uint32_t off_toep, off_bar, off_x;  // byte offsets in shared memory
    uint32_t idesc;     // instruction descriptor (kind::f16, fp32 accumulation)
};

// ------------------------------------------------------------------ tcgen05 wrappers

// Shared-memory matrix descriptor: start address, leading (K-direction) and stride
// (M/N-direction) byte offsets between 8x16-byte core matrices, no swizzle.
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version of sm_100-family MMAs
    return d;
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns of tensor memory (lane = thread of the warp).
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// The same, 8 columns.
__device__ __forceinline__ void tc_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
}
// The same, 4 columns.
__device__ __forceinline__ void tc_ld4(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
__device__ __forceinline__ void tc_ld(uint32_t taddr, uint32_t (&r)[16]) { tc_ld16(taddr, r); }
__device__ __forceinline__ void tc_ld(uint32_t taddr, uint32_t (&r)[8]) { tc_ld8(taddr, r); }
__device__ __forceinline__ void tc_ld(uint32_t taddr, uint32_t (&r)[4]) { tc_ld4(taddr, r); }

__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bulk copy of `bytes` contiguous bytes (16-byte aligned, a multiple of 16) from global to
// shared memory, completion counted on `bar`.
__device__ __forceinline__ void tc_bulk_load(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bounded wait that also gives up as soon as another role has aborted the CTA.  On running
// out of time it records the timeout and raises the abort flag itself.  Between polls the
// warp sleeps, up to `max_sleep_ns`: the warps that wait most of the time (epilogue,
// feeders) then leave the issue slots of their sub-partition to the issuers.
template <class Args>
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, const Args& a,
                                        volatile int* abort_flag, uint32_t max_sleep_ns = 32) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    uint32_t sleep_ns = 8;
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (global_ns() - t0 > a.wait_ns) {
            *abort_flag = 1;
            record_status(a.status, DWC_DEVSTAT_TIMEOUT);
            return false;
        }
        __nanosleep(sleep_ns);
        if (sleep_ns < max_sleep_ns) sleep_ns *= 2;
    }
    return true;
}

// The same wait by every lane of a warp, with one outcome for the whole warp (a warp that
// goes on runs warp-collective instructions, so no lane may have given up alone).
template <class Args>
__device__ __forceinline__ bool tc_wait_warp(uint64_t* bar, uint32_t parity, const Args& a,
                                             volatile int* abort_flag, uint32_t max_sleep_ns = 32) {
    return __all_sync(0xffffffffu, tc_wait(bar, parity, a, abort_flag, max_sleep_ns));
}

// A feeder never leaves with copies in flight: after its last fill it waits (bounded, even
// after an abort) for the fills still open in each of its `slots` ring slots, the fills
// `count - slots` .. `count - 1` (earlier fills completed before their slot was refilled).
template <class Args>
__device__ __forceinline__ void tc_drain(uint64_t* full, uint32_t first_slot, uint32_t slots,
                                         uint32_t count, const Args& a) {
    for (uint32_t k = count >= slots ? count - slots : 0; k < count; ++k)
        if (!mbar_wait(&full[first_slot + k % slots], (k / slots) & 1u, a.wait_ns)) {
            record_status(a.status, DWC_DEVSTAT_TIMEOUT);
            return;
        }
}

// Row tile `t`: first virtual output row v0 and the rows [v_lo, v_hi) the tile owns (tiles of
// one image's rows are mrows apart).
struct TcTile {
    int v0, v_lo, v_hi;
};
__device__ __forceinline__ TcTile tc_tile(const TcArgs& a, int t) {
    TcTile r;
    if (a.kimg > 0) {
        const int n0 = t * a.kimg;
        r.v0 = n0 * a.S;
        r.v_lo = r.v0;
        r.v_hi = min(a.N, n0 + a.kimg) * a.S;
    } else {
        const int n = t / a.bands, b = t - n * a.bands;
        r.v0 = n * a.S + a.mrows * b;
        r.v_lo = r.v0;
        r.v_hi = n * a.S + min(a.OH, a.mrows * (b + 1));
    }
    return r;
}

// Unit u -> (row tile, column tile, channel group); the channel group is fastest, so CTAs
// running at the same time read neighbouring planes of the stacked copy from L2.
__device__ __forceinline__ void tc_unit(const TcArgs& a, uint32_t u, int& t, int& j, int& g) {
    g = static_cast<int>(u % static_cast<uint32_t>(a.ncg));
    const uint32_t q = u / static_cast<uint32_t>(a.ncg);
    j = static_cast<int>(q % a.col_tiles);
    t = static_cast<int>(q / a.col_tiles);
}

// The CG channels of one output pixel, one or two 16-byte streaming stores (fp32), or one
// 8- or 16-byte store of values rounded to nearest even (bf16, fp16).
template <class OutT, int CG>
__device__ __forceinline__ void tc_store_pixel(OutT* dst, const float (&v)[CG]) {
    if constexpr (std::is_same<OutT, float>::value && CG == 2) {
        __stcs(reinterpret_cast<float2*>(dst), make_float2(v[0], v[1]));
    } else if constexpr (std::is_same<OutT, float>::value) {
#pragma unroll
        for (int c = 0; c < CG; c += 4)
            __stcs(reinterpret_cast<float4*>(dst + c), make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]));
    } else {
        uint32_t h[CG / 2];
#pragma unroll
        for (int c = 0; c < CG; c += 2) {
            if constexpr (std::is_same<OutT, __nv_bfloat16>::value) {
                const __nv_bfloat162 b = __float22bfloat162_rn(make_float2(v[c], v[c + 1]));
                h[c / 2] = *reinterpret_cast<const uint32_t*>(&b);
            } else {
                const __half2 b = __float22half2_rn(make_float2(v[c], v[c + 1]));
                h[c / 2] = *reinterpret_cast<const uint32_t*>(&b);
            }
        }
        if constexpr (CG == 2) {
            __stcs(reinterpret_cast<uint32_t*>(dst), h[0]);
        } else if constexpr (CG == 4) {
            __stcs(reinterpret_cast<uint2*>(dst), make_uint2(h[0], h[1]));
        } else {
            __stcs(reinterpret_cast<uint4*>(dst), make_uint4(h[0], h[1], h[2], h[3]));
        }
    }
}

// ------------------------------------------------------------------ plane-major stacked copy

// Plane-major stacked copy of `src` (nn x h x w x C, 16-bit):
//   dst[c][p][ro + v][e] = src[n][v % S - pad_h][8 p + e - lp][c],  n = v / S,  zero outside,
// for planes p < wp / 8 and plane rows ro + v in [0, vp) (zero rows before and after the
// V = nn * S virtual rows).  A tile is 16 virtual rows x one plane x
// CT channels: pixels are read as 16-byte pieces of 8 channels (whole 128-byte lines for 64
// channels), and every thread writes the 8 columns of one channel and row as 16 bytes,
// consecutive threads along the rows of a plane.
struct TcStackArgs {
    const void* src;
    void* dst;
    int nn, h, w, C, pad_h, S, lp, np;   // np: planes (wp / 8)
    int V, ro, vp;      // virtual rows; zero rows before them; rows of a plane
    int CT, piece_shift;
    int tiles;          // ceil(vp / 16) * np * (C / CT)
    FastDiv fd_np, fd_ct, fd_S;
};

constexpr int kStackRows = 16;
constexpr int kStackWords = 33;   // a (column, row) pixel's 64 channels as 32 words + 1 pad

// One tile of copy `a` (the block's threads; `tile` is the block's shared staging).
template <typename T>
__device__ __forceinline__ void tc_stack_tile(const TcStackArgs& a, int tt, uint32_t* tile) {
    const T* X = static_cast<const T*>(a.src);
    T* P = static_cast<T*>(a.dst);
    const int pieces = a.CT / 8;
    {
        uint32_t cb, pl;
        const uint32_t q = a.fd_ct.divmod(static_cast<uint32_t>(tt), cb);
        const int rb = static_cast<int>(a.fd_np.divmod(q, pl));
        const int c0 = a.CT * static_cast<int>(cb);
        const int v0 = rb * kStackRows;
        __syncthreads();   // the previous tile's reads are done
        for (int idx = threadIdx.x; idx < kStackRows * 8 * pieces; idx += blockDim.x) {
            const int i = idx >> a.piece_shift, j = idx - (i << a.piece_shift);
            const int r = i >> 3, e = i & 7;   // row of the tile, column of the plane
            const int v = v0 + r - a.ro;        // virtual row
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (v >= 0 && v < a.V) {
                uint32_t hr;
                const int n = static_cast<int>(a.fd_S.divmod(static_cast<uint32_t>(v), hr));
                const int hh = static_cast<int>(hr) - a.pad_h;
                const int col = 8 * static_cast<int>(pl) + e - a.lp;
                if (hh >= 0 && hh < a.h && col >= 0 && col < a.w)
                    val = __ldg(reinterpret_cast<const uint4*>(
                        X + ((static_cast<size_t>(n) * a.h + hh) * a.w + col) * a.C + c0 + 8 * j));
            }
            uint32_t* d = tile + (e * kStackRows + r) * kStackWords + 4 * j;
            d[0] = val.x; d[1] = val.y; d[2] = val.z; d[3] = val.w;
        }
        __syncthreads();
        // task (channel pair cp, row r): the pair's word of the plane's 8 columns
        for (int idx = threadIdx.x; idx < (a.CT / 2) * kStackRows; idx += blockDim.x) {
            const int r = idx & (kStackRows - 1), cp = idx >> 4;
            const int v = v0 + r;               // plane row
            if (v >= a.vp) continue;
            uint32_t wd[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) wd[e] = tile[(e * kStackRows + r) * kStackWords + cp];
            uint4 lo, hi;
            lo.x = __byte_perm(wd[0], wd[1], 0x5410); hi.x = __byte_perm(wd[0], wd[1], 0x7632);
            lo.y = __byte_perm(wd[2], wd[3], 0x5410); hi.y = __byte_perm(wd[2], wd[3], 0x7632);
            lo.z = __byte_perm(wd[4], wd[5], 0x5410); hi.z = __byte_perm(wd[4], wd[5], 0x7632);
            lo.w = __byte_perm(wd[6], wd[7], 0x5410); hi.w = __byte_perm(wd[6], wd[7], 0x7632);
            const size_t plane = static_cast<size_t>(a.vp) * 8;   // elements of one plane
            T* dst = P + (static_cast<size_t>(c0 + 2 * cp) * a.np + pl) * plane + static_cast<size_t>(v) * 8;
            *reinterpret_cast<uint4*>(dst) = lo;
            *reinterpret_cast<uint4*>(dst + static_cast<size_t>(a.np) * plane) = hi;
        }
    }
}

inline bool tc_stack_args(TcStackArgs& q, const void* src, void* dst, int nn, int h, int w, int C, int pad_h,
                          int S, int lp, int wp, int ro, int vp) {
    q.src = src; q.dst = dst;
    q.nn = nn; q.h = h; q.w = w; q.C = C; q.pad_h = pad_h; q.S = S; q.lp = lp; q.np = wp / 8;
    q.CT = C % 64 == 0 ? 64 : (C % 32 == 0 ? 32 : (C % 16 == 0 ? 16 : 8));
    q.piece_shift = q.CT == 64 ? 3 : (q.CT == 32 ? 2 : (q.CT == 16 ? 1 : 0));
    const long long V = static_cast<long long>(nn) * S;
    const long long tiles = (static_cast<long long>(vp) + kStackRows - 1) / kStackRows * q.np * (C / q.CT);
    if (V >= (1LL << 31) || tiles >= (1LL << 30)) return false;
    q.V = static_cast<int>(V);
    q.ro = ro;
    q.vp = vp;
    q.tiles = static_cast<int>(tiles);
    q.fd_np.init(static_cast<uint32_t>(q.np));
    q.fd_ct.init(static_cast<uint32_t>(C / q.CT));
    q.fd_S.init(static_cast<uint32_t>(S));
    return true;
}


// ------------------------------------------------------------------ preparation kernel

struct TcPrepArgs {
    TcStackArgs st;     // the plane-major stacked copy of the input
    const void* w;      // FH x FW x C, 16-bit
    void* runs;         // C x FHI runs of (pair + 1) * 8 * NCM rows of 8 values, 16-bit
    int C, FH, FW, NN, NCM;
    int FHI, pair;      // run items per channel; 1: two filter rows' runs interleaved
    int run_tasks;           // C * FHI * (pair + 1) * 8 * NCM: one 16-byte row of a run
    int run_blocks;          // blocks [0, run_blocks) write the runs, the rest the copy
    // divisions by launch constants (all operands below 2^31)
    FastDiv fd_C, fd_rows;
};

constexpr int kTcPrepThreads = 256;

template <typename T, bool FLIP>
__global__ void __launch_bounds__(kTcPrepThreads) tc_prep_kernel(const TcPrepArgs a) {
    pdl_trigger();   // the main kernel may be scheduled now (it waits for this grid)
    __shared__ uint32_t tile[8 * kStackRows * kStackWords];
    if (static_cast<int>(blockIdx.x) >= a.run_blocks) {
        // the plane-major stacked copy, tile by tile
        const int nb = static_cast<int>(gridDim.x) - a.run_blocks;
        for (int tt = static_cast<int>(blockIdx.x) - a.run_blocks; tt < a.st.tiles; tt += nb)
            tc_stack_tile<T>(a.st, tt, tile);
    } else {
        // Runs: row r of the run of (c, fh) holds z[r .. r+7], z[i] = filt(fh, i - (NN-1)),
        // zero outside the filter; filt is w, or w rotated by 180 degrees (backward data).
        // In pairs, item i holds the runs of filter rows 2i and 2i+1 (zeros past the filter)
        // interleaved by core matrix: core matrix 2d + h of the item is core matrix d of row
        // 2i + h.  The channel is the fastest task index, so a warp's tap loads are contiguous.
        const uint16_t* Wt = static_cast<const uint16_t*>(a.w);
        uint16_t* R = static_cast<uint16_t*>(a.runs);
        const int rows = 8 * a.NCM * (a.pair + 1);
        const int stride = a.run_blocks * static_cast<int>(blockDim.x);
        for (int task = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x); task < a.run_tasks;
             task += stride) {
            uint32_t cu, ru;
            const uint32_t q = a.fd_C.divmod(static_cast<uint32_t>(task), cu);
            const int fi = static_cast<int>(a.fd_rows.divmod(q, ru));
            const int c = static_cast<int>(cu);
            int r = static_cast<int>(ru), fh = fi;
            if (a.pair) {
                const int cm = r >> 3;
                fh = 2 * fi + (cm & 1);
                r = ((cm >> 1) << 3) | (r & 7);
            }
            uint4 o = make_uint4(0u, 0u, 0u, 0u);
            // rows r + 7 < NN - 1 or r > NN + FW - 2 hold no tap (most of a run): zeros, with no
            // tap computed (the test is uniform over a warp, whose lanes differ in c only)
            const int f0 = r - (a.NN - 1);
            if (fh < a.FH && f0 + 7 >= 0 && f0 < a.FW) {
                const int fhe = FLIP ? a.FH - 1 - fh : fh;
                const uint16_t* wrow = Wt + static_cast<size_t>(fhe) * a.FW * a.C + c;
                uint32_t z[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int f = f0 + e;
                    z[e] = (f >= 0 && f < a.FW) ? wrow[static_cast<size_t>(FLIP ? a.FW - 1 - f : f) * a.C] : 0u;
                }
                o.x = z[0] | (z[1] << 16);
                o.y = z[2] | (z[3] << 16);
                o.z = z[4] | (z[5] << 16);
                o.w = z[6] | (z[7] << 16);
            }
            *reinterpret_cast<uint4*>(R + ((static_cast<size_t>(c) * a.FHI + fi) * rows + ru) * 8) = o;
        }
    }
}

// ------------------------------------------------------------------ main kernel

template <typename T, class OutT, int CG, bool PAIR>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_rows_kernel(const TcArgs a) {
    // issuers per channel: 1 (each issuer owns whole channels), or 2 in groups of 2 channels
    // (filter-row parities into two partial sums, one filter row per ring item)
    constexpr int PART = CG >= kTcIssuers ? 1 : kTcIssuers / CG;
    static_assert(CG * PART % kTcIssuers == 0 && PART <= 2, "issuers divide the group's channels");
    // paired rows: 4 channels, one per issuer, 2 NN <= 64 accumulator columns each
    static_assert(!PAIR || CG == kTcIssuers, "paired rows take groups of 4 channels");
    constexpr int CH_STEP = kTcIssuers / PART;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* planes = smem;
    unsigned char* toep = smem + a.off_toep;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* plane_full = bars;
    uint64_t* plane_empty = plane_full + kTcMaxPlanes;
    uint64_t* toep_full = plane_empty + kTcMaxPlanes;
    uint64_t* toep_empty = toep_full + kTcMaxToep;
    uint64_t* d_full = toep_empty + kTcMaxToep;   // [2]
    uint64_t* d_empty = d_full + 2;               // [2]
    uint64_t* mma_done = d_empty + 2;             // [kTcIssuers]
    uint64_t* x_full = mma_done + kTcIssuers;     // [epilogue warp][channel pair]
    uint64_t* x_empty = x_full + 2 * kTcEpiWarps;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(x_empty + 2 * kTcEpiWarps);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.ps; ++s) {
            mbar_init(&plane_full[s], 1);    // the plane feeder (plus the copies' bytes)
            mbar_init(&plane_empty[s], PART);   // the issuers of its channel
        }
        for (int s = 0; s < kTcMaxToep; ++s) {
            mbar_init(&toep_full[s], 1);
            mbar_init(&toep_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&d_full[s], kTcIssuers);
            mbar_init(&d_empty[s], kTcEpiWarps);
        }
        for (int i = 0; i < kTcIssuers; ++i) mbar_init(&mma_done[i], 1);
        for (int i = 0; i < 2 * kTcEpiWarps; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // launched as a programmatic dependent of the preparation kernel: its stacked copy and
    // runs are complete and visible past this point
    pdl_wait();

    if (warp >= kTcMmaWarp && warp < kTcMmaWarp + kTcIssuers) {
        // ------------------------------------------------------------- MMA issue
        // Issuer `is` takes the channels c of the group with c % 4 == is, all filter rows; or
        // (PART 2) channel is / 2, the filter rows of parity is % 2.
        const int is = warp - kTcMmaWarp;
        const int par = is % PART;
        if (lane == 0) {
            uint32_t db = 0, dphase = 0;
            bool ok = true;
            // Descriptors are built once; the start-address field (bits 0-13, 16-byte units)
            // then advances by plain additions: a plane slot, a filter row (16 bytes; 32 for a
            // pair), a K-step (two planes of A, two core matrices of T; four of a pair), a run.
            const uint64_t adesc0 = tc_sdesc(smem_addr(planes), a.MR * 16u, 128u);
            const uint64_t bdesc0 = tc_sdesc(smem_addr(toep), PAIR ? 256u : 128u, 128u);
            const uint32_t a_row = PAIR ? 2u : 1u;     // A advance per item row
            const uint32_t b_ks = PAIR ? 32u : 16u;    // T advance per K-step
            const uint32_t a_ks = 2u * a.MR;           // A advance per K-step (16-byte units)
            const uint32_t a_slot = a.plane_bytes >> 4, b_run = a.toep_bytes >> 4;
            const uint32_t b_slot = static_cast<uint32_t>(a.rps) * b_run;
            const uint32_t idesc = a.idesc;
            const uint32_t ps = static_cast<uint32_t>(a.ps);
            // this issuer's ring: barrier slots is * kTcRingSlots + [0, rslots) and the shared
            // memory slots is * rslots + [0, rslots), filled in order with the runs of exactly
            // the (channel, filter rows) items it takes
            const uint32_t ring0 = static_cast<uint32_t>(is) * kTcRingSlots;
            const uint32_t rmask = static_cast<uint32_t>(a.rslots) - 1u;
            const uint32_t sring0 = static_cast<uint32_t>(is * a.rslots);
            uint32_t item = 0;
            uint32_t pos0 = 0;   // plane-ring position of the unit's first channel
            for (uint32_t u = blockIdx.x; u < a.units && ok; u += gridDim.x, pos0 += CG) {
                if (!tc_wait(&d_empty[db], dphase ^ 1u, a, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t dcol = tmem + db * kTcDCols;
                for (int ch = is / PART; ch < CG && ok; ch += CH_STEP) {
                    // channel ch of this unit sits at plane-ring position pos0 + ch (the
                    // plane feeder fills the ring in order; this issuer skips the others)
                    const uint32_t pos = pos0 + static_cast<uint32_t>(ch);
                    const uint32_t pslot = pos % ps, pphase = (pos / ps) & 1u;
                    if (!tc_wait(&plane_full[pslot], pphase, a, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ap = adesc0 + pslot * a_slot;
                    const uint32_t dch =
                        dcol + static_cast<uint32_t>(PAIR ? ch * 2 * a.NN : (par * CG + ch) * a.NN);
                    // item: filter rows (pairs of rows) fh0 .. fh0 + rps - 1 (fewer at the end),
                    // or (PART 2) filter row fh0 of this issuer's parity
                    for (int fh0 = par; fh0 < a.FHI; fh0 += PART * a.rps, ++item) {
                        const uint32_t slot = ring0 + (item & rmask);
                        const uint32_t phase = (item >> a.rshift) & 1u;
                        if (!tc_wait(&toep_full[slot], phase, a, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t sslot = sring0 + (item & rmask);
                        const int nr = min(a.rps, a.FHI - fh0);
                        for (int rr = 0; rr < nr; ++rr) {
                            uint64_t ad = ap + static_cast<uint32_t>(fh0 + rr) * a_row;
                            uint64_t bd = bdesc0 + sslot * b_slot + rr * b_run;
                            tc_mma(dch, ad, bd, idesc, (fh0 + rr) != par ? 1u : 0u);
                            for (int ks = 1; ks < a.KS; ++ks) {
                                ad += a_ks;
                                bd += b_ks;
                                tc_mma(dch, ad, bd, idesc, 1u);
                            }
                        }
                        tc_commit(&toep_empty[slot]);   // slot free once these MMAs finish
                    }
                    if (!ok) break;
                    tc_commit(&plane_empty[pslot]);
                }
                if (!ok) break;
                tc_commit(&d_full[db]);
                db ^= 1u;
                if (db == 0) dphase ^= 1u;
            }
            // every MMA issued has completed before the tensor memory is released
            tc_commit(&mma_done[is]);
            if (!mbar_wait(&mma_done[is], 0, a.wait_ns)) record_status(a.status, DWC_DEVSTAT_TIMEOUT);
        }
        __syncwarp();
    } else if (warp < kTcEpiWarps && PAIR) {
        // ------------------------------------------------------------- epilogue, paired rows
        // Output row m of the tile = D[m, even half] + D[m + 1, odd half].  Per unit, warps
        // 1-3 first publish their lane 0's odd halves (lane 31 of the warp before needs them),
        // then every warp sums its lanes' even halves and the next lanes' odd halves.
        const int quad = warp;
        const int m = quad * 32 + lane;
        float* xbuf = reinterpret_cast<float*>(smem + a.off_x);
        const uint32_t nn2 = 2u * static_cast<uint32_t>(a.NN);
        uint32_t db = 0, dphase = 0;
        for (uint32_t u = blockIdx.x; u < a.units; u += gridDim.x) {
            int t, j, g;
            tc_unit(a, u, t, j, g);
            if (!tc_wait_warp(&d_full[db], dphase, a, abort_flag, 1024)) break;
            tc_fence_after();
            const TcTile tl = tc_tile(a, t);
            const int v = tl.v0 + m;
            uint32_t rr;
            const int n = static_cast<int>(a.fd_S.divmod(static_cast<uint32_t>(v), rr));
            const int r = static_cast<int>(rr);
            const bool row_ok = m < a.mrows && v >= tl.v_lo && v < tl.v_hi && r < a.OH;
            const int ow0 = j * a.TWc;
            const int ow_end = min(a.OW, ow0 + a.TWc);
            const int c0 = a.cbase + g * CG;
            OutT* orow = static_cast<OutT*>(a.out) +
                         (static_cast<size_t>(row_ok ? n : 0) * a.OH + (row_ok ? r : 0)) *
                             static_cast<size_t>(a.OW) * a.C + c0;
            // columns of channel ch: ch * 2 NN + 16 b + 8 h + e, output column block b
            // (reversed), half h
            const uint32_t dbase = tmem + db * kTcDCols + (static_cast<uint32_t>(quad * 32) << 16);
            const int xs = quad * 2 + static_cast<int>(db);   // this warp's exchange slot
            if (quad > 0) {
                if (!tc_wait_warp(&x_empty[xs], dphase ^ 1u, a, abort_flag, 1024)) break;
                float* xb = xbuf + xs * kTcXFloats;
                for (int cb = 0; cb < a.NN; cb += 8) {
                    uint32_t h[CG][8];
#pragma unroll
                    for (int ch = 0; ch < CG; ++ch) tc_ld8(dbase + ch * nn2 + 2 * cb + 8, h[ch]);
                    tc_wait_ld();
                    if (lane == 0) {
#pragma unroll
                        for (int ch = 0; ch < CG; ++ch)
#pragma unroll
                            for (int e = 0; e < 8; ++e) xb[ch * a.NN + cb + e] = __uint_as_float(h[ch][e]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_full[xs]);
            }
            const int xn_slot = xs + 2;                      // the next warp's slot
            const float* xn = xbuf + (quad < kTcEpiWarps - 1 ? xn_slot : 0) * kTcXFloats;
            if (quad < kTcEpiWarps - 1 && !tc_wait_warp(&x_full[xn_slot], dphase, a, abort_flag, 1024))
                break;
            for (int cb = 0; cb < a.NN; cb += 8) {
                uint32_t d[CG][16];
#pragma unroll
                for (int ch = 0; ch < CG; ++ch) tc_ld16(dbase + ch * nn2 + 2 * cb, d[ch]);
                tc_wait_ld();
                float o[CG][8];
#pragma unroll
                for (int ch = 0; ch < CG; ++ch)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float nx = __shfl_down_sync(0xffffffffu, __uint_as_float(d[ch][8 + e]), 1);
                        if (lane == 31) nx = quad < kTcEpiWarps - 1 ? xn[ch * a.NN + cb + e] : 0.f;
                        o[ch][e] = __uint_as_float(d[ch][e]) + nx;
                    }
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int ow = ow0 + a.NN - 1 - (cb + e);   // reversed columns
                        if (ow < ow0 || ow >= ow_end) continue;
                        float vals[CG];
#pragma unroll
                        for (int ch = 0; ch < CG; ++ch) vals[ch] = o[ch][e];
                        tc_store_pixel<OutT, CG>(orow + static_cast<size_t>(ow) * a.C, vals);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (quad < kTcEpiWarps - 1) mbar_arrive(&x_empty[xn_slot]);
                mbar_arrive(&d_empty[db]);
            }
            db ^= 1u;
            if (db == 0) dphase ^= 1u;
        }
    } else if (warp < kTcEpiWarps) {
        // ------------------------------------------------------------- epilogue
        const int quad = warp;   // one warp per quadrant, every column
        const int m = quad * 32 + lane;   // accumulator row = tensor-memory lane
        uint32_t db = 0, dphase = 0;
        for (uint32_t u = blockIdx.x; u < a.units; u += gridDim.x) {
            int t, j, g;
            tc_unit(a, u, t, j, g);
            if (!tc_wait_warp(&d_full[db], dphase, a, abort_flag, 1024)) break;
            tc_fence_after();
            const TcTile tl = tc_tile(a, t);
            const int v = tl.v0 + m;
            uint32_t rr;
            const int n = static_cast<int>(a.fd_S.divmod(static_cast<uint32_t>(v), rr));
            const int r = static_cast<int>(rr);
            const bool row_ok = v >= tl.v_lo && v < tl.v_hi && r < a.OH;
            const int ow0 = j * a.TWc;
            const int ow_end = min(a.OW, ow0 + a.TWc);
            const int c0 = a.cbase + g * CG;
            OutT* orow = static_cast<OutT*>(a.out) +
                         (static_cast<size_t>(row_ok ? n : 0) * a.OH + (row_ok ? r : 0)) *
                             static_cast<size_t>(a.OW) * a.C + c0;
            const uint32_t dcol = tmem + db * kTcDCols + (static_cast<uint32_t>(quad * 32) << 16);
            // columns per round: CG x CW sums (of PART partials each) in registers (32 values)
            constexpr int CW = 32 / (CG * PART);
            for (int cc = 0; cc < a.NN; cc += CW) {
                uint32_t acc[PART][CG][CW];
#pragma unroll
                for (int pp = 0; pp < PART; ++pp)
#pragma unroll
                    for (int ch = 0; ch < CG; ++ch) tc_ld(dcol + (pp * CG + ch) * a.NN + cc, acc[pp][ch]);
                tc_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < CW; ++q) {
                        const int ow = ow0 + a.NN - 1 - (cc + q);   // reversed columns
                        if (ow < ow0 || ow >= ow_end) continue;
                        float vals[CG];
#pragma unroll
                        for (int ch = 0; ch < CG; ++ch) {
                            vals[ch] = __uint_as_float(acc[0][ch][q]);
                            if constexpr (PART == 2) vals[ch] += __uint_as_float(acc[1][ch][q]);
                        }
                        tc_store_pixel<OutT, CG>(orow + static_cast<size_t>(ow) * a.C, vals);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_empty[db]);
            db ^= 1u;
            if (db == 0) dphase ^= 1u;
        }
    } else if (warp < kTcPlaneWarp) {
        // ------------------------------------------------------------- run feeders
        // Feeder i copies, in order, the runs of the items issuer i takes: for each of its
        // channels, rps filter rows at a time (the runs of one channel are consecutive in
        // the run table, so an item is one bulk copy).
        const int fi = warp - kTcFeed0;
        const int fpar = fi % PART;
        if (lane == 0) {
            const uint32_t ring0 = static_cast<uint32_t>(fi) * kTcRingSlots;
            const uint32_t rmask = static_cast<uint32_t>(a.rslots) - 1u;
            const uint32_t sring0 = static_cast<uint32_t>(fi * a.rslots);
            const uint32_t slot_bytes = static_cast<uint32_t>(a.rps) * a.toep_bytes;
            uint32_t item = 0;
            bool ok = true;
            for (uint32_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
                int t, j, g;
                tc_unit(a, u, t, j, g);
                for (int ch = fi / PART; ch < CG && ok; ch += CH_STEP) {
                    const unsigned char* src =
                        a.runs + static_cast<size_t>(a.cbase + g * CG + ch) * a.FHI * a.toep_bytes;
                    for (int fh0 = fpar; fh0 < a.FHI; fh0 += PART * a.rps, ++item) {
                        const uint32_t slot = ring0 + (item & rmask);
                        const uint32_t phase = (item >> a.rshift) & 1u;
                        if (!tc_wait(&toep_empty[slot], phase ^ 1u, a, abort_flag)) { ok = false; break; }
                        const uint32_t bytes = static_cast<uint32_t>(min(a.rps, a.FHI - fh0)) * a.toep_bytes;
                        mbar_arrive_expect_tx(&toep_full[slot], bytes);
                        tc_bulk_load(toep + static_cast<size_t>(sring0 + (item & rmask)) * slot_bytes,
                                     src + static_cast<size_t>(fh0) * a.toep_bytes, bytes, &toep_full[slot]);
                    }
                }
            }
            tc_drain(toep_full, ring0, static_cast<uint32_t>(a.rslots), item, a);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- plane feeder
        // The unit's CG planes, in channel order, at ring positions pos, pos+1, ...: lane b
        // copies plane b of the channel (MR rows from the tile's first virtual row, one bulk
        // copy of a contiguous band of the plane-major copy; a plane outside the copy comes
        // from the zero band).
        const size_t pbytes = static_cast<size_t>(a.vp) * 16;
        const uint32_t ps = static_cast<uint32_t>(a.ps);
        const int kc = 2 * a.KS;
        const uint32_t band = static_cast<uint32_t>(a.MR) * 16u;
        uint32_t pos = 0;
        bool ok = true;
        for (uint32_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
            int t, j, g;
            tc_unit(a, u, t, j, g);
            const TcTile tl = tc_tile(a, t);
            const int p0 = (j * a.TWc + a.x0) / 8;   // first plane of the column tile
            for (int ch = 0; ch < CG; ++ch, ++pos) {
                const uint32_t slot = pos % ps, phase = (pos / ps) & 1u;
                if (!tc_wait_warp(&plane_empty[slot], phase ^ 1u, a, abort_flag)) { ok = false; break; }
                if (lane == 0) mbar_arrive_expect_tx(&plane_full[slot], a.plane_bytes);
                __syncwarp();
                if (lane < kc) {
                    const int c = a.cbase + g * CG + ch, pl = p0 + lane;
                    const unsigned char* src =
                        pl >= 0 && pl < a.np
                            ? a.planes + (static_cast<size_t>(c) * a.np + pl) * pbytes + static_cast<size_t>(tl.v0) * 16
                            : a.zeros;
                    tc_bulk_load(planes + static_cast<size_t>(slot) * a.plane_bytes + static_cast<size_t>(lane) * band,
                                 src, band, &plane_full[slot]);
                }
            }
        }
        if (lane == 0) tc_drain(plane_full, 0, ps, pos, a);
        __syncwarp();
    }

    // every role is done (or gave up): release the tensor memory
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTcTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host side

// Cycles of one M=128 MMA step (K = 16) with both operands in shared memory, measured on
// GB300: a floor of ~46 cycles per instruction, the 128 B/clock operand read rate of shared
// memory, and 4096 multiply-adds per clock.
inline double tc_mma_cycles(int n) {
    return std::max({46.0, (kTcM + n) / 4.0, n / 2.0});
}
// An issuing thread's cycles per ring item (wait, fences, commit) and per MMA it issues,
// fitted to the kernel's measured unit times (bf16 32x56x56x128 31x31, N = 64: items of 6 and
// 12 MMAs took ~1600 and ~2700 cycles): four issuers together then issue an MMA about every
// 46 cycles, as fast as the tensor core runs the N = 64 MMAs.
constexpr double kTcItemIssueCycles = 500.0;
constexpr double kTcMmaIssueCycles = 183.0;
// The epilogue's cycles per output pixel of a unit (128 rows x the tile's columns; every lane
// stores its own row, so each store touches 32 cache lines), fitted to the kernel's measured
// times where it, not the MMAs, sets the pace (small filters: bf16 64x56x56x128 9x9 and 17x17,
// 64x28x28x256 13x13); paired rows read the accumulators half as often again.
constexpr double kTcEpiPixelCycles = 1.5;

struct TcPlan {
    TcArgs a;
    size_t smem;
    int cg;
    bool pair;
    int Lp, Wp;                       // stacked copy: left padding, row length (columns)
    size_t planes_bytes, runs_bytes;  // scratch: stacked copy, run table
};

// Launch plan for a stride-1 problem as the row kernel sees it; false if the shape does not
// fit the kernel (the caller then takes another kernel).
inline bool tc_plan(const RowConv& p, TcPlan& P) {
    TcArgs& a = P.a;
    // 16-byte copies of 8 channels in the preparation
    if (p.C % 8 != 0 || p.FH < 1 || p.FW < 1 || p.FW > 256 || p.OH < 1 || p.OW < 1) return false;
    a.N = p.N; a.C = p.C; a.OH = p.OH; a.OW = p.OW; a.FH = p.FH;
    // virtual rows per image: the image's rows and padding, shared with the next image
    a.S = std::max({p.pad_h + p.H, p.OH + p.FH - 1 - p.pad_h, p.OH});
    // row tiles of `mrows` output rows: whole images, or bands of one image
    auto row_layout = [&](int mrows, int& kimg, int& bands) -> long long {
        if (p.OH <= mrows) {
            kimg = std::min(p.N, (mrows - p.OH) / a.S + 1);
            bands = 1;
            return kimg > 0 ? (p.N + kimg - 1) / kimg : 0;   // (no images: no tiles)
        }
        kimg = 0;
        bands = (p.OH + mrows - 1) / mrows;
        return static_cast<long long>(p.N) * bands;
    };
    if (static_cast<long long>(p.N + 1) * a.S + 2 * kTcM >= (1LL << 31)) return false;
    a.MR = (p.FH + kTcM - 1 + 7) / 8 * 8;
    if (a.MR > kTcMaxBox) return false;   // staged rows per plane
    // Row pairing, column tile, channel group and filter rows per ring item, chosen together
    // by an estimate of the busiest SM's cycles: per unit (units spread evenly over the SMs,
    // whole units only) the longer of the tensor core's MMA time and an issuer's time (a fixed
    // cost per ring item and per MMA) and the epilogue's time, plus, where shared memory cannot
    // hold the planes of two units (the next unit's planes then wait for the end of the
    // current one), the planes' copy time at 64 bytes per cycle.  Groups of 2 channels (two issuers per channel, two
    // partial sums) make units half as large, which evens out the last wave of units over
    // the SMs.  Column tiles own a multiple of 8 columns (every tile's first plane starts on
    // an 8-column boundary of the stacked copy).  Constraints: two accumulator buffers of
    // partials x CG x NN columns (paired rows: of 4 channels x 2 NN columns) in tensor memory,
    // the planes and the run rings in shared memory.
    const int cap = device_info().max_smem_optin;
    const int sms = device_info().sm_count;
    double best = 1e30;
    int best_nt = 0, best_cg = 0, best_ps = 0, best_rps = 0, best_twc = 0, best_rslots = 0;
    int best_pair = 0;
    const int mode = tc_row_pairs_mode();
    for (int pair = mode == 2 ? 1 : 0; pair <= (mode == 1 ? 0 : 1); ++pair) {
        int kimg, bands;
        const long long row_tiles = row_layout(kTcM - pair, kimg, bands);
        const int fhi = pair ? (p.FH + 1) / 2 : p.FH;
        for (int nt = 1; nt <= 64; ++nt) {
            const int twc = ((p.OW + nt - 1) / nt + 7) / 8 * 8;
            if (nt > 1 && (p.OW + twc - 1) / twc < nt) continue;
            const int nn = pair ? twc : (twc + 15) / 16 * 16;
            if ((pair ? 2 * kTcIssuers * nn : nn) > kTcDCols) continue;
            const int ks = (nn + p.FW - 1 + 15) / 16;
            const int ncm = nn / 8 + 2 * ks - 1;
            const size_t run = static_cast<size_t>(pair + 1) * ncm * 128;
            const size_t plane = static_cast<size_t>(2 * ks) * a.MR * 16;
            const long long tiles = row_tiles * ((p.OW + twc - 1) / twc);
            for (int rps = kTcRunsPerSlot; rps >= 1; --rps)
            for (int cg = 4; cg >= 2; cg /= 2)
            for (int rslots = kTcRingSlots; rslots >= 2; rslots /= 2) {
                const int part = cg >= kTcIssuers ? 1 : kTcIssuers / cg;   // partial sums
                if (part * cg * nn > kTcDCols || p.C % cg != 0 || (part > 1 && rps > 1)) continue;
                if (pair && cg != kTcIssuers) continue;
                const size_t fixed = static_cast<size_t>(kTcIssuers) * rslots * rps * run + kTcBarBytes +
                                     (pair ? kTcXBytes : 0);
                if (fixed >= static_cast<size_t>(cap)) continue;
                const int ps = static_cast<int>(std::min<size_t>(kTcMaxPlanes, (cap - fixed) / plane));
                if (ps < cg + 1) continue;   // the next unit's planes must fill while one computes
                const long long units = tiles * (p.C / cg);
                const double tensor = cg * fhi * ks * tc_mma_cycles((pair + 1) * nn);
                const int rows_per_issuer = (fhi + part - 1) / part;
                const double issue = (cg * part / kTcIssuers) * ((rows_per_issuer + rps - 1) / rps) *
                                     (kTcItemIssueCycles + rps * ks * kTcMmaIssueCycles);
                const double epi = kTcEpiPixelCycles * kTcM * twc * (pair ? 1.1 : 1.0);
                // (two partial sums cost the epilogue a second read of the accumulators and the
                // stores carry half as many channels: measured ~10 % per unit)
                const double unit = (std::max({tensor, issue, epi}) +
                                     (ps >= 2 * cg ? 0.0 : static_cast<double>(cg) * plane / 64.0)) *
                                    (part > 1 ? 1.1 : 1.0);
                const double cost = static_cast<double>((units + sms - 1) / sms) * unit;
                if (cost < best) {
                    best = cost; best_nt = nt; best_cg = cg; best_ps = ps; best_rps = rps; best_twc = twc;
                    best_rslots = rslots; best_pair = pair;
                }
            }
        }
    }
    if (best_nt == 0) return false;
    a.pair = best_pair;
    a.mrows = kTcM - best_pair;
    a.FHI = best_pair ? (p.FH + 1) / 2 : p.FH;
    const long long row_tiles = row_layout(a.mrows, a.kimg, a.bands);
    a.TWc = best_twc;
    a.NN = best_pair ? a.TWc : (a.TWc + 15) / 16 * 16;
    a.col_tiles = static_cast<uint32_t>((p.OW + a.TWc - 1) / a.TWc);
    a.KS = (a.NN + p.FW - 1 + 15) / 16;
    a.NCM = a.NN / 8 + 2 * a.KS - 1;
    a.plane_bytes = static_cast<uint32_t>(2 * a.KS) * a.MR * 16u;
    a.toep_bytes = static_cast<uint32_t>(a.pair + 1) * a.NCM * 128u;
    P.cg = best_cg;
    P.pair = best_pair != 0;
    a.cbase = 0;
    a.ncg = p.C / best_cg;
    const long long tiles = row_tiles * a.col_tiles;
    const long long units = tiles * a.ncg;
    if (units >= (1LL << 31)) return false;
    a.units = static_cast<uint32_t>(units);
    a.fd_S.init(static_cast<uint32_t>(a.S));
    a.ps = best_ps;
    a.rps = best_rps;
    a.rslots = best_rslots;
    a.rshift = best_rslots == 4 ? 2 : 1;
    // stacked copy: input column w at column w + Lp, Lp = pad_w mod 8, so that a tile's first
    // column j*TWc - pad_w lands on a multiple of 8 (x0 = Lp - pad_w); the copy spans the
    // image (planes outside it are read from a zero band)
    P.Lp = p.pad_w % 8;
    a.x0 = P.Lp - p.pad_w;
    P.Wp = (P.Lp + p.W + 7) / 8 * 8;
    // plane-major copy: the V virtual rows of every 8-column plane, then MR zero rows (the
    // last tile's band reads past V)
    a.np = P.Wp / 8;
    const long long vp = static_cast<long long>(p.N) * a.S + a.MR;
    if (vp >= (1LL << 31)) return false;
    a.vp = static_cast<uint32_t>(vp);
    P.planes_bytes = static_cast<size_t>(p.C) * a.np * a.vp * 16;
    P.runs_bytes = static_cast<size_t>(p.C) * a.FHI * a.toep_bytes;
    // shared memory: plane ring, run rings, barriers, the paired rows' exchange; one CTA per
    // SM (each allocates all of tensor memory): ask for more than half of it
    const size_t toep_ring = static_cast<size_t>(kTcIssuers) * a.rslots * a.rps * a.toep_bytes;
    a.off_toep = static_cast<uint32_t>(static_cast<size_t>(a.ps) * a.plane_bytes);
    a.off_bar = a.off_toep + static_cast<uint32_t>(toep_ring);
    a.off_x = a.off_bar + kTcBarBytes;
    P.smem = std::max<size_t>(a.off_x + (a.pair ? kTcXBytes : 0), static_cast<size_t>(cap) / 2 + 1024);
    return true;
}

template <typename T>
inline uint32_t tc_idesc(int n) {
    const uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;  // bf16 : fp16
    return (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(kTcM >> 4) << 24);
}

// One launch of the main kernel with groups of CG channels (filter rows in pairs or single).
template <typename T, class OutT, int CG, bool PAIR>
cudaError_t launch_tc_main(const TcArgs& a, size_t smem, cudaStream_t stream) {
    auto kern = tc_rows_kernel<T, OutT, CG, PAIR>;
    static DeviceOnce smem_opt_in;
    const cudaError_t err = opt_in_smem(kern, smem_opt_in, device_info().max_smem_optin);
    if (err != cudaSuccess) return err;
    const unsigned grid = static_cast<unsigned>(
        std::min<long long>(a.units, static_cast<long long>(device_info().sm_count)));
    // a programmatic dependent of the preparation kernel before it: its set-up (barriers,
    // tensor memory) overlaps the preparation's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, class OutT>
cudaError_t launch_tc_main_cg(int cg, bool pair, const TcArgs& a, size_t smem, cudaStream_t stream) {
    if (pair) return cg == 4 ? launch_tc_main<T, OutT, 4, true>(a, smem, stream) : cudaErrorNotSupported;
    switch (cg) {
        case 2: return launch_tc_main<T, OutT, 2, false>(a, smem, stream);
        case 4: return launch_tc_main<T, OutT, 4, false>(a, smem, stream);
        default: return cudaErrorNotSupported;
    }
}

template <typename T, class OutT = float>
cudaError_t launch_tc_rows(const RowConv& p) {
    TcPlan P;
    if (!tc_plan(p, P)) return cudaErrorNotSupported;
    if (P.a.units == 0) return cudaSuccess;
    const TcArgs& a = P.a;
    // scratch of this call: the stacked copy, the run table, a zero band (128-byte aligned)
    const size_t runs_off = (P.planes_bytes + 127) / 128 * 128;
    const size_t z_off = runs_off + (P.runs_bytes + 127) / 128 * 128;
    const size_t z_bytes = (static_cast<size_t>(a.MR) * 16 + 127) / 128 * 128;
    const long long run_tasks = static_cast<long long>(p.C) * a.FHI * 8 * a.NCM * (a.pair + 1);
    if (run_tasks >= (1LL << 31)) return cudaErrorNotSupported;
    // preparation: the plane-major stacked copy, the runs, and the zero band
    TcPrepArgs q;
    if (!tc_stack_args(q.st, p.in, nullptr, p.N, p.H, p.W, p.C, p.pad_h, a.S, P.Lp, P.Wp, 0,
                       static_cast<int>(a.vp)))
        return cudaErrorNotSupported;
    void* scratch = nullptr;
    if (scratch_alloc(&scratch, z_off + z_bytes, p.stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return cudaErrorNotSupported;   // the caller takes another kernel
    }
    unsigned char* base = static_cast<unsigned char*>(scratch);
    q.st.dst = base;
    q.w = p.w; q.runs = base + runs_off;
    q.C = p.C; q.FH = p.FH; q.FW = p.FW; q.NN = a.NN; q.NCM = a.NCM;
    q.FHI = a.FHI; q.pair = a.pair;
    q.run_tasks = static_cast<int>(run_tasks);
    q.fd_C.init(static_cast<uint32_t>(p.C));
    q.fd_rows.init(static_cast<uint32_t>(8 * a.NCM * (a.pair + 1)));
    const int sms = device_info().sm_count;
    q.run_blocks = static_cast<int>(
        std::min<long long>((run_tasks + kTcPrepThreads - 1) / kTcPrepThreads, 4LL * sms));
    const int plane_blocks = static_cast<int>(std::min<long long>(q.st.tiles, 16LL * sms));
    const unsigned prep_grid = static_cast<unsigned>(q.run_blocks + plane_blocks);
    cudaError_t err = cudaMemsetAsync(base + z_off, 0, z_bytes, p.stream);
    if (err == cudaSuccess) {
        if (p.flip) tc_prep_kernel<T, true><<<prep_grid, kTcPrepThreads, 0, p.stream>>>(q);
        else tc_prep_kernel<T, false><<<prep_grid, kTcPrepThreads, 0, p.stream>>>(q);
        err = cudaGetLastError();
    }
    // the main kernel
    TcArgs m = a;
    m.planes = base;
    m.zeros = base + z_off;
    m.runs = base + runs_off;
    m.out = p.out;
    m.status = p.status;
    m.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    m.idesc = tc_idesc<T>(a.NN * (a.pair + 1));
    if (err == cudaSuccess) err = launch_tc_main_cg<T, OutT>(P.cg, P.pair, m, P.smem, p.stream);
    // stream-ordered: the memory returns to the pool once the kernels have run
    scratch_free(scratch, p.stream);
    return err;
}

}  // namespace dwc
