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
//    indices, so the whole matrix is N/8 + K/8 - 1 distinct core matrices laid end to end,
//    and a descriptor with both strides 128 bytes reads every block of the K x N matrix.
//    The epilogue undoes the reversal.
//  * Rows of the tile run through several images: image n occupies the S rows starting at
//    virtual row n*S (S = image rows + padding shared with the next image), so one 128-row
//    MMA covers, for example, two 56-row images; rows in the gaps are computed and dropped.
//
// Warp roles per CTA (one CTA per SM, persistent over units of (row tile, column tile, group
// of CG = 4 or 8 channels)):
//  * 4 epilogue warps -- warp w reads the 32-lane quadrant w of the accumulators
//    (tcgen05.ld) and writes the CG channels of a pixel with 16-byte stores;
//  * 4 MMA warps: one lane each issues the MMAs of every fourth channel of the group (a
//    single thread issues an MMA only every ~100 cycles, an M=128 N=32 MMA takes 40); the
//    first also allocates the tensor memory;
//  * 8 builder warps, two per issuer taking turns: write the Toeplitz core matrices of the
//    issuer's (channel, filter row) items into its ring (one warp builds an item in about
//    0.4 us, the tensor core takes four items, one per ring, in about 0.33 us); one of them
//    stages the filters;
//  * 6 loader warps: gather the unit's input rows (CG channels, 8 or 16 bytes, per load) and
//    store them transposed into the per-channel planes (zeros in the padding).
// Groups of at least four channels keep the scattered global accesses of the gather and the
// stores (one cache line per pixel, whatever its width) well below the tensor core's time.
// Stages pass through mbarrier rings; every wait has a time limit and a shared abort flag,
// so a lost arrival ends the kernel (status word set) instead of hanging it.  Backward data
// uses the same kernel with the filter read rotated by 180 degrees.
#pragma once

#include <algorithm>
#include <type_traits>

#include "dwc_device.cuh"
#include "dwc_host.h"

namespace dwc {

constexpr int kTcM = 128;           // MMA rows (tensor-memory lanes)
// Roles (22 warps; warp w runs on sub-partition w % 4):
//   0-3   epilogue, warp w reading the 32-lane quadrant w of tensor memory
//   4-7   MMA issuers, one lane each: issuer i takes the channels c with c % 4 == i, every
//         filter row of them (one thread issues an MMA only every ~100 cycles, four keep
//         the tensor core's pace); warp 4 also allocates the tensor memory
//   8-15  Toeplitz builders, warps 8 + i and 12 + i feeding issuer i's ring in turn
//   16-21 loaders
constexpr int kTcEpiWarps = 4;
constexpr int kTcMmaWarp = 4;       // first MMA warp
constexpr int kTcIssuers = 4;       // MMA-issuing threads (one per MMA warp)
constexpr int kTcBuild0 = kTcMmaWarp + kTcIssuers;
constexpr int kTcBuildWarps = 8;     // two per issuer ring
constexpr int kTcLoad0 = kTcBuild0 + kTcBuildWarps;
constexpr int kTcLoadWarps = 6;
constexpr int kTcWarps = kTcLoad0 + kTcLoadWarps;
constexpr int kTcRingSlots = 4;     // Toeplitz slots per issuer ring (a power of two)
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcTmemCols = 512;
constexpr int kTcDCols = 256;       // columns of one accumulator buffer (two buffers)
constexpr int kTcMaxPlanes = 16;
constexpr int kTcMaxToep = 16;      // kTcIssuers rings of kTcRingSlots
// barriers (plane and Toeplitz rings, two accumulator buffers, the final MMA barrier), the
// tensor-memory address and the abort flag
constexpr int kTcMaxZ = 12;          // Toeplitz run of at most 32 * (kTcMaxZ - 1) rows
constexpr int kTcBarBytes =
    ((2 * kTcMaxPlanes + 2 * kTcMaxToep + 2 * 2 + kTcIssuers + 2 * 2) * 8 + 8 + 127) / 128 * 128;
static_assert(kTcBuildWarps == 2 * kTcIssuers && kTcIssuers * kTcRingSlots == kTcMaxToep &&
                  kTcRingSlots % 2 == 0,
              "builder warps i and i + kTcIssuers feed issuer i's ring, alternate items");

struct TcArgs {
    const void* x;      // N x H x W x C, 16-bit
    const void* w;      // FH x FW x C, 16-bit
    void* out;          // N x OH x OW x C, OutT
    unsigned int* status;
    unsigned long long wait_ns;
    int N, H, W, C, OH, OW, FH, FW, pad_h, pad_w;
    int S;              // virtual rows per image
    int kimg;           // images per row tile (0: tiles are 128-row bands of one image)
    int bands;          // row tiles per image when kimg == 0
    int NN;             // MMA N (output columns of a column tile, multiple of 16)
    int TWc;            // output columns a column tile owns (<= NN)
    int KS;             // K-steps of 16
    int MR;             // staged rows per plane (>= FH + 127, multiple of 8)
    int NCM;            // Toeplitz core matrices: NN/8 + 2*KS - 1
    int ncg;            // channel groups (C / CG)
    int ps, ts;         // plane / Toeplitz ring slots
    uint32_t units, col_tiles;
    FastDiv fd_S;
    uint32_t plane_bytes, toep_bytes;
    uint32_t off_toep, off_wst, off_bar;   // byte offsets in shared memory
    uint32_t wst_bytes;  // one filter staging slot: FH x FW taps x 8 channels, 16-bit, padded
    uint32_t wst_tx;     // bytes one filter copy delivers (FH * FW * 16, unpadded)
    int ws;              // filter staging slots (2, or 1 where two do not fit)
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
// Generic-proxy shared-memory writes become visible to the tensor cores' async proxy.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

// Bounded wait that also gives up as soon as another role has aborted the CTA.  On running
// out of time it records the timeout and raises the abort flag itself.  Between polls the
// warp sleeps, up to `max_sleep_ns`: the warps that wait most of the time (epilogue,
// loaders) then leave the issue slots of their sub-partition to the issuers and builders.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, const TcArgs& a,
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
__device__ __forceinline__ bool tc_wait_warp(uint64_t* bar, uint32_t parity, const TcArgs& a,
                                             volatile int* abort_flag, uint32_t max_sleep_ns = 32) {
    return __all_sync(0xffffffffu, tc_wait(bar, parity, a, abort_flag, max_sleep_ns));
}

// Row tile `t`: first virtual output row v0 and the rows [v_lo, v_hi) the tile owns.
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
        r.v0 = n * a.S + kTcM * b;
        r.v_lo = r.v0;
        r.v_hi = n * a.S + min(a.OH, kTcM * (b + 1));
    }
    return r;
}

// Unit u -> (row tile, column tile, channel group); the channel group is fastest, so CTAs
// running at the same time read the same input pixels (other channels of them) from L2.
__device__ __forceinline__ void tc_unit(const TcArgs& a, uint32_t u, int& t, int& j, int& g) {
    g = static_cast<int>(u % static_cast<uint32_t>(a.ncg));
    const uint32_t q = u / static_cast<uint32_t>(a.ncg);
    j = static_cast<int>(q % a.col_tiles);
    t = static_cast<int>(q / a.col_tiles);
}

template <int CG>
struct TcPix;   // CG 16-bit channels of one pixel, as loaded
template <>
struct TcPix<4> {
    using V = uint2;
    __device__ static __forceinline__ V zero() { return make_uint2(0u, 0u); }
};
template <>
struct TcPix<8> {
    using V = uint4;
    __device__ static __forceinline__ V zero() { return make_uint4(0u, 0u, 0u, 0u); }
};

// 16-bit channel `ch` (0 <= ch < CG) of a loaded pixel, in the low half of a word
// (the high half is garbage).
template <int CG>
__device__ __forceinline__ uint32_t tc_word(const typename TcPix<CG>::V& v, int ch) {
    if constexpr (CG == 4) {
        return ch < 2 ? v.x : v.y;
    } else {
        return ch < 2 ? v.x : (ch < 4 ? v.y : (ch < 6 ? v.z : v.w));
    }
}

// Two adjacent columns of channel ch packed into one word (lo column in the low half).
template <int CG>
__device__ __forceinline__ uint32_t tc_pair(const typename TcPix<CG>::V& lo,
                                            const typename TcPix<CG>::V& hi, int ch) {
    return __byte_perm(tc_word<CG>(lo, ch), tc_word<CG>(hi, ch), (ch & 1) ? 0x7632u : 0x5410u);
}

// The CG channels of one output pixel, one or two 16-byte streaming stores (fp32), or one
// 8- or 16-byte store of values rounded to nearest even (bf16, fp16).
template <class OutT, int CG>
__device__ __forceinline__ void tc_store_pixel(OutT* dst, const float (&v)[CG]) {
    if constexpr (std::is_same<OutT, float>::value) {
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
        if constexpr (CG == 4) {
            __stcs(reinterpret_cast<uint2*>(dst), make_uint2(h[0], h[1]));
        } else {
            __stcs(reinterpret_cast<uint4*>(dst), make_uint4(h[0], h[1], h[2], h[3]));
        }
    }
}

template <typename T, bool FLIP, class OutT, int CG>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_rows_kernel(const __grid_constant__ CUtensorMap wmap, const TcArgs a) {
    static_assert(CG % kTcIssuers == 0, "every issuer takes whole channels of the group");
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* planes = smem;
    unsigned char* toep = smem + a.off_toep;
    unsigned char* wst = smem + a.off_wst;   // two filter staging slots [FH][FW][8 channels]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* plane_full = bars;
    uint64_t* plane_empty = plane_full + kTcMaxPlanes;
    uint64_t* toep_full = plane_empty + kTcMaxPlanes;
    uint64_t* toep_empty = toep_full + kTcMaxToep;
    uint64_t* d_full = toep_empty + kTcMaxToep;   // [2]
    uint64_t* d_empty = d_full + 2;               // [2]
    uint64_t* mma_done = d_empty + 2;             // [kTcIssuers]
    uint64_t* w_full = mma_done + kTcIssuers;     // [2] filter staging slots
    uint64_t* w_empty = w_full + 2;               // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(w_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.ps; ++s) {
            mbar_init(&plane_full[s], kTcLoadWarps);
            mbar_init(&plane_empty[s], 1);   // the issuer of its channel
        }
        for (int s = 0; s < a.ts; ++s) {
            mbar_init(&toep_full[s], 1);
            mbar_init(&toep_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&d_full[s], kTcIssuers);
            mbar_init(&d_empty[s], kTcEpiWarps);
        }
        for (int i = 0; i < kTcIssuers; ++i) mbar_init(&mma_done[i], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], kTcBuildWarps);
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

    if (warp >= kTcMmaWarp && warp < kTcMmaWarp + kTcIssuers) {
        // ------------------------------------------------------------- MMA issue
        // Issuer `is` takes the channels c of the group with c % 4 == is, all filter rows.
        const int is = warp - kTcMmaWarp;
        if (lane == 0) {
            uint32_t db = 0, dphase = 0;
            bool ok = true;
            // Descriptors are built once; the start-address field (bits 0-13, 16-byte units)
            // then advances by plain additions: a plane slot, a filter row (16 bytes), a
            // K-step (two planes of A, two core matrices of T).
            const uint64_t adesc0 = tc_sdesc(smem_addr(planes), a.MR * 16u, 128u);
            const uint64_t bdesc0 = tc_sdesc(smem_addr(toep), 128u, 128u);
            const uint32_t a_ks = 2u * a.MR;           // A advance per K-step (16-byte units)
            const uint32_t a_slot = a.plane_bytes >> 4, b_slot = a.toep_bytes >> 4;
            const uint32_t idesc = a.idesc;
            const uint32_t ps = static_cast<uint32_t>(a.ps);
            // this issuer's Toeplitz ring: slots [is * kTcRingSlots, (is + 1) * kTcRingSlots),
            // filled in order with the runs of exactly the (channel, filter row) items it takes
            const uint32_t ring0 = static_cast<uint32_t>(is) * kTcRingSlots;
            uint32_t item = 0;
            uint32_t pos0 = 0;   // plane-ring position of the unit's first channel
            for (uint32_t u = blockIdx.x; u < a.units && ok; u += gridDim.x, pos0 += CG) {
                if (!tc_wait(&d_empty[db], dphase ^ 1u, a, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t dcol = tmem + db * kTcDCols;
                for (int ch = is; ch < CG && ok; ch += kTcIssuers) {
                    // channel ch of this unit sits at plane-ring position pos0 + ch (the
                    // loaders fill the ring in order; this issuer skips the other channels)
                    const uint32_t pos = pos0 + static_cast<uint32_t>(ch);
                    const uint32_t pslot = pos % ps, pphase = (pos / ps) & 1u;
                    if (!tc_wait(&plane_full[pslot], pphase, a, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ap = adesc0 + pslot * a_slot;
                    const uint32_t dch = dcol + static_cast<uint32_t>(ch * a.NN);
                    for (int fh = 0; fh < a.FH; ++fh, ++item) {
                        const uint32_t slot = ring0 + (item & (kTcRingSlots - 1));
                        const uint32_t phase = (item / kTcRingSlots) & 1u;
                        if (!mbar_try_wait(&toep_full[slot], phase) &&
                            !tc_wait(&toep_full[slot], phase, a, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        uint64_t ad = ap + static_cast<uint32_t>(fh);
                        uint64_t bd = bdesc0 + slot * b_slot;
                        tc_mma(dch, ad, bd, idesc, fh != 0 ? 1u : 0u);
                        for (int ks = 1; ks < a.KS; ++ks) {
                            ad += a_ks;
                            bd += 16u;
                            tc_mma(dch, ad, bd, idesc, 1u);
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
            const int c0 = g * CG;
            OutT* orow = static_cast<OutT*>(a.out) +
                         (static_cast<size_t>(row_ok ? n : 0) * a.OH + (row_ok ? r : 0)) *
                             static_cast<size_t>(a.OW) * a.C + c0;
            const uint32_t dcol = tmem + db * kTcDCols + (static_cast<uint32_t>(quad * 32) << 16);
            // columns per round: CG x CW sums in registers (32 values)
            constexpr int CW = 32 / CG;
            for (int cc = 0; cc < a.NN; cc += CW) {
                uint32_t acc[CG][CW];
#pragma unroll
                for (int ch = 0; ch < CG; ++ch) tc_ld(dcol + ch * a.NN + cc, acc[ch]);
                tc_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < CW; ++q) {
                        const int ow = ow0 + a.NN - 1 - (cc + q);   // reversed columns
                        if (ow < ow0 || ow >= ow_end) continue;
                        float vals[CG];
#pragma unroll
                        for (int ch = 0; ch < CG; ++ch) vals[ch] = __uint_as_float(acc[ch][q]);
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
    } else if (warp >= kTcLoad0) {
        // ------------------------------------------------------------- loaders
        using Pix = TcPix<CG>;
        using V = typename Pix::V;
        const int lt = (warp - kTcLoad0) * 32 + lane;   // 0 .. 32*kTcLoadWarps-1
        const T* X = static_cast<const T*>(a.x);
        const int KC = 2 * a.KS;
        const int tasks = a.MR * KC;  // (row, 8-column chunk), row fastest
        Ring pr;
        for (uint32_t u = blockIdx.x; u < a.units; u += gridDim.x) {
            int t, j, g;
            tc_unit(a, u, t, j, g);
            const TcTile tl = tc_tile(a, t);
            const int col0 = j * a.TWc - a.pad_w;
            const int c0 = g * CG;
            // the CG planes of this unit: slots pr, pr+1, ... (each released by the MMA)
            Ring q = pr;
            bool ok = true;
            uint32_t slots[CG];
#pragma unroll
            for (int ch = 0; ch < CG; ++ch) {
                if (ok && !tc_wait_warp(&plane_empty[q.slot], q.phase ^ 1u, a, abort_flag, 512)) ok = false;
                slots[ch] = q.slot;
                q.next(a.ps);
            }
            if (!ok) break;
            // TB tasks per thread per round: all their loads are in flight before the first
            // transposed store (the loads are what takes time)
            constexpr int TB = 8 / CG;   // 32 registers of loaded pixels
            constexpr int NT = 32 * kTcLoadWarps;
            for (int base = lt; base < tasks; base += TB * NT) {
                V px[TB][8];
                int tb_b[TB], tb_r[TB];
#pragma unroll
                for (int k = 0; k < TB; ++k) {
                    const int task = base + k * NT;
                    const int b = task / a.MR, rr = task - b * a.MR;
                    tb_b[k] = b;
                    tb_r[k] = rr;
                    // rows no MMA reads (and tasks past the end) are neither loaded nor stored
                    const bool live = task < tasks && rr < a.FH + kTcM - 1;
                    uint32_t rem;
                    const int vi = tl.v0 + rr;
                    const int n = static_cast<int>(a.fd_S.divmod(static_cast<uint32_t>(vi), rem));
                    const int h = static_cast<int>(rem) - a.pad_h;
                    const bool row_in = live && n < a.N && h >= 0 && h < a.H;
                    const int cb = col0 + 8 * b;
                    const T* src = X + ((static_cast<size_t>(row_in ? n : 0) * a.H + (row_in ? h : 0)) *
                                            a.W) * static_cast<size_t>(a.C) + c0;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int col = cb + e;
                        px[k][e] = (row_in && col >= 0 && col < a.W)
                                       ? __ldg(reinterpret_cast<const V*>(src + static_cast<size_t>(col) * a.C))
                                       : Pix::zero();
                    }
                    if (!live) tb_r[k] = -1;
                }
#pragma unroll
                for (int k = 0; k < TB; ++k) {
                    if (tb_r[k] < 0) continue;
#pragma unroll
                    for (int ch = 0; ch < CG; ++ch) {
                        uint4 o;
                        o.x = tc_pair<CG>(px[k][0], px[k][1], ch);
                        o.y = tc_pair<CG>(px[k][2], px[k][3], ch);
                        o.z = tc_pair<CG>(px[k][4], px[k][5], ch);
                        o.w = tc_pair<CG>(px[k][6], px[k][7], ch);
                        *reinterpret_cast<uint4*>(planes + static_cast<size_t>(slots[ch]) * a.plane_bytes +
                                                  (static_cast<size_t>(tb_b[k]) * a.MR + tb_r[k]) * 16u) = o;
                    }
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int ch = 0; ch < CG; ++ch) mbar_arrive(&plane_full[slots[ch]]);
            }
            pr = q;
        }
    } else {
        // ------------------------------------------------------------- Toeplitz builders
        // Builder warps i and i + 4 write, in turn (even and odd items), the Toeplitz runs of
        // the (channel, filter row) items MMA issuer i takes into that issuer's ring.  The unit's
        // filters (8 channels around the group) arrive by one TMA copy per unit into one of
        // the staging slots (two where they fit: the next unit's copy then travels while this
        // unit's runs are built).
        const int bidx = warp - kTcBuild0;
        const int ring = bidx % kTcIssuers;                  // the ring (issuer) this warp feeds
        const uint32_t turn = static_cast<uint32_t>(bidx / kTcIssuers);   // its items' parity
        const int rows = 8 * a.NCM;
        const int nz = (rows + 7 + 31) / 32;   // z chunks a lane holds (<= kTcMaxZ)
        const uint32_t ring0 = static_cast<uint32_t>(ring) * kTcRingSlots;
        uint32_t item = 0;
        bool ok = true;
        // Staging slot k % ws holds the filters of the CTA's unit k.  Builder warp 0's lane 0
        // issues the copies: units 0 .. ws-1 up front, unit k + ws once every builder has
        // released unit k's slot.
        const uint32_t ws = static_cast<uint32_t>(a.ws);
        uint32_t issued = 0;   // filter copies issued
        auto issue_stage = [&](uint32_t kk) -> bool {
            const uint32_t uu = blockIdx.x + kk * gridDim.x;
            const uint32_t sl = kk % ws, n = kk / ws;
            if (!tc_wait(&w_empty[sl], (n & 1u) ^ 1u, a, abort_flag)) return false;
            int t_, j_, g_;
            tc_unit(a, uu, t_, j_, g_);
            mbar_arrive_expect_tx(&w_full[sl], a.wst_tx);
            tma_load_3d(wst + sl * a.wst_bytes, &wmap, &w_full[sl], (g_ * CG) & ~7, 0, 0);
            ++issued;
            return true;
        };
        if (bidx == 0 && lane == 0) {
            prefetch_tensormap(&wmap);
            for (uint32_t kk = 0; kk < ws && ok; ++kk)
                if (blockIdx.x + kk * gridDim.x < a.units) ok = issue_stage(kk);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        uint32_t k = 0;   // unit index within this CTA
        for (uint32_t u = blockIdx.x; u < a.units && ok; u += gridDim.x, ++k) {
            int t, j, g;
            tc_unit(a, u, t, j, g);
            const uint32_t sl = k % ws;
            if (!tc_wait_warp(&w_full[sl], (k / ws) & 1u, a, abort_flag)) { ok = false; break; }
            // channel ch of the group sits at lane (g*CG) % 8 + ch of each staged tap
            const uint16_t* wtap = reinterpret_cast<const uint16_t*>(wst + sl * a.wst_bytes) +
                                   ((g * CG) & 7);
            for (int ch = ring; ch < CG && ok; ch += kTcIssuers) {
                for (int fh = 0; fh < a.FH; ++fh, ++item) {
                    if ((item & 1u) != turn) continue;   // the other warp's item
                    const uint32_t slot = ring0 + (item & (kTcRingSlots - 1));
                    const uint32_t phase = (item / kTcRingSlots) & 1u;
                    if (!tc_wait_warp(&toep_empty[slot], phase ^ 1u, a, abort_flag)) { ok = false; break; }
                    const int fhe = FLIP ? a.FH - 1 - fh : fh;
                    const uint16_t* wr = wtap + static_cast<size_t>(fhe) * a.FW * 8 + ch;
                    unsigned char* dst = toep + static_cast<size_t>(slot) * a.toep_bytes;
                    // Row r of the core-matrix run is z[r .. r+7] with z[i] = filt(fh, i - (NN-1))
                    // (zero outside the filter).  Lane l holds z[32c + l] for every chunk c and
                    // gathers its rows r = 32c + l with 8 shuffles each; all loads first, then
                    // all shuffles, so that their latencies overlap.
                    uint32_t z[kTcMaxZ];
#pragma unroll
                    for (int c = 0; c < kTcMaxZ; ++c) {
                        const int f = 32 * c + lane - (a.NN - 1);
                        z[c] = (c < nz && f >= 0 && f < a.FW) ? wr[(FLIP ? a.FW - 1 - f : f) * 8] : 0u;
                    }
#pragma unroll
                    for (int c = 0; c + 1 < kTcMaxZ; ++c) {
                        if (32 * c >= rows) break;
                        uint32_t wv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            wv[e] = __shfl_sync(0xffffffffu, lane < e ? z[c + 1] : z[c], (lane + e) & 31);
                        const int r = 32 * c + lane;
                        if (r < rows) {
                            uint4 v;
                            v.x = __byte_perm(wv[0], wv[1], 0x5410);
                            v.y = __byte_perm(wv[2], wv[3], 0x5410);
                            v.z = __byte_perm(wv[4], wv[5], 0x5410);
                            v.w = __byte_perm(wv[6], wv[7], 0x5410);
                            *reinterpret_cast<uint4*>(dst + static_cast<size_t>(r) * 16u) = v;
                        }
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&toep_full[slot]);
                }
            }
            // this warp is done with the staged filters of unit k; the slot takes unit k + ws
            __syncwarp();
            if (lane == 0) mbar_arrive(&w_empty[sl]);
            if (bidx == 0 && lane == 0 && ok && u + ws * gridDim.x < a.units) ok = issue_stage(k + ws);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        // never leave with a filter copy in flight: wait (bounded) for the last copy of each
        // staging slot (earlier ones completed before their slot was reused)
        if (bidx == 0 && lane == 0) {
            for (uint32_t kk = issued >= ws ? issued - ws : 0; kk < issued; ++kk)
                if (!mbar_wait(&w_full[kk % ws], (kk / ws) & 1u, a.wait_ns)) {
                    record_status(a.status, DWC_DEVSTAT_TIMEOUT);
                    break;
                }
        }
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

struct TcPlan {
    TcArgs a;
    size_t smem;
    int cg;
};

// Launch plan for a stride-1 problem as the row kernel sees it; false if the shape does not
// fit the kernel (the caller then takes another kernel).
inline bool tc_plan(const RowConv& p, TcPlan& P) {
    TcArgs& a = P.a;
    // the filter copy is a TMA box of 8 channels x FW x FH (each at most 256)
    if (p.C % 8 != 0 || p.FH < 1 || p.FW < 1 || p.FH > 256 || p.FW > 256 || p.OH < 1 || p.OW < 1)
        return false;
    a.N = p.N; a.H = p.H; a.W = p.W; a.C = p.C; a.OH = p.OH; a.OW = p.OW;
    a.FH = p.FH; a.FW = p.FW; a.pad_h = p.pad_h; a.pad_w = p.pad_w;
    // virtual rows per image: the image's rows and padding, shared with the next image
    a.S = std::max({p.pad_h + p.H, p.OH + p.FH - 1 - p.pad_h, p.OH});
    if (p.OH <= kTcM) {
        a.kimg = std::min(p.N, (kTcM - p.OH) / a.S + 1);
        a.bands = 1;
    } else {
        a.kimg = 0;
        a.bands = (p.OH + kTcM - 1) / kTcM;
    }
    const long long row_tiles = a.kimg > 0 ? (p.N + a.kimg - 1) / a.kimg
                                           : static_cast<long long>(p.N) * a.bands;
    if (static_cast<long long>(p.N + 1) * a.S + 2 * kTcM >= (1LL << 31)) return false;
    a.MR = (p.FH + kTcM - 1 + 7) / 8 * 8;
    // Column tile and channel group, chosen together by an estimate of the busiest SM's
    // cycles: the MMAs of its units (units spread evenly over the SMs, whole units only),
    // plus, where shared memory cannot hold the planes of two units (the next unit's gather
    // then waits for the end of the current one), the gather's one cache line per pixel.
    // Constraints: two accumulator buffers of CG x NN columns in tensor memory, the
    // builders' run limit, and the planes, Toeplitz rings and filter staging in shared memory.
    const int cap = device_info().max_smem_optin;
    const int sms = device_info().sm_count;
    const size_t wst_bytes = static_cast<size_t>((p.FH * p.FW * 16 + 127) / 128 * 128);
    double best = 1e30;
    int best_nt = 0, best_cg = 0, best_ps = 0, best_ws = 0;
    for (int nt = 1; nt <= 32; ++nt) {
        const int twc = (p.OW + nt - 1) / nt;
        const int nn = (twc + 15) / 16 * 16;
        if (nt > 1 && (p.OW + twc - 1) / twc < nt) continue;
        const int ks = (nn + p.FW - 1 + 15) / 16;
        const int ncm = nn / 8 + 2 * ks - 1;
        if (8 * ncm > 32 * (kTcMaxZ - 1)) continue;   // the builders' run limit
        const size_t plane = static_cast<size_t>(2 * ks) * a.MR * 16;
        const size_t toep_ring = static_cast<size_t>(kTcMaxToep) * ncm * 128;
        const long long tiles = row_tiles * ((p.OW + twc - 1) / twc);
        for (int cg = 8; cg >= 4; cg /= 2) {
            if (cg * nn > kTcDCols || p.C % cg != 0) continue;
            // plane slots beside one or two filter staging slots; two where that still
            // leaves room for two units' planes (or costs no plane)
            auto slots = [&](int w) -> int {
                const size_t fixed = w * wst_bytes + kTcBarBytes + toep_ring;
                if (fixed >= static_cast<size_t>(cap)) return 0;
                return static_cast<int>(std::min<size_t>(kTcMaxPlanes, (cap - fixed) / plane));
            };
            const int ps2 = slots(2), ps1 = slots(1);
            const int ws = (ps2 >= 2 * cg || ps2 == ps1) ? 2 : 1;
            const int ps = ws == 2 ? ps2 : ps1;
            if (ps < cg + 1) continue;   // the next unit's planes must fill while one computes
            const long long units = tiles * (p.C / cg);
            const double unit = cg * p.FH * ks * tc_mma_cycles(nn) +
                                (ps >= 2 * cg ? 0.0 : static_cast<double>(a.MR) * 16 * ks);
            const double cost = static_cast<double>((units + sms - 1) / sms) * unit;
            if (cost < best) {
                best = cost; best_nt = nt; best_cg = cg; best_ps = ps; best_ws = ws;
            }
        }
    }
    if (best_nt == 0) return false;
    a.TWc = (p.OW + best_nt - 1) / best_nt;
    a.NN = (a.TWc + 15) / 16 * 16;
    a.col_tiles = static_cast<uint32_t>((p.OW + a.TWc - 1) / a.TWc);
    a.KS = (a.NN + p.FW - 1 + 15) / 16;
    a.NCM = a.NN / 8 + 2 * a.KS - 1;
    a.plane_bytes = static_cast<uint32_t>(2 * a.KS) * a.MR * 16u;
    a.toep_bytes = static_cast<uint32_t>(a.NCM) * 128u;
    P.cg = best_cg;
    a.ncg = p.C / best_cg;
    const long long units = row_tiles * a.col_tiles * a.ncg;
    if (units >= (1LL << 31)) return false;
    a.units = static_cast<uint32_t>(units);
    a.fd_S.init(static_cast<uint32_t>(a.S));
    // shared memory: plane ring, Toeplitz ring, filter staging slots (one TMA box of the
    // FH x FW taps of 8 channels each), barriers
    a.wst_tx = static_cast<uint32_t>(p.FH) * p.FW * 16u;
    a.wst_bytes = (a.wst_tx + 127u) / 128u * 128u;
    a.ts = kTcMaxToep;
    a.ws = best_ws;
    a.ps = best_ps;
    const size_t toep_ring = static_cast<size_t>(a.ts) * a.toep_bytes;
    const size_t wst = static_cast<size_t>(a.ws) * a.wst_bytes;
    a.off_toep = static_cast<uint32_t>(static_cast<size_t>(a.ps) * a.plane_bytes);
    a.off_wst = a.off_toep + static_cast<uint32_t>(toep_ring);
    a.off_bar = a.off_wst + static_cast<uint32_t>(wst);
    // one CTA per SM (each allocates all of tensor memory): ask for more than half of it
    P.smem = std::max<size_t>(a.off_bar + kTcBarBytes, static_cast<size_t>(cap) / 2 + 1024);
    return true;
}

template <typename T>
inline uint32_t tc_idesc(int n) {
    const uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;  // bf16 : fp16
    return (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(kTcM >> 4) << 24);
}

template <typename T, bool FLIP, class OutT, int CG>
cudaError_t launch_tc_inst(const TcPlan& P, const RowConv& p) {
    TcArgs a = P.a;
    // filter taps as 8-channel TMA boxes: the whole FH x FW filter of 8 channels per copy
    CUtensorMap wmap;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p.C, (cuuint64_t)p.FW, (cuuint64_t)p.FH};
        const cuuint64_t strides[2] = {(cuuint64_t)p.C * 2, (cuuint64_t)p.FW * p.C * 2};
        const cuuint32_t box[3] = {8u, (cuuint32_t)p.FW, (cuuint32_t)p.FH};
        if (encode_tiled(&wmap, Elem<T>::kTmaType, 3, const_cast<void*>(p.w), dims, strides,
                         box) != CUDA_SUCCESS)
            return cudaErrorNotSupported;
    }
    a.x = p.in; a.w = p.w; a.out = p.out;
    a.status = p.status;
    a.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    a.idesc = tc_idesc<T>(a.NN);
    auto kern = tc_rows_kernel<T, FLIP, OutT, CG>;
    static DeviceOnce smem_opt_in;
    {
        const cudaError_t err = opt_in_smem(kern, smem_opt_in, device_info().max_smem_optin);
        if (err != cudaSuccess) return err;
    }
    const unsigned grid = static_cast<unsigned>(
        std::min<long long>(a.units, static_cast<long long>(device_info().sm_count)));
    kern<<<grid, kTcThreads, P.smem, p.stream>>>(wmap, a);
    return cudaGetLastError();
}

template <typename T, class OutT = float>
cudaError_t launch_tc_rows(const RowConv& p) {
    TcPlan P;
    if (!tc_plan(p, P)) return cudaErrorNotSupported;
    if (P.a.units == 0) return cudaSuccess;
    switch (P.cg) {
        case 4: return p.flip ? launch_tc_inst<T, true, OutT, 4>(P, p) : launch_tc_inst<T, false, OutT, 4>(P, p);
        case 8: return p.flip ? launch_tc_inst<T, true, OutT, 8>(P, p) : launch_tc_inst<T, false, OutT, 8>(P, p);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
