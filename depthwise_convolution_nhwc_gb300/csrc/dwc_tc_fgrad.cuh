// dwc_tc_fgrad.cuh -- filter gradient on the 5th-generation tensor cores (tcgen05 MMA,
// accumulators in tensor memory) for 16-bit inputs, fp32 accumulation.
//
// The filter gradient of "Flash-DWC: Making Depthwise Convolution Compute-Efficient on GPUs"
// (§3.3, the reduction of x * dy over images and output pixels for every tap), written as
// an MMA whose two operands are plain input rows.  For one channel and the stacked rows of
// every image (the layout of the forward kernel's preparation: image n on the S virtual rows
// from n*S, zero rows between images, so that dy row v meets x row v + fh for filter row fh):
//
//   D_j[m, n] = sum_r x[r + fh0, X0 + m] * dy[r - j, n0 + n]     (j = 0..3)
//   dw[fh0 + j, fw] = sum_n D_j[n + fw, n]                        (a diagonal of D_j)
//
// where X0 = n0 - pad_w (the x column of output column n0 at tap 0), m runs over the x
// columns a tile of dy can meet and r over all virtual rows.  Per K-step of 16 rows four MMAs
// of M=128, K=16 share A = 16 rows of x; MMA j takes B = the staged dy band read from a start
// address j rows earlier: the dy rows j above A's rows.  Two shapes of a tile:
//  * wide (rows of 44+ outputs): 64 dy columns (N=64) against 128 x columns;
//  * narrow (rows of at most 32 outputs): 32 dy columns (N=32) against two bands of 64 x
//    columns stacked in M, the second staged 4 rows lower -- its half of D_j holds filter row
//    fh0 + 4 + j -- so that a unit of 8 filter rows uses all of M for a narrow dy tile.
// (Rows per MMA of 2 or 4 -- N = 128 or 256 over shifted dy bands, 2 or 1 issuers -- read A
// once per 2 or 4 rows but took 1.1x and 1.7x the time on bf16 32x56x56x128 31x31: fewer
// threads do not issue the wider MMAs as fast as the tensor core runs them, and one
// accumulator cannot take MMAs from two threads.)  Both operands are read in the MN-major
// core-matrix layout: 8 columns of a row are 16 contiguous bytes, consecutive rows 16 bytes
// apart, so a band of an 8-column plane lands in shared memory exactly as the stacked copy
// holds it.  A unit is (channel, group of filter rows) over every row and column tile: its
// accumulators hold the whole sum, so the epilogue writes dw directly (no partial slices)
// after summing the diagonals.
//
// Two launches: a preparation kernel writes the stacked copies of x (the forward's padding)
// and of dy (no padding), plane-major -- every 8-column plane of a channel holds its virtual
// rows contiguously, with zero rows before and after -- then the main kernel, which moves
// each stage's plane bands with bulk copies (2 KB contiguous each).  Tensor-map boxes of
// these bands (16-byte inner rows) ran at one row per clock: 3300 clocks a stage, twice the
// stage's MMA time.  Warp roles (9 warps, one persistent CTA per SM): warps 0-3 epilogue
// (warp w reads the 32-lane quadrant w of the accumulators), warps 4-7 the MMA issuers (one
// lane each; issuer j owns the filter rows of shift j of every unit; warp 4 allocates the
// tensor memory), warp 8 the copy producer (lane i copies plane band i of a stage: 16 x bands
// of 128 rows, 8 or 4 dy bands of 131 rows).  Every wait is bounded.
#pragma once

#include "dwc_tc.cuh"

namespace dwc {

constexpr int kTfgKB = 128;          // virtual rows per stage (8 K-steps of 16)
constexpr int kTfgStages = 4;
constexpr int kTfgXPlanes = 16;      // 128 x columns of A (one or two bands)
constexpr int kTfgShifts = 4;        // dy row shifts: MMAs (and issuers) per K-step
constexpr int kTfgDyRows = kTfgKB + kTfgShifts - 1;   // 131 rows of a dy band
constexpr int kTfgRO = kTfgShifts - 1;                // zero rows before row 0 of a plane
constexpr int kTfgEpiWarps = 4;
constexpr int kTfgMmaWarp = 4;
constexpr int kTfgTmaWarp = kTfgMmaWarp + kTfgShifts;
constexpr int kTfgThreads = (kTfgTmaWarp + 1) * 32;
constexpr int kTfgXBytes = kTfgXPlanes * kTfgKB * 16;                    // 32 KB
constexpr int kTfgRowFloats = 65;    // epilogue staging: 128 rows of up to 64 columns + 1 pad
constexpr int kTfgEpiBytes = 128 * kTfgRowFloats * 4;

// The two tile shapes (NARROW: 32 dy columns against two x bands of 64 columns).
template <bool NARROW>
struct TfgShape {
    static constexpr int kDyCols = NARROW ? 32 : 64;          // dy columns of a tile (MMA N)
    static constexpr int kDyPlanes = kDyCols / 8;
    static constexpr int kXBands = NARROW ? 2 : 1;            // x bands stacked in M
    static constexpr int kBandPlanes = kTfgXPlanes / kXBands;  // planes of a band
    static constexpr int kBandShift = 4;                      // rows between the x bands
    static constexpr int kRows = kTfgShifts * kXBands;        // filter rows of a unit
    static constexpr int kMaxFW = kBandPlanes * 8 - kDyCols + 1;
    static constexpr int kDyBytes = kDyPlanes * kTfgDyRows * 16;
    static constexpr int kStageBytes = kTfgXBytes + kDyBytes;
    static constexpr int kBarOff = kTfgStages * kStageBytes + kTfgEpiBytes;
    // barriers: full and empty per stage, two accumulator buffers, the epilogue's own, one
    // per issuer; then the tensor-memory address and the abort flag
    static constexpr int kBarBytes = (2 * kTfgStages + 2 * 2 + 1 + kTfgShifts) * 8 + 8;
    static constexpr int kSmem = kBarOff + 256;
    static_assert(kBarBytes <= 256, "barrier area");
    static_assert(kTfgShifts * kDyCols <= kTcDCols, "a unit's accumulators in one buffer");
};

struct TcFgArgs {
    const unsigned char* xpl;    // stacked x: C x npx planes x vp rows x 16 bytes
    const unsigned char* dypl;   // stacked dy: C x npd planes x vp rows x 16 bytes
    const unsigned char* zeros;  // kTfgDyRows * 16 zero bytes
    float* dw;          // FH x FW x C
    unsigned int* status;
    unsigned long long wait_ns;
    int npx, npd;       // planes of the stacked copies
    uint32_t vp;        // rows of a plane (virtual row v at row v + kTfgRO)
    int C, FH, FW;
    int groups;         // filter-row groups (of the tile shape's kRows) per channel
    int col_tiles;      // dy column tiles
    int row_blocks;     // stages of kTfgKB virtual rows per column tile
    int x0;             // stacked x column of dy column 0 at tap 0 (a multiple of 8, <= 0)
    uint32_t units;     // C * groups
    uint32_t idesc;
};

template <typename T, bool NARROW>
__global__ void __launch_bounds__(kTfgThreads, 1)
tc_fgrad_kernel(const TcFgArgs a) {
    using Sh = TfgShape<NARROW>;
    extern __shared__ __align__(1024) unsigned char smem[];
    float* stage_d = reinterpret_cast<float*>(smem + kTfgStages * Sh::kStageBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kBarOff);
    uint64_t* full = bars;                        // [kTfgStages]
    uint64_t* empty = full + kTfgStages;          // [kTfgStages]
    uint64_t* d_full = empty + kTfgStages;        // [2]
    uint64_t* d_empty = d_full + 2;               // [2]
    uint64_t* epi_bar = d_empty + 2;              // the epilogue warps' own barrier
    uint64_t* mma_done = epi_bar + 1;             // [kTfgShifts]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + kTfgShifts);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTfgStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kTfgShifts);   // every issuer's MMAs on the stage
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&d_full[s], kTfgShifts);
            mbar_init(&d_empty[s], kTfgEpiWarps);
        }
        mbar_init(epi_bar, kTfgEpiWarps);
        for (int q = 0; q < kTfgShifts; ++q) mbar_init(&mma_done[q], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kTfgMmaWarp) {
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
    const uint32_t iters = static_cast<uint32_t>(a.col_tiles * a.row_blocks);   // stages per unit
    // launched as a programmatic dependent of the stacking kernel: both copies and the zero
    // band are complete and visible past this point
    pdl_wait();

    if (warp == kTfgTmaWarp) {
        // ------------------------------------------------------------- copy producer
        // Lane i < 16: x plane p = i % kBandPlanes of band h = i / kBandPlanes, rows
        // r0 + fh0 + 4 h .. + 127, from column kDyCols t + x0; lane 16 + p: dy plane p, rows
        // r0 - 3 .. r0 + 127, from column kDyCols t.  A plane outside a stacked copy comes
        // from the zero buffer (with several column tiles its rows would otherwise enter
        // accumulator rows that other tiles fill).
        const size_t pbytes = static_cast<size_t>(a.vp) * 16;
        uint32_t k = 0;
        bool ok = true;
        for (uint32_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
            const int c = static_cast<int>(u / static_cast<uint32_t>(a.groups));
            const int fh0 = Sh::kRows * static_cast<int>(u % static_cast<uint32_t>(a.groups));
            for (uint32_t it = 0; it < iters; ++it, ++k) {
                const int t = static_cast<int>(it / static_cast<uint32_t>(a.row_blocks));
                const int r0 = static_cast<int>(it % static_cast<uint32_t>(a.row_blocks)) * kTfgKB;
                const uint32_t s = k % kTfgStages, ph = (k / kTfgStages) & 1u;
                if (!tc_wait_warp(&empty[s], ph ^ 1u, a, abort_flag)) { ok = false; break; }
                unsigned char* st = smem + s * Sh::kStageBytes;
                if (lane == 0) mbar_arrive_expect_tx(&full[s], Sh::kStageBytes);
                __syncwarp();
                if (lane < kTfgXPlanes) {
                    const int h = lane / Sh::kBandPlanes;
                    const int pl = (Sh::kDyCols * t + a.x0) / 8 + lane % Sh::kBandPlanes;
                    const unsigned char* src =
                        pl >= 0 && pl < a.npx
                            ? a.xpl + (static_cast<size_t>(c) * a.npx + pl) * pbytes +
                                  static_cast<size_t>(kTfgRO + r0 + fh0 + Sh::kBandShift * h) * 16
                            : a.zeros;
                    tc_bulk_load(st + lane * (kTfgKB * 16), src, kTfgKB * 16, &full[s]);
                } else if (lane < kTfgXPlanes + Sh::kDyPlanes) {
                    const int i = lane - kTfgXPlanes, pl = Sh::kDyPlanes * t + i;
                    const unsigned char* src =
                        pl < a.npd ? a.dypl + (static_cast<size_t>(c) * a.npd + pl) * pbytes +
                                         static_cast<size_t>(kTfgRO + r0 - (kTfgShifts - 1)) * 16
                                   : a.zeros;
                    tc_bulk_load(st + kTfgXBytes + i * (kTfgDyRows * 16), src, kTfgDyRows * 16, &full[s]);
                }
            }
        }
        if (lane == 0) tc_drain(full, 0, kTfgStages, k, a);
        __syncwarp();
    } else if (warp >= kTfgMmaWarp) {
        // ------------------------------------------------------------- MMA issue
        // shift j: accumulator columns kDyCols j .. (both x bands in the MMA's M)
        const int j = warp - kTfgMmaWarp;
        if (lane == 0) {
            // MN-major descriptors: K-direction groups of 8 rows 128 bytes apart, M/N-direction
            // groups of 8 columns (planes) one plane band apart; a K-step is 16 rows (256 B).
            // B starts 3 - j rows into the staged dy band: the dy rows j above A's rows.
            const uint64_t xd0 = tc_sdesc(smem_addr(smem), 128u, kTfgKB * 16u);
            const uint64_t dd0 = tc_sdesc(smem_addr(smem + kTfgXBytes), 128u, kTfgDyRows * 16u) +
                                 static_cast<uint32_t>(kTfgShifts - 1 - j);
            const uint32_t stage16 = Sh::kStageBytes >> 4;
            uint32_t db = 0, dphase = 0, k = 0;
            bool ok = true;
            for (uint32_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
                if (!tc_wait(&d_empty[db], dphase ^ 1u, a, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + db * kTcDCols + static_cast<uint32_t>(Sh::kDyCols * j);
                for (uint32_t it = 0; it < iters; ++it, ++k) {
                    const uint32_t s = k % kTfgStages, ph = (k / kTfgStages) & 1u;
                    if (!tc_wait(&full[s], ph, a, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    uint64_t ad = xd0 + s * stage16, bd = dd0 + s * stage16;
#pragma unroll
                    for (int ks = 0; ks < kTfgKB / 16; ++ks) {
                        tc_mma(d, ad, bd, a.idesc, (it | ks) != 0 ? 1u : 0u);
                        ad += 16u;   // 16 rows = 256 bytes
                        bd += 16u;
                    }
                    tc_commit(&empty[s]);
                }
                if (!ok) break;
                tc_commit(&d_full[db]);
                db ^= 1u;
                if (db == 0) dphase ^= 1u;
            }
            tc_commit(&mma_done[j]);
            if (!mbar_wait(&mma_done[j], 0, a.wait_ns)) record_status(a.status, DWC_DEVSTAT_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- epilogue
        // Per shift j of the unit: the 128 x kDyCols accumulator tile goes to shared memory
        // (row m = lane of quadrant w), then thread t sums diagonals t, t + 128, ... of the
        // kXBands x FW (band h, tap fw): dw[fh0 + 4 h + j][fw] = sum_n D_j[64 h + n + fw][n].
        const int quad = warp;
        const int m = quad * 32 + lane;
        uint32_t db = 0, dphase = 0, eph = 0;
        bool ok = true;
        for (uint32_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
            const int c = static_cast<int>(u / static_cast<uint32_t>(a.groups));
            const int fh0 = Sh::kRows * static_cast<int>(u % static_cast<uint32_t>(a.groups));
            if (!tc_wait_warp(&d_full[db], dphase, a, abort_flag, 1024)) break;
            tc_fence_after();
            const uint32_t dq = tmem + db * kTcDCols + (static_cast<uint32_t>(quad * 32) << 16);
            for (int j = 0; j < kTfgShifts && ok; ++j) {
                for (int cb = 0; cb < Sh::kDyCols; cb += 16) {
                    uint32_t v[16];
                    tc_ld16(dq + j * Sh::kDyCols + cb, v);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) stage_d[m * kTfgRowFloats + cb + e] = __uint_as_float(v[e]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(epi_bar);
                if (!tc_wait_warp(epi_bar, eph, a, abort_flag, 256)) { ok = false; break; }
                eph ^= 1u;
                for (int task = m; task < Sh::kXBands * a.FW; task += 128) {
                    const int h = task / a.FW, fw = task - h * a.FW;
                    const int fh = fh0 + Sh::kBandShift * h + j;
                    if (fh >= a.FH) continue;
                    const float* col = stage_d + (Sh::kBandPlanes * 8 * h + fw) * kTfgRowFloats;
                    float sum = 0.f;
#pragma unroll 8
                    for (int n = 0; n < Sh::kDyCols; ++n) sum += col[n * (kTfgRowFloats + 1)];
                    a.dw[(static_cast<size_t>(fh) * a.FW + fw) * a.C + c] = sum;
                }
                // every thread is done reading before the next shift overwrites the tile
                __syncwarp();
                if (lane == 0) mbar_arrive(epi_bar);
                if (!tc_wait_warp(epi_bar, eph, a, abort_flag, 256)) { ok = false; break; }
                eph ^= 1u;
            }
            if (!ok) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_empty[db]);
            db ^= 1u;
            if (db == 0) dphase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTfgMmaWarp) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTcTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host side

// The stacked copies of x and dy (the forward preparation's layout; dy without padding).
struct TcFgPlan {
    int S;              // virtual rows per image
    long long V;        // N * S
    int Lp, Wp;         // x copy: left padding, row length (a multiple of 8)
    int Wdp;            // dy copy: row length (a multiple of 8)
    size_t x_bytes, dy_bytes;
    bool narrow;        // the narrow tile shape (rows of at most 32 outputs)
    TcFgArgs a;
};

inline bool tc_fgrad_plan(const FilterGrad& p, TcFgPlan& P) {
    using Wide = TfgShape<false>;
    using Narrow = TfgShape<true>;
    if (p.FH < 1 || p.FW < 1 || p.C % 8 != 0 || p.N < 1) return false;
    P.narrow = p.OW <= Narrow::kDyCols && p.FW <= Narrow::kMaxFW;
    if (!P.narrow && p.FW > Wide::kMaxFW) return false;
    const int rows = P.narrow ? Narrow::kRows : Wide::kRows;
    const int dycols = P.narrow ? Narrow::kDyCols : Wide::kDyCols;
    if (device_info().max_smem_optin < (P.narrow ? Narrow::kSmem : Wide::kSmem)) return false;
    P.S = std::max({p.pad + p.H, p.OH + p.FH - 1 - p.pad, p.OH});
    P.V = static_cast<long long>(p.N) * P.S;
    if (P.V + 2 * kTfgKB >= (1LL << 31)) return false;
    P.Lp = p.pad % 8;
    P.Wp = (P.Lp + p.W + 7) / 8 * 8;
    P.Wdp = (p.OW + 7) / 8 * 8;
    TcFgArgs& a = P.a;
    a.C = p.C; a.FH = p.FH; a.FW = p.FW;
    a.groups = (p.FH + rows - 1) / rows;
    a.col_tiles = (p.OW + dycols - 1) / dycols;
    a.row_blocks = static_cast<int>((P.V + kTfgShifts - 1 + kTfgKB - 1) / kTfgKB);
    a.x0 = P.Lp - p.pad;
    a.npx = P.Wp / 8;
    a.npd = P.Wdp / 8;
    // rows of a plane: kTfgRO zero rows, the V virtual rows, and zero rows up to the last
    // stage's x rows (r0 + fh0 + 4 h + 127 for the last row block, filter-row group and band)
    const long long vp = kTfgRO + static_cast<long long>(a.row_blocks) * kTfgKB + rows * a.groups;
    if (vp >= (1LL << 31)) return false;
    a.vp = static_cast<uint32_t>(vp);
    P.x_bytes = static_cast<size_t>(p.C) * a.npx * a.vp * 16;
    P.dy_bytes = static_cast<size_t>(p.C) * a.npd * a.vp * 16;
    const long long units = static_cast<long long>(p.C) * a.groups;
    if (units >= (1LL << 31)) return false;
    a.units = static_cast<uint32_t>(units);
    return true;
}

// Instruction descriptor: kind::f16, fp32 accumulation, both operands MN-major, M=128, N=n.
template <typename T>
inline uint32_t tc_fgrad_idesc(int n) {
    const uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | (1u << 15) | (1u << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(kTcM >> 4) << 24);
}

// Both stacked copies of a call (the tiles of x, then those of dy) and the zero band.
template <typename T>
__global__ void __launch_bounds__(256) tc_stack_pm_kernel(const TcStackArgs ax, const TcStackArgs ady,
                                                          uint4* zeros, int zero_words) {
    pdl_trigger();   // the main kernel may be scheduled now (it waits for this grid)
    __shared__ uint32_t tile[8 * kStackRows * kStackWords];   // [column][row][words]
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < zero_words; i += blockDim.x) zeros[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int tt = blockIdx.x; tt < ax.tiles + ady.tiles; tt += gridDim.x) {
        if (tt < ax.tiles) tc_stack_tile<T>(ax, tt, tile);
        else tc_stack_tile<T>(ady, tt - ax.tiles, tile);
    }
}

template <typename T, bool NARROW>
cudaError_t launch_tc_fgrad_main(const TcFgArgs& a, cudaStream_t stream) {
    auto kern = tc_fgrad_kernel<T, NARROW>;
    static DeviceOnce smem_opt_in;
    const cudaError_t err = opt_in_smem(kern, smem_opt_in, device_info().max_smem_optin);
    if (err != cudaSuccess) return err;
    const unsigned grid = static_cast<unsigned>(
        std::min<long long>(a.units, static_cast<long long>(device_info().sm_count)));
    // a programmatic dependent of the stacking kernel before it: its set-up overlaps the
    // stacking's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTfgThreads);
    cfg.dynamicSmemBytes = TfgShape<NARROW>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T>
cudaError_t launch_tc_fgrad(const FilterGrad& p) {
    TcFgPlan P;
    if (!tc_fgrad_plan(p, P)) return cudaErrorNotSupported;
    // scratch of this call: the stacked x, the stacked dy, a zero band (128-byte aligned parts)
    const size_t dy_off = (P.x_bytes + 127) / 128 * 128;
    const size_t z_off = dy_off + (P.dy_bytes + 127) / 128 * 128;
    const size_t z_bytes = (kTfgDyRows * 16 + 127) / 128 * 128;
    void* scratch = nullptr;
    if (scratch_alloc(&scratch, z_off + z_bytes, p.stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return cudaErrorNotSupported;   // the caller takes another kernel
    }
    unsigned char* base = static_cast<unsigned char*>(scratch);
    const int vp = static_cast<int>(P.a.vp);
    TcStackArgs sx, sdy;
    if (!tc_stack_args(sx, p.x, base, p.N, p.H, p.W, p.C, p.pad, P.S, P.Lp, P.Wp, kTfgRO, vp) ||
        !tc_stack_args(sdy, p.dy, base + dy_off, p.N, p.OH, p.OW, p.C, 0, P.S, 0, P.Wdp, kTfgRO, vp)) {
        scratch_free(scratch, p.stream);
        return cudaErrorNotSupported;
    }
    const unsigned sgrid = static_cast<unsigned>(
        std::min<long long>(static_cast<long long>(sx.tiles) + sdy.tiles, 16LL * device_info().sm_count));
    tc_stack_pm_kernel<T><<<sgrid, 256, 0, p.stream>>>(sx, sdy, reinterpret_cast<uint4*>(base + z_off),
                                                       static_cast<int>(z_bytes / 16));
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) {
        TcFgArgs a = P.a;
        a.xpl = base;
        a.dypl = base + dy_off;
        a.zeros = base + z_off;
        a.dw = p.dw;
        a.status = p.status;
        a.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
        a.idesc = tc_fgrad_idesc<T>(P.narrow ? TfgShape<true>::kDyCols : TfgShape<false>::kDyCols);
        err = P.narrow ? launch_tc_fgrad_main<T, true>(a, p.stream) : launch_tc_fgrad_main<T, false>(a, p.stream);
    }
    scratch_free(scratch, p.stream);
    return err;
}

}  // namespace dwc
