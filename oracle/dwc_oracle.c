/*
 * dwc_oracle.c -- fp64 CPU oracle for depthwise 2-D convolution (DWC).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the CUDA
 * library is checked against.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load it.  It shares no code, header, table or helper with the
 * CUDA library, and the CUDA library never calls it.
 *
 * What it computes is the plain definition, written out loop by loop in fp64:
 *
 *   Flash-DWC: Making Depthwise Convolution Compute-Efficient on GPUs,
 *     §2.1 and Fig. 1 -- every channel has its own FH x FW filter (IC = OC) and every
 *       output element is the FH*FW inner product of its input patch with that filter;
 *     §2.3 "unified channels-last layout" -- X is N x IH x IW x C, Y is N x OH x OW x C,
 *       the filter is FH x FW x C (channel last everywhere);
 *     §5.1 "backward propagation" -- backward data (BDC) convolves dY with the filter
 *       rotated by 180 degrees; backward filter (BFC) correlates X with dY and yields an
 *       FH x FW x C filter gradient;
 *     §5.2 "kernel fusion" -- batch normalisation and an activation applied to X before
 *       the forward DWC (BN + Act + DWC).
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *   - forward is a cross-correlation (no filter flip), the convention of the framework
 *     the pages compare their outputs against (§6.3.2) and the one under which the
 *     180-degree rotation of §5.1 is the adjoint;
 *   - zero padding p on both sides of both spatial axes, one stride s on both axes,
 *     OH = floor((H + 2p - FH) / s) + 1 and likewise OW;
 *   - a tap that falls outside the image contributes nothing (equal to multiplying a
 *     zero pad for finite inputs);
 *   - backward data for any stride is the exact adjoint of the forward map.  The full
 *     tensor routine scatters (loop over outputs and taps, add into dX); the per-element
 *     routine gathers (for one dX element, find every (output, tap) pair that reads it).
 *     The two forms are written independently so that each checks the other.
 *
 * Parallelism: OpenMP over independent output blocks only (never inside a sum), so the
 * summation order of every output element is fixed: fh outer, fw inner for forward and
 * backward data; n, oh, ow for the filter gradient.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Output extent along one axis: floor((in + 2p - f) / s) + 1, or 0 if the filter does
 * not fit even once. */
int dwc_oracle_out_dim(int in, int f, int s, int p)
{
    long num = (long)in + 2L * p - f;
    if (s < 1 || num < 0) return 0;
    return (int)(num / s) + 1;
}

int dwc_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void dwc_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

static inline size_t nhwc(int n, int h, int w, int c, int H, int W, int C)
{
    return (((size_t)n * H + h) * W + w) * C + c;
}

static inline size_t hwc(int fh, int fw, int c, int FW, int C)
{
    return ((size_t)fh * FW + fw) * C + c;
}

/* One forward output: Y[n,oh,ow,c] = sum_{fh,fw} X[n, oh*s+fh-p, ow*s+fw-p, c] * W[fh,fw,c]. */
static double fwd_one(const double *x, const double *w, int n, int oh, int ow, int c,
                      int H, int W, int C, int FH, int FW, int s, int p)
{
    double acc = 0.0;
    for (int fh = 0; fh < FH; ++fh) {
        int ih = oh * s + fh - p;
        if (ih < 0 || ih >= H) continue;
        for (int fw = 0; fw < FW; ++fw) {
            int iw = ow * s + fw - p;
            if (iw < 0 || iw >= W) continue;
            acc += x[nhwc(n, ih, iw, c, H, W, C)] * w[hwc(fh, fw, c, FW, C)];
        }
    }
    return acc;
}

/* Forward DWC over the whole output tensor y[N][OH][OW][C]. */
void dwc_oracle_fwd(const double *x, const double *w, double *y,
                    int N, int H, int W, int C, int FH, int FW, int s, int p)
{
    int OH = dwc_oracle_out_dim(H, FH, s, p);
    int OW = dwc_oracle_out_dim(W, FW, s, p);
    long rows = (long)N * OH;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        int n = (int)(r / OH), oh = (int)(r % OH);
        for (int ow = 0; ow < OW; ++ow)
            for (int c = 0; c < C; ++c)
                y[nhwc(n, oh, ow, c, OH, OW, C)] =
                    fwd_one(x, w, n, oh, ow, c, H, W, C, FH, FW, s, p);
    }
}

/* Forward DWC at selected outputs only: idx[k] is a flat index into y[N][OH][OW][C]. */
void dwc_oracle_fwd_at(const double *x, const double *w, const int64_t *idx, long count,
                       double *out, int N, int H, int W, int C, int FH, int FW, int s, int p)
{
    int OH = dwc_oracle_out_dim(H, FH, s, p);
    int OW = dwc_oracle_out_dim(W, FW, s, p);
    (void)N;
#pragma omp parallel for schedule(static)
    for (long k = 0; k < count; ++k) {
        int64_t i = idx[k];
        int c = (int)(i % C);  i /= C;
        int ow = (int)(i % OW); i /= OW;
        int oh = (int)(i % OH); i /= OH;
        int n = (int)i;
        out[k] = fwd_one(x, w, n, oh, ow, c, H, W, C, FH, FW, s, p);
    }
}

/* Backward data, scatter form: every forward product X[n,ih,iw,c]*W[fh,fw,c] that fed
 * Y[n,oh,ow,c] sends dY[n,oh,ow,c]*W[fh,fw,c] back to dX[n,ih,iw,c].  dx is N x H x W x C
 * (the forward input shape) and is overwritten. */
void dwc_oracle_bwd_data(const double *dy, const double *w, double *dx,
                         int N, int H, int W, int C, int FH, int FW, int s, int p)
{
    int OH = dwc_oracle_out_dim(H, FH, s, p);
    int OW = dwc_oracle_out_dim(W, FW, s, p);
    /* one (n, c) pair per task: the scatter for one image and channel touches only
     * that image and channel of dx, so tasks never collide */
    long tasks = (long)N * C;
#pragma omp parallel for schedule(static)
    for (long t = 0; t < tasks; ++t) {
        int n = (int)(t / C), c = (int)(t % C);
        for (int ih = 0; ih < H; ++ih)
            for (int iw = 0; iw < W; ++iw)
                dx[nhwc(n, ih, iw, c, H, W, C)] = 0.0;
        for (int oh = 0; oh < OH; ++oh)
            for (int ow = 0; ow < OW; ++ow) {
                double g = dy[nhwc(n, oh, ow, c, OH, OW, C)];
                for (int fh = 0; fh < FH; ++fh) {
                    int ih = oh * s + fh - p;
                    if (ih < 0 || ih >= H) continue;
                    for (int fw = 0; fw < FW; ++fw) {
                        int iw = ow * s + fw - p;
                        if (iw < 0 || iw >= W) continue;
                        dx[nhwc(n, ih, iw, c, H, W, C)] += g * w[hwc(fh, fw, c, FW, C)];
                    }
                }
            }
    }
}

/* Backward data, gather form, at selected elements of dx[N][H][W][C]:
 * dX[n,ih,iw,c] = sum over (fh, fw) with (ih + p - fh) and (iw + p - fw) divisible by s
 * and the quotients (oh, ow) inside the output, of dY[n,oh,ow,c] * W[fh,fw,c]. */
void dwc_oracle_bwd_data_at(const double *dy, const double *w, const int64_t *idx, long count,
                            double *out, int N, int H, int W, int C, int FH, int FW, int s, int p)
{
    int OH = dwc_oracle_out_dim(H, FH, s, p);
    int OW = dwc_oracle_out_dim(W, FW, s, p);
    (void)N;
#pragma omp parallel for schedule(static)
    for (long k = 0; k < count; ++k) {
        int64_t i = idx[k];
        int c = (int)(i % C);  i /= C;
        int iw = (int)(i % W); i /= W;
        int ih = (int)(i % H); i /= H;
        int n = (int)i;
        double acc = 0.0;
        for (int fh = 0; fh < FH; ++fh) {
            int th = ih + p - fh;
            if (th < 0 || th % s != 0) continue;
            int oh = th / s;
            if (oh >= OH) continue;
            for (int fw = 0; fw < FW; ++fw) {
                int tw = iw + p - fw;
                if (tw < 0 || tw % s != 0) continue;
                int ow = tw / s;
                if (ow >= OW) continue;
                acc += dy[nhwc(n, oh, ow, c, OH, OW, C)] * w[hwc(fh, fw, c, FW, C)];
            }
        }
        out[k] = acc;
    }
}

/* One filter-gradient element:
 * dW[fh,fw,c] = sum_{n,oh,ow} X[n, oh*s+fh-p, ow*s+fw-p, c] * dY[n,oh,ow,c]. */
static double bwd_filter_one(const double *x, const double *dy, int fh, int fw, int c,
                             int N, int H, int W, int C, int s, int p, int OH, int OW)
{
    double acc = 0.0;
    for (int n = 0; n < N; ++n)
        for (int oh = 0; oh < OH; ++oh) {
            int ih = oh * s + fh - p;
            if (ih < 0 || ih >= H) continue;
            for (int ow = 0; ow < OW; ++ow) {
                int iw = ow * s + fw - p;
                if (iw < 0 || iw >= W) continue;
                acc += x[nhwc(n, ih, iw, c, H, W, C)] * dy[nhwc(n, oh, ow, c, OH, OW, C)];
            }
        }
    return acc;
}

/* Filter gradient over the whole dw[FH][FW][C] (overwritten). */
void dwc_oracle_bwd_filter(const double *x, const double *dy, double *dw,
                           int N, int H, int W, int C, int FH, int FW, int s, int p)
{
    int OH = dwc_oracle_out_dim(H, FH, s, p);
    int OW = dwc_oracle_out_dim(W, FW, s, p);
    long total = (long)FH * FW * C;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < total; ++t) {
        int c = (int)(t % C);
        int fw = (int)((t / C) % FW);
        int fh = (int)(t / ((long)C * FW));
        dw[t] = bwd_filter_one(x, dy, fh, fw, c, N, H, W, C, s, p, OH, OW);
    }
}

/* Filter gradient at selected flat indices of dw[FH][FW][C]. */
void dwc_oracle_bwd_filter_at(const double *x, const double *dy, const int64_t *idx, long count,
                              double *out, int N, int H, int W, int C, int FH, int FW, int s, int p)
{
    int OH = dwc_oracle_out_dim(H, FH, s, p);
    int OW = dwc_oracle_out_dim(W, FW, s, p);
    (void)FH;
#pragma omp parallel for schedule(dynamic, 1)
    for (long k = 0; k < count; ++k) {
        int64_t i = idx[k];
        int c = (int)(i % C);  i /= C;
        int fw = (int)(i % FW); i /= FW;
        int fh = (int)i;
        out[k] = bwd_filter_one(x, dy, fh, fw, c, N, H, W, C, s, p, OH, OW);
    }
}

/* Batch normalisation with given per-channel statistics, then an activation, element by
 * element: the BN + Act that the pages fuse in front of a forward DWC (Flash-DWC, §5.2
 * "kernel fusion").  For every pixel row of C channels:
 *
 *   z[.., c] = act((x[.., c] - mean[c]) / sqrt(var[c] + eps) * gamma[c] + beta[c])
 *
 * with act 0 = identity, 1 = ReLU max(v, 0), 2 = ReLU6 min(max(v, 0), 6).  The DWC that
 * follows zero-pads z itself (its out-of-image taps contribute nothing), so the fused
 * forward is dwc_oracle_fwd applied to z. */
void dwc_oracle_bn_act(const double *x, const double *mean, const double *var,
                       const double *gamma, const double *beta, double eps, int act,
                       double *z, long pixels, int C)
{
#pragma omp parallel for schedule(static)
    for (long q = 0; q < pixels; ++q) {
        for (int c = 0; c < C; ++c) {
            double v = (x[(size_t)q * C + c] - mean[c]) / sqrt(var[c] + eps) * gamma[c] + beta[c];
            if (act >= 1 && v < 0.0) v = 0.0;
            if (act == 2 && v > 6.0) v = 6.0;
            z[(size_t)q * C + c] = v;
        }
    }
}
