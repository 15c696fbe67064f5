/*
 * dwc_testing.h -- fault injection for tests of libdwc_gb300.so's failure path, and kernel
 * selection for tests that run every kernel on the same shapes.
 *
 * No counterpart in the paper.  The injected failure is made on the host side and involves
 * no GPU fault: a kernel is told not to issue some of its own input copies, so its compute
 * warps wait until their wait limit (dwc_set_wait_limit_ns) runs out, record the timeout in
 * the device status word and end.  No copy is in flight at that point.
 */
#ifndef DWC_GB300_TESTING_H
#define DWC_GB300_TESTING_H

#include "dwc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The next launch of the row-streaming kernel (dwc_fwd / dwc_bwd_data on a shape that
 * dwc_path reports as 1, stride 1) issues no input copy in its first CTA.  That CTA's
 * outputs are left unwritten and dwc_device_status() then returns DWC_ERR_TIMEOUT.  The
 * request is consumed by that one launch; launches of other kernels leave it pending.  Not
 * for production use. */
void dwc_testing_stall_next_row_launch(void);

/* Kernel family for the 16-bit forward / backward-data calls made from now on, where that
 * family can run the shape (else the automatic choice): 0 = automatic (the default),
 * 1 = CUDA-core row kernel, 2 = tcgen05 tensor-core kernel, 4 = warp-level MMA kernel (the
 * family numbers of dwc_path, which reports the choice).  It also bypasses the small-map
 * kernels for 16-bit inputs.  For 16-bit filter gradients of square filters outside the
 * small-map shapes: 2 takes the tcgen05 kernel where it fits, 4 the warp-level MMA kernel
 * where it fits, 1 the CUDA-core kernel.  Lets tests run every kernel on the same shapes and benchmarks
 * compare them.  Returns the previous preference, or -1 (nothing changed) for an unknown
 * family.  Not for production use. */
int dwc_testing_prefer_family(int family);

/* Filter rows per MMA of the tcgen05 kernel for the calls made from now on: 0 = the launch
 * plan's choice (the default), 1 = one filter row per MMA, 2 = two filter rows per MMA (the
 * paired-row form: one MMA of twice the width against the same input rows).  A shape the
 * forced form cannot run takes another kernel.  Lets tests run both forms of the kernel on
 * the same shapes.  Returns the previous mode, or -1 (nothing changed) for an unknown mode.
 * Not for production use. */
int dwc_testing_tc_row_pairs(int mode);

#ifdef __cplusplus
}
#endif

#endif /* DWC_GB300_TESTING_H */
