/*
 * fathom_probe.h -- measurement helpers used to put roofline denominators
 * beside the scan's numbers.  Not part of the method.
 *
 * The Fathom article ("Where the memory lives changes the answer", "One
 * measurement worth carrying around") and the Rootconf proposal stress that
 * with the index in host memory the scan is bounded by the host link, so the
 * link's own streaming-read rate is the denominator for the host-resident
 * scan.  This probe measures it with the same access pattern the scan uses:
 * coalesced 16-byte loads issued by the GPU's SMs (zero-copy), with no copy
 * engine involved.
 */
#ifndef FATHOM_PROBE_H
#define FATHOM_PROBE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Stream-read `bytes` (a multiple of 16, > 0) from `buf` (device memory or
 * pinned, mapped host memory; 16-byte aligned) with a grid of
 * blocks_per_sm x (number of SMs) CTAs of `threads` threads (a multiple of 32,
 * <= 1024).  The XOR of everything read is written to *sink (device uint32)
 * so the loads cannot be elided.  Asynchronous on `stream`.
 * Returns FATHOM_OK or FATHOM_EINVAL / FATHOM_ECUDA (see fathom.h). */
int fathom_probe_stream_read(const void* buf, size_t bytes, int blocks_per_sm, int threads, uint32_t* sink,
                             void* stream);

/* Integer ALU rate, for the machine balance of integer operations per byte of
 * bandwidth ([A] "Where this does not work": about five integer operations per
 * byte on an A100 or H100, so a scan that is arithmetic-bound on one of them is
 * on all).  A grid of blocks_per_sm x (number of SMs) CTAs of `threads`
 * threads; every thread runs 8 independent chains of `iters` steps, each step
 * two right shifts and one three-input XOR: 24 * iters ALU operations per
 * thread.  *sink (device uint32) keeps the result live.  Asynchronous. */
int fathom_probe_int_ops(int iters, int blocks_per_sm, int threads, uint32_t* sink, void* stream);

/* Number of SMs of the current device (the probes' grid unit). */
int fathom_probe_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* FATHOM_PROBE_H */
