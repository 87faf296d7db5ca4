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

#ifdef __cplusplus
}
#endif

#endif /* FATHOM_PROBE_H */
