/*
 * pa_probe.h -- a measurement helper exported by libpa.so beside the attention
 * ABI of pa.h.
 *
 * The paged-attention kernels only read the KV cache (the writes are the small
 * query-sized output), so the ceiling they are measured against is how fast
 * this GPU's HBM can be READ, which a read+write copy does not show. This call
 * is a plain streaming read of a device buffer, nothing else: the reference
 * pages have no counterpart; it exists so that a roofline fraction can be
 * taken against a read measured on the same GPU in the same process.
 */
#ifndef PA_PROBE_H
#define PA_PROBE_H

#include <stddef.h>
#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * pa_hbm_read_probe -- read `bytes` of device memory once (asynchronous).
 *
 * buf            device, 32-byte aligned; `bytes` a multiple of 32 and > 0.
 * ctas_per_sm    1..8: the grid is the device's SM count times this, 512
 *                threads a CTA, each thread keeping 8 loads of 32 bytes in
 *                flight (L1 bypassed, L2 evict-first).
 * sink           device uint32; every CTA XORs the XOR of what it read into
 *                it, so the loads cannot be dropped (its value means nothing).
 * stream         a cudaStream_t (NULL = legacy default stream).
 *
 * Returns PA_ERR_INVALID_ARG for a bad argument (before any launch) and
 * PA_ERR_CUDA when the launch fails. Time it with events on `stream`;
 * bytes / time is the read bandwidth.
 */
pa_status pa_hbm_read_probe(const void* buf, size_t bytes, int ctas_per_sm, uint32_t* sink,
                            void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PA_PROBE_H */
