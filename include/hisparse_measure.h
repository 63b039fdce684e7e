/*
 * hisparse_measure.h -- measurement kernels that sit beside the resolver in
 * libhisparse.so.  They are not part of the decode path; the benchmark and
 * tests use them to set up the conditions the pages describe.
 *
 * Sources:
 *   [Guide] "HiSparse: Hierarchical Sparse Attention" (SGLang user guide),
 *           Shared-index prefetch: skip layers' host-to-device copies
 *           overlap the compute of the layers in between.
 *   [Arch]  "HiSparse local KV offload architecture", Performance
 *           invariants: hot misses copy directly from registered pinned
 *           host memory.
 * Return codes are those of hisparse.h.
 */
#ifndef HISPARSE_MEASURE_H
#define HISPARSE_MEASURE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * hisparse_synthetic_compute: a stand-in for the compute of the layers
 * between an anchor and its skip layers ([Guide] Shared-index prefetch).
 * Each of `num_threads` threads (rounded up to whole 256-thread CTAs) runs
 * `iters` dependent fp32 fused multiply-adds on one element of `buf` (device
 * float [n], n >= num_threads) and writes it back; no tensor cores, no
 * memory traffic to speak of.  The grid is ceil(num_threads / 256) CTAs of
 * 256 threads, so a caller can leave room on every SM for other kernels.
 * Errors: INVALID_ARG.
 */
int hisparse_synthetic_compute(float *buf, int64_t n, int32_t num_threads,
                               int32_t iters, void *stream);

/*
 * hisparse_link_probe: measure what SM loads and stores over the host link
 * can move ([Arch] Performance invariants: misses copy directly from pinned
 * host memory).  Copies `bytes` (a multiple of 16) from `src` to `dst` with
 * 16-byte vector loads and stores, `num_ctas` CTAs of 1024 threads (0 = one
 * per SM).  For host-to-device, `src` is a pinned host pointer mapped into
 * the device address space (cudaHostAlloc with cudaHostAllocMapped, as
 * torch's pin_memory gives on this platform) and `dst` device memory; for
 * device-to-host, the reverse.  Both must be 16-byte aligned.
 * Errors: INVALID_ARG, ALIGNMENT.
 */
int hisparse_link_probe(const void *src, void *dst, int64_t bytes, int32_t num_ctas,
                        void *stream);

#ifdef __cplusplus
}
#endif
#endif /* HISPARSE_MEASURE_H */
