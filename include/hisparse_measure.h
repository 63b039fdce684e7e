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
 * Decode-step layer work is memory-bound, so the stand-in is a bf16
 * elementwise stream: `passes` times over `buf` (device, `bytes` bytes of
 * bf16, a multiple of 16, 16-byte aligned) it sets y <- 0.999 y + 0.001
 * (fp32 math, bf16 storage), moving 2 * bytes through HBM per pass.  No
 * tensor cores, no host-link traffic.  Grid: ctas_per_sm CTAs of 256
 * threads per SM, each looping over the buffer, so a caller can leave
 * thread slots and issue bandwidth for other kernels on every SM.
 * Errors: INVALID_ARG, ALIGNMENT, CUDA.
 */
int hisparse_synthetic_compute(void *buf, int64_t bytes, int32_t passes, int32_t ctas_per_sm,
                               void *stream);

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

/*
 * hisparse_link_gather: the miss copy's access pattern without the
 * resolver: for i < n, row i of `dst` (device, n * row_bytes bytes) <- row
 * rows[i] of `src` (pinned host memory mapped into the device address
 * space, rows of row_bytes bytes), 16-byte loads with 8 in flight per
 * thread, `num_ctas` CTAs of 1024 threads (0 = one per SM).  Rows under
 * 1 KB are read as the resolve kernel's miss copy reads them: each warp
 * load covers 512 bytes of the 64-byte-aligned span around one row, lanes
 * outside the row idle, and every thread keeps a rolling window of 8 loads;
 * longer rows are read as consecutive 16-byte chunks.  rows: device
 * int64 [n], each in [0, rows of src) -- the caller guarantees the range;
 * the kernel does not check it.  row_bytes a positive multiple of 16; src
 * and dst 16-byte aligned.  Measures what random rows reach over the host
 * link for a given burst ([Arch] Performance invariants), and reads a pool
 * in random order once at set-up: the first random-order reads of a freshly
 * pinned pool are much slower than later ones, and a sequential read does
 * not remove that.  Errors: INVALID_ARG, ALIGNMENT, CUDA.
 */
int hisparse_link_gather(const void *src, int64_t row_bytes, const int64_t *rows, int64_t n,
                         void *dst, int32_t num_ctas, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* HISPARSE_MEASURE_H */
