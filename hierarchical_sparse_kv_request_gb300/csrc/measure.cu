// measure.cu -- measurement kernels: a stand-in compute kernel and a host-link
// probe.  Neither is on the decode path.
//
// [Guide] "HiSparse: Hierarchical Sparse Attention", Shared-index prefetch:
// the skip layers' copies overlap the compute of the layers in between; the
// stand-in compute kernel plays that compute.  [Arch] "HiSparse local KV
// offload architecture", Performance invariants: misses copy directly from
// pinned host memory; the probe measures what SM loads over the host link
// can move.
#include "hs_common.cuh"

namespace hs {
namespace {

__global__ void __launch_bounds__(256) synthetic_compute_kernel(float *buf, int32_t n,
                                                                int32_t iters)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float x = buf[i], y = 1.0f + 1e-7f * (float)(i & 1023);
    // four independent chains keep the FMA pipe busy without memory traffic
    float a0 = x, a1 = x + 1.f, a2 = x + 2.f, a3 = x + 3.f;
    for (int it = 0; it < iters; ++it) {
        a0 = fmaf(a0, y, 1e-6f);
        a1 = fmaf(a1, y, -1e-6f);
        a2 = fmaf(a2, y, 2e-6f);
        a3 = fmaf(a3, y, -2e-6f);
    }
    buf[i] = a0 + a1 + a2 + a3;
}

constexpr int PROBE_NT = 1024;
constexpr int PROBE_UNROLL = 8;

__global__ void __launch_bounds__(PROBE_NT) link_probe_kernel(const uint8_t *src, uint8_t *dst,
                                                              int64_t chunks)
{
    const int64_t stride = (int64_t)gridDim.x * PROBE_NT;
    for (int64_t e = (int64_t)blockIdx.x * PROBE_NT + threadIdx.x; e < chunks;
         e += stride * PROBE_UNROLL) {
        uint4 v[PROBE_UNROLL];
#pragma unroll
        for (int u = 0; u < PROBE_UNROLL; ++u) {
            const int64_t ee = e + u * stride;
            if (ee < chunks) v[u] = ld_host_v4(src + ee * 16);
        }
#pragma unroll
        for (int u = 0; u < PROBE_UNROLL; ++u) {
            const int64_t ee = e + u * stride;
            if (ee < chunks) st_v4(dst + ee * 16, v[u]);
        }
    }
}

}  // namespace

cudaError_t launch_synthetic_compute(float *buf, int32_t num_threads, int32_t iters,
                                     cudaStream_t s)
{
    const int blocks = (num_threads + 255) / 256;
    synthetic_compute_kernel<<<blocks, 256, 0, s>>>(buf, num_threads, iters);
    return cudaGetLastError();
}

cudaError_t launch_link_probe(const void *src, void *dst, int64_t bytes, int num_ctas,
                              cudaStream_t s)
{
    link_probe_kernel<<<num_ctas, PROBE_NT, 0, s>>>(static_cast<const uint8_t *>(src),
                                                    static_cast<uint8_t *>(dst), bytes / 16);
    return cudaGetLastError();
}

}  // namespace hs
