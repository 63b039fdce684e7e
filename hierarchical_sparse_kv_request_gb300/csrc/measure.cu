// measure.cu -- measurement kernels: a stand-in compute kernel and a host-link
// probe.  Neither is on the decode path.
//
// [Guide] "HiSparse: Hierarchical Sparse Attention", Shared-index prefetch:
// the skip layers' copies overlap the compute of the layers in between; the
// stand-in compute kernel plays that compute (a memory-bound bf16 stream,
// as decode-step layer work is).  [Arch] "HiSparse local KV
// offload architecture", Performance invariants: misses copy directly from
// pinned host memory; the probe measures what SM loads over the host link
// can move.
#include <cuda_bf16.h>

#include "hs_common.cuh"

namespace hs {
namespace {

// y <- 0.999 y + 0.001 over a bf16 buffer, `passes` times: an HBM-bound
// elementwise stream like the memory-bound layer work of a decode step.  Each
// thread moves 16-byte vectors with 4 in flight; fp32 math, bf16 in and out
// (round to nearest even through the cuda_bf16 conversions).
__global__ void __launch_bounds__(256) synthetic_compute_kernel(uint4 *buf, int64_t vecs,
                                                                int32_t passes)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int p = 0; p < passes; ++p) {
        for (int64_t v0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v0 < vecs;
             v0 += stride * 4) {
            uint4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v0 + u * stride < vecs) x[u] = buf[v0 + u * stride];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (v0 + u * stride >= vecs) continue;
                __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&x[u]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float2 f = __bfloat1622float2(h[q]);
                    f.x = fmaf(f.x, 0.999f, 0.001f);
                    f.y = fmaf(f.y, 0.999f, 0.001f);
                    h[q] = __float22bfloat162_rn(f);
                }
                buf[v0 + u * stride] = x[u];
            }
        }
    }
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

// Row gather: dst row i <- src row rows[i], `row_chunks` 16-byte chunks a
// row, 8 chunks in flight per thread.  Idx is the chunk index type: 32-bit
// whenever the chunks fit, so no load waits behind a 64-bit division.
// Two mappings, as the miss copy of the resolve kernel has:
//  - flat: consecutive threads take consecutive chunks, across row
//    boundaries; each thread loads its 8 and then stores them;
//  - aligned (rows under 1 KB): a warp task is 512 bytes of the 64-byte-
//    aligned span around one row, one 16-byte piece per lane (lanes whose
//    piece lies outside the row move nothing), so no 64-byte unit of host
//    memory is split between two warp loads; a rolling window of 8 loads per
//    thread.  Measured on GB300 for ~10,450 random 656-byte rows after an L2
//    flush: 39.1 us against 40.1 us flat.
template <typename Idx>
__global__ void __launch_bounds__(PROBE_NT) link_gather_kernel(const uint8_t *src, uint8_t *dst,
                                                               const int64_t *rows, Idx total,
                                                               Idx row_chunks)
{
    const Idx stride = (Idx)gridDim.x * PROBE_NT;
    const int64_t B = (int64_t)row_chunks * 16;
    for (Idx e = (Idx)blockIdx.x * PROBE_NT + threadIdx.x; e < total;
         e += stride * PROBE_UNROLL) {
        uint4 v[PROBE_UNROLL];
#pragma unroll
        for (int u = 0; u < PROBE_UNROLL; ++u) {
            const Idx ee = e + (Idx)u * stride;
            if (ee < total) {
                const Idx i = ee / row_chunks, c = ee - i * row_chunks;
                v[u] = ld_host_v4(src + rows[i] * B + (int64_t)c * 16);
            }
        }
#pragma unroll
        for (int u = 0; u < PROBE_UNROLL; ++u) {
            const Idx ee = e + (Idx)u * stride;
            if (ee < total) st_v4(dst + (int64_t)ee * 16, v[u]);
        }
    }
}

// Warp tasks of the aligned mapping: task e is the h-th 512 bytes of the
// aligned span around row q = e / H (H tasks a row).
template <typename Idx>
struct SpanTask {
    const uint8_t *src;
    const int64_t *rows;
    int64_t B;
    Idx first, stride, limit;
    int H, CH, lane;
    int64_t items;
    // row q and chunk c of the thread's n-th task; false if it moves nothing
    __device__ __forceinline__ bool at(int64_t n, Idx &q, int &c) const
    {
        if (n >= items) return false;
        const Idx e = first + (Idx)n * stride;
        q = e / (Idx)H;
        const int h = (int)(e - q * (Idx)H);
        const int delta = (int)((reinterpret_cast<uintptr_t>(src + rows[q] * B) >> 4) & 3);
        c = h * 32 + lane - delta;
        return c >= 0 && c < CH;
    }
};

template <typename Idx>
__global__ void __launch_bounds__(PROBE_NT) link_gather_aligned_kernel(const uint8_t *src, uint8_t *dst,
                                                                       const int64_t *rows, Idx n,
                                                                       int row_chunks)
{
    SpanTask<Idx> m;
    m.src = src;
    m.rows = rows;
    m.B = (int64_t)row_chunks * 16;
    m.CH = row_chunks;
    m.H = (row_chunks + 3 + 31) / 32;   // a span reaches 3 chunks before the row
    m.lane = (int)(threadIdx.x & 31);
    m.first = (Idx)((blockIdx.x * PROBE_NT + threadIdx.x) >> 5);
    m.stride = (Idx)(gridDim.x * (PROBE_NT / 32));
    m.limit = n * (Idx)m.H;
    m.items = m.limit > m.first ? ((int64_t)m.limit - m.first + m.stride - 1) / m.stride : 0;
    uint4 pv[PROBE_UNROLL];
#pragma unroll
    for (int u = 0; u < PROBE_UNROLL; ++u) {
        Idx q;
        int c;
        if (m.at(u, q, c)) pv[u] = ld_host_v4(src + rows[q] * m.B + c * 16);
    }
    for (int64_t n0 = 0; n0 < m.items; n0 += PROBE_UNROLL) {
#pragma unroll
        for (int u = 0; u < PROBE_UNROLL; ++u) {
            Idx q;
            int c;
            if (m.at(n0 + u, q, c)) st_v4(dst + (int64_t)q * m.B + c * 16, pv[u]);
            if (m.at(n0 + u + PROBE_UNROLL, q, c)) pv[u] = ld_host_v4(src + rows[q] * m.B + c * 16);
        }
    }
}

}  // namespace

cudaError_t launch_link_gather(const void *src, int64_t row_bytes, const int64_t *rows, int64_t n,
                               void *dst, int num_ctas, cudaStream_t s)
{
    const int64_t chunks = row_bytes / 16;
    const uint8_t *sp = static_cast<const uint8_t *>(src);
    uint8_t *dp = static_cast<uint8_t *>(dst);
    if (row_bytes < kAlignedRowsBelow) {
        // tasks: n * H; the last task index, plus one stride, must not wrap
        const int64_t H = (chunks + 3 + 31) / 32;
        const int64_t reach = n * H + (int64_t)num_ctas * (PROBE_NT / 32) * (PROBE_UNROLL + 1);
        if (reach <= (int64_t)UINT32_MAX)
            link_gather_aligned_kernel<uint32_t><<<num_ctas, PROBE_NT, 0, s>>>(sp, dp, rows, (uint32_t)n,
                                                                               (int)chunks);
        else
            link_gather_aligned_kernel<int64_t><<<num_ctas, PROBE_NT, 0, s>>>(sp, dp, rows, n, (int)chunks);
        return cudaGetLastError();
    }
    const int64_t total = n * chunks;
    // the 32-bit kernel's last stride step must not wrap either
    const int64_t reach = total + (int64_t)num_ctas * PROBE_NT * PROBE_UNROLL;
    if (reach <= (int64_t)UINT32_MAX)
        link_gather_kernel<uint32_t><<<num_ctas, PROBE_NT, 0, s>>>(sp, dp, rows, (uint32_t)total,
                                                                   (uint32_t)chunks);
    else
        link_gather_kernel<int64_t><<<num_ctas, PROBE_NT, 0, s>>>(sp, dp, rows, total, chunks);
    return cudaGetLastError();
}

cudaError_t launch_synthetic_compute(void *buf, int64_t bytes, int32_t passes, int32_t ctas,
                                     cudaStream_t s)
{
    synthetic_compute_kernel<<<ctas, 256, 0, s>>>(static_cast<uint4 *>(buf), bytes / 16, passes);
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
