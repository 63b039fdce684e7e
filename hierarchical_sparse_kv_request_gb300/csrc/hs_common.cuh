// hs_common.cuh -- types and device helpers shared by the resolver's kernels.
//
// Sources (page title, section):
//   [Guide] "HiSparse: Hierarchical Sparse Attention": Decode Workflow,
//           Shared-index prefetch.
//   [Arch]  "HiSparse local KV offload architecture": Hot lookup and LRU,
//           Performance invariants.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace hs {

constexpr int kStatusOk = 0;
constexpr int kStatusBadIndex = 1;
constexpr int kStatusDuplicate = 2;
constexpr int kStatusBadSeqLen = 3;
constexpr int kStatusBadPosition = 4;
constexpr int kStatusBadResident = 5;
constexpr int kStatusNoHostRow = 6;
constexpr int kStatusCapacity = 7;
constexpr int kStatusCopyTimeout = 8;
constexpr int32_t kResidentFlag = 1 << 30;  // marks a row of the resident pool
// Rows shorter than this many bytes are copied (and gathered by the link
// probe) in 64-byte-aligned spans of 512-byte warp tasks; longer rows as
// consecutive 16-byte chunks.  Measured on GB300: faster for 656-byte rows,
// slower for 1152-byte ones.
constexpr int64_t kAlignedRowsBelow = 1024;

// Hot state of one state-owning layer.  Per request r:
//   tok2slot[host_off[r] + t]  slot holding token t, or -1   (host_cap[r] ints)
//   slot2tok[r*D + s]          token in slot s, or -1
//   last_used[r*D + s]         tick of the last call that selected slot s
//   lru[r*D + i]               the i-th least recently used slot; the list
//                              is kept sorted by (last_used, slot)
//   tick[r]                    ticks of the request's calls so far
struct HotState {
    int32_t *tok2slot;
    int32_t *slot2tok;
    uint32_t *last_used;
    uint16_t *lru;
    uint32_t *tick;
    // Optional (null: not kept): resbits[r*res_words + t/32] bit t%32 is set
    // exactly when token t of request r has a slot (tok2slot >= 0).  Every
    // kernel that changes the maps keeps it; the resolve kernel stages a
    // request's row to tell misses from hits before the slots are known.
    uint32_t *resbits;
    int32_t res_words;   // words per request row (a multiple of 4)
};

// Storage of one layer: the pinned host pool as seen from the device and
// the device hot buffer.
struct LayerStore {
    const uint8_t *host;  // [host rows][B] (device-visible pinned memory)
    uint8_t *dev;         // [R][D][B]
};

// host_off[r] is request r's first token->slot entry.  Without a paged pool
// (hb == 0) it is also the first host row of the request's contiguous region
// of host_cap[r] rows.  With a paged pool (hb > 0), token t of request r is
// pool row host_tbl[r * tbl_stride + t / hb] * hb + t % hb, or has no host
// row when that entry is -1; a pool holds pool_rows rows per layer.
struct Geometry {
    int32_t R, k, D;
    int64_t B;             // multiple of 16
    int32_t chunks;        // B / 16
    const int64_t *host_off;  // device [R]
    const int64_t *host_cap;  // device [R]
    const int32_t *host_tbl;  // device [R][tbl_stride] host block ids, or null
    int32_t hb;               // token rows per host block; 0 = no paged pool
    int32_t tbl_stride;       // multiple of 4 (16-byte rows)
    int64_t pool_rows;
};

// Host row of token t of request r (see Geometry), or -1 when its block is
// not reserved.
__device__ __forceinline__ int64_t host_row_of(const Geometry &g, int r, int64_t t)
{
    if (g.hb == 0) return g.host_off[r] + t;
    const int32_t id = g.host_tbl[(int64_t)r * g.tbl_stride + t / g.hb];
    return id < 0 ? -1 : (int64_t)id * g.hb + t % g.hb;
}

// Per-request status word: an error with code c sets bit c; calls that
// succeed leave the word alone, so an error stays visible until the caller
// clears the word (no device readback on the decode path: [Arch]
// Performance invariants).  An atomic OR: the CTAs of several layers of one
// launch, or of overlapping launches, may record into the same word.
__device__ __forceinline__ void record_status(int32_t *status, int r, int code)
{
    atomicOr(status + r, 1 << code);
}

// ---------------------------------------------------------------------------
// Memory access helpers.
// ---------------------------------------------------------------------------

// 16-byte load of pinned host memory through the device's address space.
// The host pool is read-only while a kernel reads it (backups are separate,
// stream-ordered launches), so the non-coherent path is safe; L1 is bypassed
// because every host byte is read once.
__device__ __forceinline__ uint4 ld_host_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_dev_v4(const void *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ void st_v4(void *p, uint4 v)
{
    *reinterpret_cast<uint4 *>(p) = v;
}

// ---------------------------------------------------------------------------
// Block-wide exclusive prefix sum of one uint32 per thread.
// `warp_tot` is shared scratch of NT/32 words.  The function starts and ends
// with a barrier so it can be called back to back.
// ---------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *warp_tot,
                                                         uint32_t &total)
{
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < NW ? warp_tot[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NW) warp_tot[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    total = warp_tot[NW - 1];
    return (warp ? warp_tot[warp - 1] : 0u) + x - v;
}

// ---------------------------------------------------------------------------
// Kernel launchers (defined in the .cu files).
// ---------------------------------------------------------------------------
// How the resolve kernel tells misses from hits (each needs the staged
// slot->token row and more shared memory than the one before):
//   kLookupGather    gather the token->slot map for the top-k row;
//   kLookupInverse   an inverse token->slot table built in shared memory
//                    from the staged slot->token row;
//   kLookupResident  misses first from the request's staged resident-token
//                    bitmap row (HotState::resbits), then the inverse table
//                    for the hits' slots.
constexpr int32_t kLookupGather = 0, kLookupInverse = 1, kLookupResident = 2;

// Byte offsets of the resolve kernel's shared-memory regions (a launch-time
// constant: the host lays the regions out once per launch, so no thread
// recomputes the layout).
struct ResolveSmem {
    uint32_t hit, sel, miss, lru, s2t, inv, res, dup, tbl, chunk, vict, lrow, avict, bar, cnt, stage;
};

struct ResolveLaunch {
    const int32_t *topk;
    const int32_t *seq_lens;
    int32_t *out;
    int32_t *plan_rows;    // may be null
    int32_t *plan_counts;  // may be null
    int32_t *status;
    HotState st;
    LayerStore store;
    Geometry g;
    int32_t max_cap;       // largest host capacity (sizes the miss bitmap)
    bool fused_copy;       // copy the misses in this kernel
    bool stage_s2t;        // stage the slot->token row in shared memory
    int32_t lookup;        // with stage_s2t, kLookup*: how misses and hits are told apart
    const int32_t *resident;  // [R][res_max_blocks] resident block ids, or null
    int32_t res_max_blocks;
    int32_t res_block_size;
    int32_t *deferred;        // [R]: 1 = misses left to the copy grid; null = never defer
    int64_t defer_bytes;      // defer a request whose misses exceed this many bytes
    uint32_t protect_calls;   // slots selected by the last this many calls are kept (0: off)
    int32_t stage_rows;       // misses fetched into shared memory by the bulk-copy engine
                              // (0: none; only with fused_copy and no deferral)
    bool programmatic;        // launch with a programmatic dependency on the stream's
                              // previous kernel (it waits for it on the device)
    bool aligned_rows;        // copy in 64-byte-aligned spans of whole rows (else flat)
    bool wait_late;           // with programmatic: read the inputs and this layer's state
                              // before waiting for the previous kernel (which the host
                              // has checked wrote none of it); wait before writing
    int32_t ncopy;            // copier CTAs per request (a cluster of 1 + ncopy CTAs:
                              // the resolver does no copy); 0: the resolver copies.
                              // Needs fused_copy, no deferral and stage_rows == 0.
    ResolveSmem smem;         // filled by launch_resolve
};

// Shared-memory bytes the resolve kernel needs for this geometry
// (tbl_stride: the host block table row staged per request, 0 = none;
// stage_rows rows of B bytes for the bulk-copy engine).
size_t resolve_smem_bytes(int k, int D, int max_cap, bool stage_s2t, int lookup, int tbl_stride,
                          int stage_rows, int64_t B);
// The most rows the bulk-copy engine can stage within max_smem (at most k).
int resolve_stage_rows(int k, int D, int max_cap, bool stage_s2t, int lookup, int tbl_stride,
                       int64_t B, size_t max_smem);
int resolve_threads();
// Allow every instantiation of the resolve kernel up to `smem` bytes of
// dynamic shared memory (called at handle creation, outside any capture).
cudaError_t resolve_prepare(size_t smem);
// Clusters of `ctas` resolve CTAs with `smem` bytes each that the GPU can
// hold at once (the resolve instantiation for top_k k).
constexpr int kMaxCopyCtas = 4;
cudaError_t resolve_max_clusters(int k, int ctas, size_t smem, int *clusters);
cudaError_t launch_resolve(const ResolveLaunch &a, cudaStream_t s);

constexpr int kMaxReplayLayers = 16;  // layers one replay launch copies for

struct ReplayLaunch {
    const int32_t *plan_rows;
    const int32_t *plan_counts;
    LayerStore store[kMaxReplayLayers];  // the layers to copy into, in order
    int num_layers;
    Geometry g;
    int num_ctas;
    bool programmatic;  // launched right after a resolve (programmatic dependency)
    const int32_t *only_if;  // [R] or null: copy only requests whose entry is nonzero
};
size_t replay_smem_bytes(int R);  // below the 48 KB default for R <= 8192
// Load the replay, backup, prefill and table kernels up front (at handle
// creation, outside any capture), so no first launch waits for a load.
cudaError_t copy_prepare();
cudaError_t launch_replay(const ReplayLaunch &a, cudaStream_t s);

constexpr int kMaxBackupLayers = 16;   // layers one backup launch writes

struct BackupLayer {
    const uint8_t *rows;      // device [R][B]: the layer's new rows
    uint8_t *host;            // layer's pinned pool (device-visible)
    uint8_t *dev;             // layer's hot buffer
    HotState st;              // tok2slot == nullptr for a skip layer
};

struct BackupLaunch {
    BackupLayer layer[kMaxBackupLayers];
    int num_layers;
    const int32_t *positions; // device [R], shared by the layers
    Geometry g;
    int32_t *status;
    bool programmatic;        // as ResolveLaunch::programmatic
};
cudaError_t launch_backup(const BackupLaunch &a, cudaStream_t s);

// Per-layer descriptor, kept in device memory for kernels that walk all
// layers in one launch (prefill).  st.tok2slot == nullptr marks a skip layer.
struct LayerDescDev {
    const uint8_t *host;
    uint8_t *dev;
    HotState st;
};
cudaError_t launch_prefill(const int32_t *seq_lens, const LayerDescDev *layers, int num_layers,
                           const Geometry &g, int32_t *status, cudaStream_t s);

// Runs of host block table entries to set: entry first[i] + j becomes
// value[i] + j for j < len[i], or -1 for every j when value[i] < 0.  Passed
// by value, so a launch needs no host buffer that outlives the call.
constexpr int kTableRuns = 128;
struct TableRuns {
    int32_t n;
    int32_t first[kTableRuns];
    int32_t value[kTableRuns];
    int32_t len[kTableRuns];
};
cudaError_t launch_table_runs(int32_t *table, const TableRuns &runs, cudaStream_t s);

cudaError_t launch_synthetic_compute(void *buf, int64_t bytes, int32_t passes, int32_t ctas,
                                     cudaStream_t s);
cudaError_t launch_link_probe(const void *src, void *dst, int64_t bytes, int num_ctas,
                              cudaStream_t s);
cudaError_t launch_link_gather(const void *src, int64_t row_bytes, const int64_t *rows, int64_t n,
                               void *dst, int num_ctas, cudaStream_t s);

}  // namespace hs
