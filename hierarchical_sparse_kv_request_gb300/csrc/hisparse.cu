// hisparse.cu -- host side of the C ABI declared in include/hisparse.h and
// include/hisparse_measure.h: layout validation, allocation of the pinned host
// pool, hot buffers and hot state, and kernel launches.  No entry point that
// takes a stream synchronises or reads device data back.
//
// [Arch] "HiSparse local KV offload architecture", Ownership: the per-cache
// runtime owns the host/hot storage, the hot-row map and the LRU; Performance
// invariants: no device readback, one kernel per call.  [Guide] "HiSparse:
// Hierarchical Sparse Attention", HiSparse Config Parameters: top_k,
// device_buffer_size, host_to_device_ratio, swap_in_block_size.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "hisparse.h"
#include "hisparse_measure.h"
#include "hs_common.cuh"

// Scratch of the allocation-free swap-in (hisparse_swap_in_noalloc): the miss
// plan that its resolve grid hands to its copy grid lives in this fixed array
// instead of device memory obtained from cudaMalloc.  Each GPU that loads the
// library holds its own copy (HISPARSE_NOALLOC_SCRATCH_BYTES) until the
// process exits.  Layout: (host slot, slot) pairs of request r at
// [r * k * 2, ...), then R miss counts after the pairs region.  Host code only
// sees a stand-in for the symbol; hisparse_create looks up the device address
// of the array with the handle's device current and keeps it in the handle.
static __device__ __align__(256) int32_t g_noalloc_scratch[HISPARSE_NOALLOC_SCRATCH_BYTES / 4];

struct hisparse_handle {
    int device = 0;
    int num_sms = 0;
    int32_t R = 0, L = 0, k = 0, D = 0, ratio = 0;
    int64_t B = 0;
    int32_t chunks = 0;
    std::vector<int32_t> anchor;
    std::vector<int64_t> cap, off;
    int64_t total_cap = 0, max_cap = 0;
    uint8_t *host_pool = nullptr;      // pinned [L][layer_rows()][B]
    uint8_t *host_pool_dev = nullptr;  // the same memory, device address
    uint8_t *dev_buf = nullptr;        // [L][R][D][B]
    int64_t *d_off = nullptr, *d_cap = nullptr;
    int32_t *d_status = nullptr;
    int32_t *d_zero = nullptr;         // [R] zeros, for the initial prefill
    std::vector<hs::HotState> state;   // per layer; tok2slot null for skip layers
    hs::LayerDescDev *d_layers = nullptr;
    int32_t *d_plan_rows = nullptr, *d_plan_counts = nullptr;  // split-copy plan
    int32_t *d_deferred = nullptr;     // [R] requests left to the copy grid (auto mode)
    int32_t *noalloc_scratch = nullptr; // device address of g_noalloc_scratch on this device
    int32_t copy_mode = HISPARSE_COPY_FUSED;
    int32_t protect_calls = 0;  // slots selected by the last this many calls are kept
    int32_t max_stage_rows = 0; // miss rows per request the resolve CTA's shared memory holds
    int32_t stage_rows = 0;     // of those, how many the fused copy stages (set_stage_rows)
    bool programmatic = false;  // swap-ins and backups launched with a programmatic dependency
    int32_t copy_ctas = 1;      // CTAs per request that run a fused-copy swap-in (1: the
                                // resolving CTA copies; more: a cluster, see set_copy_ctas)
    // The handle's last kernel launch: its stream, and the layers whose hot
    // state, device rows or host rows it wrote (all of them after a prefill,
    // a host block table edit or a state write).  A programmatic swap-in on
    // the same stream whose layer that launch left alone reads before it
    // waits (ResolveLaunch::wait_late).
    bool last_known = false;
    cudaStream_t last_stream = nullptr;
    bool last_all = true;
    std::vector<uint8_t> last_wrote;   // [L]
    bool stage_s2t = false;   // resolve kernel stages the slot->token row
    int32_t lookup = hs::kLookupGather;  // ... and tells misses from hits this way

    // Paged host pool (hb > 0): pool_blocks blocks of hb rows per layer,
    // handed to requests by hisparse_host_reserve.  `tbl` is the host copy of
    // the block table [R][tbl_stride] (the device copy, d_tbl, follows it in
    // stream order); a request's reserved blocks are the first nblocks[r]
    // entries of its row.
    int32_t hb = 0;
    int32_t pool_blocks = 0;
    int32_t tbl_stride = 0;
    int64_t pool_rows = 0;
    std::vector<int32_t> tbl;
    std::vector<int32_t> nblocks;
    std::vector<uint64_t> used;        // one bit per block; bits past the pool are set
    int32_t free_blocks = 0;
    int32_t lowest_free = 0;           // no block below this id is free
    int32_t *d_tbl = nullptr;

    // Guard bands (HISPARSE_DEBUG_GUARDS=1 at create): every device array
    // is allocated with kGuardBytes of a known pattern on each side, and
    // hisparse_check_guards reports arrays whose bands were overwritten.
    bool guards = false;
    std::vector<std::pair<uint8_t *, size_t>> guarded;   // (array, bytes)

    int64_t layer_rows() const { return hb ? pool_rows : total_cap; }
};

namespace {

// Auto copy mode: in batches of fewer than kAutoDeferBelowRequests requests,
// a request whose misses exceed kAutoDeferBytes leaves them to the full-GPU
// copy grid (one SM moves such a volume several times slower).  From that
// batch size on, the CTAs of the batch already keep the host link busy, and
// deferring only moves every copy behind the resolve grid (measured on
// GB300: a cold call of 1 request 76 -> 29 us, of 32 requests 170 -> 191 us).
constexpr int64_t kAutoDeferBytes = 256 << 10;
constexpr int kAutoDeferBelowRequests = 8;

hs::Geometry geometry(const hisparse_handle *h)
{
    hs::Geometry g;
    g.R = h->R;
    g.k = h->k;
    g.D = h->D;
    g.B = h->B;
    g.chunks = h->chunks;
    g.host_off = h->d_off;
    g.host_cap = h->d_cap;
    g.host_tbl = h->d_tbl;
    g.hb = h->hb;
    g.tbl_stride = h->tbl_stride;
    g.pool_rows = h->pool_rows;
    return g;
}

hs::LayerStore layer_store(const hisparse_handle *h, int layer)
{
    hs::LayerStore s;
    s.host = h->host_pool_dev + (int64_t)layer * h->layer_rows() * h->B;
    s.dev = h->dev_buf + (int64_t)layer * h->R * h->D * h->B;
    return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launching calls must run with the handle's device current.
bool on_own_device(const hisparse_handle *h)
{
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == h->device;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? HISPARSE_OK : HISPARSE_ERR_CUDA; }


void note_launch_all(hisparse_handle *h, cudaStream_t s)
{
    h->last_known = true;
    h->last_stream = s;
    h->last_all = true;
}

void note_launch_layers(hisparse_handle *h, cudaStream_t s, const int32_t *layers, int n)
{
    h->last_known = true;
    h->last_stream = s;
    h->last_all = false;
    h->last_wrote.assign(h->L, 0);
    for (int i = 0; i < n; ++i) h->last_wrote[layers[i]] = 1;
}

// True if the handle's last launch was on stream s and wrote nothing of
// `layer`: a kernel launched now, programmatically behind it, may read that
// layer's state and rows before the last launch has completed.
bool left_layer_alone(const hisparse_handle *h, cudaStream_t s, int32_t layer)
{
    return h->last_known && !h->last_all && h->last_stream == s && !h->last_wrote[layer];
}

// Dynamic shared memory of the handle's resolve launches without staged rows.
size_t resolve_smem(const hisparse_handle *h)
{
    return hs::resolve_smem_bytes(h->k, h->D, (int)h->max_cap, h->stage_s2t, h->lookup,
                                  h->hb ? h->tbl_stride : 0, 0, h->B);
}

constexpr size_t kGuardBytes = 4096;
constexpr unsigned char kGuardByte = 0xA5;

template <class T>
cudaError_t dev_alloc(hisparse_handle *h, T **p, size_t count)
{
    const size_t bytes = count * sizeof(T);
    if (!h->guards) return cudaMalloc(reinterpret_cast<void **>(p), bytes);
    uint8_t *base = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&base), bytes + 2 * kGuardBytes);
    if (e != cudaSuccess) return e;
    e = cudaMemset(base, kGuardByte, bytes + 2 * kGuardBytes);
    *p = reinterpret_cast<T *>(base + kGuardBytes);
    h->guarded.emplace_back(base + kGuardBytes, bytes);
    return e;
}

void dev_free(const hisparse_handle *h, void *p)
{
    if (!p) return;
    cudaFree(h->guards ? static_cast<uint8_t *>(p) - kGuardBytes : p);
}

void release(hisparse_handle *h)
{
    if (!h) return;
    for (auto &st : h->state) {
        dev_free(h, st.tok2slot);
        dev_free(h, st.slot2tok);
        dev_free(h, st.last_used);
        dev_free(h, st.lru);
        dev_free(h, st.tick);
        dev_free(h, st.resbits);
    }
    dev_free(h, h->d_layers);
    dev_free(h, h->d_plan_rows);
    dev_free(h, h->d_plan_counts);
    dev_free(h, h->d_deferred);
    dev_free(h, h->d_status);
    dev_free(h, h->d_zero);
    dev_free(h, h->d_off);
    dev_free(h, h->d_cap);
    dev_free(h, h->d_tbl);
    dev_free(h, h->dev_buf);
    if (h->host_pool) cudaFreeHost(h->host_pool - (h->guards ? kGuardBytes : 0));
    delete h;
}

// Checks of a layout; `paged` drops the bound on summed capacities (a paged
// pool bounds the rows themselves).
int validate_layout(const hisparse_layout *l, bool paged)
{
    if (l->num_requests < 1 || l->num_layers < 1 || l->row_bytes <= 0 || l->top_k < 1 ||
        l->device_buffer_size < 1 || l->host_to_device_ratio < 1 || l->swap_in_block_size < 0)
        return HISPARSE_ERR_LAYOUT;
    if (l->row_bytes % 16 != 0) return HISPARSE_ERR_LAYOUT;
    if (l->top_k > l->device_buffer_size) return HISPARSE_ERR_LAYOUT;
    if (!l->host_capacity) return HISPARSE_ERR_INVALID_ARG;
    if (l->num_requests > HISPARSE_MAX_REQUESTS || l->top_k > HISPARSE_MAX_TOP_K ||
        l->device_buffer_size > HISPARSE_MAX_DEVICE_BUFFER)
        return HISPARSE_ERR_UNSUPPORTED;
    // a call's 16-byte miss chunks per request are counted in 32 bits
    if ((int64_t)l->top_k * (l->row_bytes / 16) > INT32_MAX) return HISPARSE_ERR_UNSUPPORTED;
    bool any_owner = false;
    for (int i = 0; i < l->num_layers; ++i) {
        const int a = l->anchor_of_layer ? l->anchor_of_layer[i] : -1;
        if (a < -1 || a >= l->num_layers || a == i) return HISPARSE_ERR_LAYOUT;
        if (a >= 0 && l->anchor_of_layer[a] != -1) return HISPARSE_ERR_LAYOUT;
        any_owner |= a == -1;
    }
    if (!any_owner) return HISPARSE_ERR_LAYOUT;
    int64_t total = 0;
    for (int r = 0; r < l->num_requests; ++r) {
        const int64_t c = l->host_capacity[r];
        if (c < 0) return HISPARSE_ERR_LAYOUT;
        if (c > HISPARSE_MAX_HOST_CAPACITY) return HISPARSE_ERR_UNSUPPORTED;
        total += c;
    }
    if (total < 1) return HISPARSE_ERR_LAYOUT;
    const int64_t limit = (int64_t)l->host_to_device_ratio * l->num_requests * l->device_buffer_size;
    if (!paged && total > limit) return HISPARSE_ERR_CAPACITY;
    return HISPARSE_OK;
}

// Lowest free block of the pool (the caller checked free_blocks > 0).
int32_t take_lowest_free(hisparse_handle *h)
{
    size_t w = (size_t)h->lowest_free / 64;
    while (h->used[w] == ~0ull) ++w;
    const int32_t id = (int32_t)(w * 64 + __builtin_ctzll(~h->used[w]));
    h->used[w] |= 1ull << (id % 64);
    --h->free_blocks;
    h->lowest_free = id + 1;
    return id;
}

void give_back(hisparse_handle *h, int32_t id)
{
    h->used[id / 64] &= ~(1ull << (id % 64));
    ++h->free_blocks;
    h->lowest_free = std::min(h->lowest_free, id);
}

// Take back a block given back by a release that is being undone.
void retake(hisparse_handle *h, int32_t id)
{
    h->used[id / 64] |= 1ull << (id % 64);
    --h->free_blocks;
}

// First table entry of request r (the table is at most 2^31 entries: its
// row must fit in the resolve kernel's shared memory).
int32_t tbl_row(const hisparse_handle *h, int32_t r) { return r * h->tbl_stride; }

// Table edits, merged into runs and applied on the stream, 128 runs a launch.
struct RunList {
    std::vector<int32_t> first, value, len;
    void add(int32_t idx, int32_t id)
    {
        const size_t n = first.size();
        if (n && value[n - 1] >= 0 && first[n - 1] + len[n - 1] == idx &&
            value[n - 1] + len[n - 1] == id) {
            ++len[n - 1];
            return;
        }
        first.push_back(idx);
        value.push_back(id);
        len.push_back(1);
    }
    void clear_range(int32_t idx, int32_t count)
    {
        first.push_back(idx);
        value.push_back(-1);
        len.push_back(count);
    }
    cudaError_t apply(int32_t *table, cudaStream_t s) const
    {
        for (size_t i0 = 0; i0 < first.size(); i0 += hs::kTableRuns) {
            hs::TableRuns tr;
            tr.n = (int32_t)std::min(first.size() - i0, (size_t)hs::kTableRuns);
            for (int32_t i = 0; i < tr.n; ++i) {
                tr.first[i] = first[i0 + i];
                tr.value[i] = value[i0 + i];
                tr.len[i] = len[i0 + i];
            }
            const cudaError_t e = hs::launch_table_runs(table, tr, s);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
};

}  // namespace

extern "C" {

int hisparse_version(void) { return 201; }

const char *hisparse_error_string(int code)
{
    switch (code) {
    case HISPARSE_OK: return "ok";
    case HISPARSE_ERR_INVALID_ARG: return "invalid argument";
    case HISPARSE_ERR_LAYOUT: return "inconsistent layout";
    case HISPARSE_ERR_CAPACITY:
        return "host capacity exceeds host_to_device_ratio * R * D (or too few free host blocks)";
    case HISPARSE_ERR_LAYER: return "layer out of range or without hot state";
    case HISPARSE_ERR_CUDA: return "CUDA runtime error";
    case HISPARSE_ERR_NO_MEMORY: return "out of pinned or device memory";
    case HISPARSE_ERR_UNSUPPORTED: return "size beyond this library's limits";
    case HISPARSE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    default: return "unknown error";
    }
}

}  // extern "C"

namespace {

int create_impl(const hisparse_layout *layout, int32_t host_block_tokens, hisparse_t *out)
{
    if (!out) return HISPARSE_ERR_INVALID_ARG;
    *out = nullptr;
    if (!layout) return HISPARSE_ERR_INVALID_ARG;
    const bool paged = host_block_tokens != 0;
    int rc = validate_layout(layout, paged);
    if (rc != HISPARSE_OK) return rc;
    int64_t pool_blocks = 0;
    if (paged) {
        if (host_block_tokens < 1) return HISPARSE_ERR_LAYOUT;
        if (host_block_tokens > HISPARSE_MAX_HOST_BLOCK_TOKENS) return HISPARSE_ERR_UNSUPPORTED;
        // [Arch] Ownership: the budget is rounded down to whole host blocks
        pool_blocks = (int64_t)layout->host_to_device_ratio * layout->num_requests *
                      layout->device_buffer_size / host_block_tokens;
        if (pool_blocks < 1) return HISPARSE_ERR_CAPACITY;
        if (pool_blocks * host_block_tokens > INT32_MAX) return HISPARSE_ERR_UNSUPPORTED;
    }

    hisparse_handle *h = new (std::nothrow) hisparse_handle;
    if (!h) return HISPARSE_ERR_NO_MEMORY;
    const char *guards = std::getenv("HISPARSE_DEBUG_GUARDS");
    h->guards = guards && guards[0] == '1';
    h->R = layout->num_requests;
    h->L = layout->num_layers;
    h->k = layout->top_k;
    h->D = layout->device_buffer_size;
    h->B = layout->row_bytes;
    h->chunks = (int32_t)(h->B / 16);
    h->ratio = layout->host_to_device_ratio;
    h->anchor.resize(h->L);
    for (int i = 0; i < h->L; ++i) h->anchor[i] = layout->anchor_of_layer ? layout->anchor_of_layer[i] : -1;
    h->cap.assign(layout->host_capacity, layout->host_capacity + h->R);
    h->off.resize(h->R);
    for (int r = 0; r < h->R; ++r) {
        h->off[r] = h->total_cap;
        h->total_cap += h->cap[r];
        if (h->cap[r] > h->max_cap) h->max_cap = h->cap[r];
    }
    if (paged) {
        h->hb = host_block_tokens;
        h->pool_blocks = (int32_t)pool_blocks;
        h->pool_rows = pool_blocks * host_block_tokens;
        const int64_t per_req = (h->max_cap + h->hb - 1) / h->hb;
        h->tbl_stride = (int32_t)std::max<int64_t>(4, (per_req + 3) / 4 * 4);
        h->tbl.assign((size_t)h->R * h->tbl_stride, -1);
        h->nblocks.assign(h->R, 0);
        h->used.assign((size_t)(pool_blocks + 63) / 64, 0ull);
        for (int64_t b = pool_blocks; b < (int64_t)h->used.size() * 64; ++b)
            h->used[b / 64] |= 1ull << (b % 64);
        h->free_blocks = h->pool_blocks;
    }

    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        release(h);
        return HISPARSE_ERR_CUDA;
    }
    int max_smem = 0;
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device);
    if (hs::resolve_smem_bytes(h->k, h->D, (int)h->max_cap, false, hs::kLookupGather, h->tbl_stride,
                               0, h->B) >
            (size_t)max_smem ||
        hs::replay_smem_bytes(h->R) > (size_t)max_smem) {
        release(h);
        return HISPARSE_ERR_UNSUPPORTED;
    }
    // The slot->token row rides in shared memory when it fits, and with it,
    // when that fits too, an inverse table over the request's tokens: the
    // hit lookup then needs no gather of the token->slot map, whose round
    // trip otherwise sits between the top-k row and the first host loads;
    // and when the request's resident-token bitmap row fits as well, the
    // misses are known from it before any slot (hs::kLookup*).  The shared
    // memory left over stages miss rows for the bulk-copy engine.
    auto fits = [&](bool s2t, int lookup) {
        return hs::resolve_smem_bytes(h->k, h->D, (int)h->max_cap, s2t, lookup, h->tbl_stride, 0,
                                      h->B) <= (size_t)max_smem;
    };
    h->stage_s2t = fits(true, hs::kLookupGather);
    h->lookup = !h->stage_s2t ? hs::kLookupGather
                : fits(true, hs::kLookupResident) ? hs::kLookupResident
                : fits(true, hs::kLookupInverse) ? hs::kLookupInverse
                : hs::kLookupGather;
    h->max_stage_rows = hs::resolve_stage_rows(h->k, h->D, (int)h->max_cap, h->stage_s2t,
                                               h->lookup, h->tbl_stride, h->B, (size_t)max_smem);
    h->stage_rows = 0;          // measured: staging is slower on the benchmarked shapes
    if (hs::resolve_prepare((size_t)max_smem) != cudaSuccess || hs::copy_prepare() != cudaSuccess) {
        release(h);
        return HISPARSE_ERR_CUDA;
    }
    // Copier CTAs by default: the most (up to 4 per request) for which the
    // GPU holds every request's cluster at once.  Measured on decode_40k
    // (32 requests): 4 CTAs per request ~1.5 us faster per call than 1.
    for (int32_t c = hs::kMaxCopyCtas; c > 1; --c) {
        int n = 0;
        if (hs::resolve_max_clusters(h->k, c, resolve_smem(h), &n) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (n >= h->R) {
            h->copy_ctas = c;
            break;
        }
    }
    // The allocation-free swap-in's scratch array: looking its address up
    // here, with the handle's device current, also loads the module that holds
    // it (CUDA loads modules lazily by default), so that call itself never
    // loads, looks up or allocates anything.
    {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            release(h);
            return HISPARSE_ERR_CUDA;
        }
        h->noalloc_scratch = static_cast<int32_t *>(p);
    }

    // Pinned host pool, mapped into the device address space.  A test hook
    // makes this allocation fail on request so the failure path is exercised.
    const size_t pool_bytes = (size_t)h->L * h->layer_rows() * h->B;
    const size_t band = h->guards ? kGuardBytes : 0;   // guard bands, see hisparse_check_guards
    const char *fail = std::getenv("HISPARSE_TEST_FAIL_PINNED_ALLOC");
    uint8_t *pool_base = nullptr;
    if ((fail && fail[0] == '1') ||
        cudaHostAlloc(reinterpret_cast<void **>(&pool_base), pool_bytes + 2 * band,
                      cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
        cudaGetLastError();
        release(h);
        return HISPARSE_ERR_NO_MEMORY;
    }
    h->host_pool = pool_base + band;
    std::memset(pool_base, kGuardByte, band);
    std::memset(h->host_pool, 0, pool_bytes);
    std::memset(h->host_pool + pool_bytes, kGuardByte, band);
    uint8_t *pool_dev = nullptr;
    if (cudaHostGetDevicePointer(reinterpret_cast<void **>(&pool_dev), pool_base, 0) != cudaSuccess) {
        release(h);
        return HISPARSE_ERR_CUDA;
    }
    h->host_pool_dev = pool_dev + band;

    const size_t buf_bytes = (size_t)h->L * h->R * h->D * h->B;
    const size_t RD = (size_t)h->R * h->D;
    bool ok = dev_alloc(h, &h->dev_buf, buf_bytes) == cudaSuccess &&
              dev_alloc(h, &h->d_off, (size_t)h->R) == cudaSuccess &&
              dev_alloc(h, &h->d_cap, (size_t)h->R) == cudaSuccess &&
              dev_alloc(h, &h->d_status, (size_t)h->R) == cudaSuccess &&
              dev_alloc(h, &h->d_zero, (size_t)h->R) == cudaSuccess &&
              dev_alloc(h, &h->d_layers, (size_t)h->L) == cudaSuccess &&
              dev_alloc(h, &h->d_plan_rows, (size_t)h->R * h->k * 2) == cudaSuccess &&
              dev_alloc(h, &h->d_plan_counts, (size_t)h->R) == cudaSuccess &&
              dev_alloc(h, &h->d_deferred, (size_t)h->R) == cudaSuccess &&
              (!paged || dev_alloc(h, &h->d_tbl, h->tbl.size()) == cudaSuccess);
    h->state.assign(h->L, hs::HotState{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0});
    // The resident-token bitmap is kept where the resolve kernel reads it:
    // with the inverse-table lookup.
    const int32_t res_words = (int32_t)(((h->max_cap + 31) / 32 + 3) / 4 * 4);
    for (int l = 0; ok && l < h->L; ++l) {
        if (h->anchor[l] >= 0) continue;
        hs::HotState &st = h->state[l];
        ok = dev_alloc(h, &st.tok2slot, (size_t)h->total_cap) == cudaSuccess &&
             dev_alloc(h, &st.slot2tok, RD) == cudaSuccess &&
             dev_alloc(h, &st.last_used, RD) == cudaSuccess &&
             dev_alloc(h, &st.lru, RD) == cudaSuccess &&
             dev_alloc(h, &st.tick, (size_t)h->R) == cudaSuccess &&
             (h->lookup < hs::kLookupResident ||
              dev_alloc(h, &st.resbits, (size_t)h->R * res_words) == cudaSuccess);
        if (st.resbits) st.res_words = res_words;
    }
    if (!ok) {
        cudaGetLastError();
        release(h);
        return HISPARSE_ERR_NO_MEMORY;
    }

    std::vector<hs::LayerDescDev> desc(h->L);
    for (int l = 0; l < h->L; ++l) {
        const hs::LayerStore s = layer_store(h, l);
        desc[l].host = s.host;
        desc[l].dev = s.dev;
        desc[l].st = h->state[l];
    }
    cudaError_t e = cudaMemcpy(h->d_off, h->off.data(), sizeof(int64_t) * h->R, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(h->d_cap, h->cap.data(), sizeof(int64_t) * h->R, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(h->d_layers, desc.data(), sizeof(hs::LayerDescDev) * h->L, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(h->dev_buf, 0, buf_bytes);
    if (e == cudaSuccess) e = cudaMemset(h->d_zero, 0, sizeof(int32_t) * h->R);
    if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(int32_t) * h->R);
    if (e == cudaSuccess) e = cudaMemset(h->d_plan_counts, 0, sizeof(int32_t) * h->R);
    if (e == cudaSuccess) e = cudaMemset(h->d_deferred, 0, sizeof(int32_t) * h->R);
    if (e == cudaSuccess && paged) e = cudaMemset(h->d_tbl, 0xFF, sizeof(int32_t) * h->tbl.size());
    // empty hot state: seq_len 0 everywhere (maps -1, LRU in slot order, ticks 0)
    if (e == cudaSuccess) e = hs::launch_prefill(h->d_zero, h->d_layers, h->L, geometry(h), h->d_status, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        release(h);
        return HISPARSE_ERR_CUDA;
    }
    *out = h;
    return HISPARSE_OK;
}

}  // namespace

extern "C" {

int hisparse_create(const hisparse_layout *layout, hisparse_t *out)
{
    return create_impl(layout, 0, out);
}

int hisparse_create_paged(const hisparse_layout *layout, int32_t host_block_tokens, hisparse_t *out)
{
    if (out) *out = nullptr;
    if (host_block_tokens < 1) return out ? HISPARSE_ERR_LAYOUT : HISPARSE_ERR_INVALID_ARG;
    return create_impl(layout, host_block_tokens, out);
}

int hisparse_host_reserve(hisparse_t h, int32_t n, const int32_t *requests,
                          const int64_t *num_tokens, void *stream)
{
    if (!h || !h->hb || n < 0 || (n > 0 && (!requests || !num_tokens)))
        return HISPARSE_ERR_INVALID_ARG;
    if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
    std::vector<int32_t> want(h->nblocks);
    for (int32_t i = 0; i < n; ++i) {
        const int32_t r = requests[i];
        if (r < 0 || r >= h->R || num_tokens[i] < 0 || num_tokens[i] > h->cap[r])
            return HISPARSE_ERR_INVALID_ARG;
        const int64_t nb = (num_tokens[i] + h->hb - 1) / h->hb;
        want[r] = (int32_t)std::max<int64_t>(want[r], nb);
    }
    int64_t need = 0;
    for (int32_t r = 0; r < h->R; ++r) need += want[r] - h->nblocks[r];
    if (need > h->free_blocks) return HISPARSE_ERR_CAPACITY;
    // [Arch] Ownership: logical host block allocation; the lowest free block
    // goes to each new table entry, in the order asked
    const std::vector<int32_t> before(h->nblocks);
    RunList runs;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t r = requests[i];
        const int64_t nb = (num_tokens[i] + h->hb - 1) / h->hb;
        while (h->nblocks[r] < nb) {
            const int32_t idx = tbl_row(h, r) + h->nblocks[r]++;
            h->tbl[idx] = take_lowest_free(h);
            runs.add(idx, h->tbl[idx]);
        }
    }
    note_launch_all(h, as_stream(stream));
    const cudaError_t e = runs.apply(h->d_tbl, as_stream(stream));
    if (e != cudaSuccess) {
        // the device table may lag the host copy: undo the host side
        for (int32_t r = 0; r < h->R; ++r)
            for (; h->nblocks[r] > before[r]; --h->nblocks[r]) {
                const int32_t idx = tbl_row(h, r) + h->nblocks[r] - 1;
                give_back(h, h->tbl[idx]);
                h->tbl[idx] = -1;
            }
    }
    return cuda_status(e);
}

int hisparse_host_release(hisparse_t h, int32_t n, const int32_t *requests, void *stream)
{
    if (!h || !h->hb || n < 0 || (n > 0 && !requests)) return HISPARSE_ERR_INVALID_ARG;
    if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (requests[i] < 0 || requests[i] >= h->R) return HISPARSE_ERR_INVALID_ARG;
    RunList runs;
    std::vector<std::pair<int32_t, std::vector<int32_t>>> freed;   // to undo a failed launch
    for (int32_t i = 0; i < n; ++i) {
        const int32_t r = requests[i];
        if (h->nblocks[r] == 0) continue;
        const int32_t row = tbl_row(h, r);
        freed.emplace_back(r, std::vector<int32_t>(&h->tbl[row], &h->tbl[row] + h->nblocks[r]));
        for (int32_t b = 0; b < h->nblocks[r]; ++b) {
            give_back(h, h->tbl[row + b]);
            h->tbl[row + b] = -1;
        }
        runs.clear_range(row, h->nblocks[r]);
        h->nblocks[r] = 0;
    }
    note_launch_all(h, as_stream(stream));
    const cudaError_t e = runs.apply(h->d_tbl, as_stream(stream));
    if (e != cudaSuccess) {
        for (auto &f : freed) {
            const int32_t row = tbl_row(h, f.first);
            for (size_t b = 0; b < f.second.size(); ++b) {
                retake(h, f.second[b]);
                h->tbl[row + b] = f.second[b];
            }
            h->nblocks[f.first] = (int32_t)f.second.size();
        }
    }
    return cuda_status(e);
}

int hisparse_host_block_table(hisparse_t h, int32_t request, int32_t *ids, int32_t max_ids,
                              int32_t *count)
{
    if (!h || !h->hb || !count || max_ids < 0 || (max_ids > 0 && !ids)) return HISPARSE_ERR_INVALID_ARG;
    if (request < 0 || request >= h->R) return HISPARSE_ERR_INVALID_ARG;
    *count = h->nblocks[request];
    const int32_t n = std::min(max_ids, h->nblocks[request]);
    if (n > 0) std::memcpy(ids, &h->tbl[tbl_row(h, request)], sizeof(int32_t) * n);
    return HISPARSE_OK;
}

int hisparse_host_pool_info(hisparse_t h, int32_t *block_tokens, int32_t *pool_blocks,
                            int32_t *free_blocks)
{
    if (!h) return HISPARSE_ERR_INVALID_ARG;
    if (block_tokens) *block_tokens = h->hb;
    if (pool_blocks) *pool_blocks = h->pool_blocks;
    if (free_blocks) *free_blocks = h->free_blocks;
    return HISPARSE_OK;
}

int hisparse_host_block_rows(hisparse_t h, int32_t layer, int32_t block, void **host_ptr)
{
    if (!h || !h->hb || !host_ptr) return HISPARSE_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->L) return HISPARSE_ERR_LAYER;
    if (block < 0 || block >= h->pool_blocks) return HISPARSE_ERR_INVALID_ARG;
    *host_ptr = h->host_pool + ((int64_t)layer * h->pool_rows + (int64_t)block * h->hb) * h->B;
    return HISPARSE_OK;
}

int hisparse_destroy(hisparse_t h)
{
    release(h);
    return HISPARSE_OK;
}

int hisparse_host_rows(hisparse_t h, int32_t layer, int32_t request, void **host_ptr)
{
    if (!h || !host_ptr || h->hb) return HISPARSE_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->L) return HISPARSE_ERR_LAYER;
    if (request < 0 || request >= h->R) return HISPARSE_ERR_INVALID_ARG;
    *host_ptr = h->host_pool + ((int64_t)layer * h->total_cap + h->off[request]) * h->B;
    return HISPARSE_OK;
}

int hisparse_device_buffer(hisparse_t h, int32_t layer, void **dev_ptr)
{
    if (!h || !dev_ptr) return HISPARSE_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->L) return HISPARSE_ERR_LAYER;
    *dev_ptr = layer_store(h, layer).dev;
    return HISPARSE_OK;
}

int hisparse_prefill(hisparse_t h, const int32_t *seq_lens, void *stream)
{
    if (!h || !seq_lens) return HISPARSE_ERR_INVALID_ARG;
    if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
    note_launch_all(h, as_stream(stream));
    return cuda_status(hs::launch_prefill(seq_lens, h->d_layers, h->L, geometry(h), h->d_status,
                                          as_stream(stream)));
}

}  // extern "C"

namespace {

int swap_in_impl(hisparse_t h, int32_t layer, const int32_t *topk_idx, const int32_t *seq_lens,
                 const int32_t *resident_blocks, int32_t max_blocks, int32_t block_size,
                 int32_t *out_slot_ids, const hisparse_plan *out_plan, void *stream)
{
    if (!h || !topk_idx || !seq_lens || !out_slot_ids) return HISPARSE_ERR_INVALID_ARG;
    if (out_plan && (!out_plan->rows || !out_plan->counts)) return HISPARSE_ERR_INVALID_ARG;
    if (resident_blocks && (max_blocks < 1 || block_size < 1)) return HISPARSE_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->L || h->anchor[layer] >= 0) return HISPARSE_ERR_LAYER;
    if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
    hs::ResolveLaunch a;
    a.topk = topk_idx;
    a.seq_lens = seq_lens;
    a.out = out_slot_ids;
    a.status = h->d_status;
    a.st = h->state[layer];
    a.store = layer_store(h, layer);
    a.g = geometry(h);
    a.max_cap = (int32_t)h->max_cap;
    const bool split = h->copy_mode == HISPARSE_COPY_SPLIT;
    const bool autom = h->copy_mode == HISPARSE_COPY_AUTO && h->R < kAutoDeferBelowRequests;
    a.fused_copy = !split;
    a.stage_s2t = h->stage_s2t;
    a.lookup = h->lookup;
    a.resident = resident_blocks;
    a.res_max_blocks = resident_blocks ? max_blocks : 0;
    a.res_block_size = resident_blocks ? block_size : 0;
    a.deferred = autom ? h->d_deferred : nullptr;
    a.defer_bytes = kAutoDeferBytes;
    a.protect_calls = (uint32_t)h->protect_calls;
    // rows go through shared memory only when this CTA copies them for sure
    a.stage_rows = (!split && !autom) ? h->stage_rows : 0;
    a.programmatic = h->programmatic;
    a.wait_late = h->programmatic && left_layer_alone(h, as_stream(stream), layer);
    a.aligned_rows = h->B < hs::kAlignedRowsBelow;
    // copier CTAs only where the resolving CTA would copy every row itself
    a.ncopy = (!split && !autom && a.stage_rows == 0) ? h->copy_ctas - 1 : 0;
    const bool wide_copy = split || autom;
    a.plan_rows = out_plan ? out_plan->rows : (wide_copy ? h->d_plan_rows : nullptr);
    a.plan_counts = out_plan ? out_plan->counts : (wide_copy ? h->d_plan_counts : nullptr);
    cudaError_t e = hs::launch_resolve(a, as_stream(stream));
    note_launch_layers(h, as_stream(stream), &layer, 1);
    if (e != cudaSuccess || !wide_copy) return cuda_status(e);
    hs::ReplayLaunch c;
    c.plan_rows = a.plan_rows;
    c.plan_counts = a.plan_counts;
    c.store[0] = a.store;
    c.num_layers = 1;
    c.g = a.g;
    c.num_ctas = h->num_sms;
    c.programmatic = true;
    c.only_if = autom ? h->d_deferred : nullptr;
    return cuda_status(hs::launch_replay(c, as_stream(stream)));
}

}  // namespace

extern "C" {

int hisparse_swap_in(hisparse_t h, int32_t layer, const int32_t *topk_idx, const int32_t *seq_lens,
                     int32_t *out_slot_ids, const hisparse_plan *out_plan, void *stream)
{
    return swap_in_impl(h, layer, topk_idx, seq_lens, nullptr, 0, 0, out_slot_ids, out_plan, stream);
}

int hisparse_swap_in_resident(hisparse_t h, int32_t layer, const int32_t *topk_idx,
                              const int32_t *seq_lens, const int32_t *resident_blocks,
                              int32_t max_blocks, int32_t block_size, int32_t *out_slot_ids,
                              const hisparse_plan *out_plan, void *stream)
{
    if (!resident_blocks) return HISPARSE_ERR_INVALID_ARG;
    return swap_in_impl(h, layer, topk_idx, seq_lens, resident_blocks, max_blocks, block_size,
                        out_slot_ids, out_plan, stream);
}

int hisparse_replay_plan_layers(hisparse_t h, const hisparse_plan *plan, const int32_t *layers,
                                int32_t num_layers, int32_t num_ctas, void *stream)
{
    if (!h || !plan || !plan->rows || !plan->counts || !layers || num_ctas < 0)
        return HISPARSE_ERR_INVALID_ARG;
    if (num_layers < 1 || num_layers > hs::kMaxReplayLayers) return HISPARSE_ERR_INVALID_ARG;
    if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
    hs::ReplayLaunch c;
    for (int i = 0; i < num_layers; ++i) {
        if (layers[i] < 0 || layers[i] >= h->L) return HISPARSE_ERR_LAYER;
        c.store[i] = layer_store(h, layers[i]);
    }
    c.num_layers = num_layers;
    c.plan_rows = plan->rows;
    c.plan_counts = plan->counts;
    c.g = geometry(h);
    c.num_ctas = num_ctas ? num_ctas : 16;
    c.programmatic = false;
    c.only_if = nullptr;
    note_launch_layers(h, as_stream(stream), layers, num_layers);
    return cuda_status(hs::launch_replay(c, as_stream(stream)));
}

int hisparse_replay_plan(hisparse_t h, const hisparse_plan *plan, int32_t layer, int32_t num_ctas,
                         void *stream)
{
    return hisparse_replay_plan_layers(h, plan, &layer, 1, num_ctas, stream);
}

int hisparse_backup_layers(hisparse_t h, const int32_t *layers, int32_t num_layers,
                           const void *rows, const int32_t *positions, void *stream)
{
    if (!h || !layers || !rows || !positions) return HISPARSE_ERR_INVALID_ARG;
    if (num_layers < 1 || num_layers > hs::kMaxBackupLayers) return HISPARSE_ERR_INVALID_ARG;
    if (!aligned16(rows)) return HISPARSE_ERR_ALIGNMENT;
    for (int32_t i = 0; i < num_layers; ++i) {
        if (layers[i] < 0 || layers[i] >= h->L) return HISPARSE_ERR_LAYER;
        for (int32_t j = 0; j < i; ++j)
            if (layers[j] == layers[i]) return HISPARSE_ERR_INVALID_ARG;
    }
    if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
    hs::BackupLaunch b;
    const int64_t layer_bytes = (int64_t)h->R * h->B;
    for (int32_t i = 0; i < num_layers; ++i) {
        const hs::LayerStore s = layer_store(h, layers[i]);
        b.layer[i].rows = static_cast<const uint8_t *>(rows) + i * layer_bytes;
        b.layer[i].host = const_cast<uint8_t *>(s.host);
        b.layer[i].dev = s.dev;
        b.layer[i].st = h->state[layers[i]];
    }
    b.num_layers = num_layers;
    b.positions = positions;
    b.g = geometry(h);
    b.status = h->d_status;
    b.programmatic = h->programmatic;
    note_launch_layers(h, as_stream(stream), layers, num_layers);
    return cuda_status(hs::launch_backup(b, as_stream(stream)));
}

int hisparse_backup(hisparse_t h, int32_t layer, const void *rows, const int32_t *positions,
                    void *stream)
{
    return hisparse_backup_layers(h, &layer, 1, rows, positions, stream);
}

int hisparse_status(hisparse_t h, int32_t **dev_status)
{
    if (!h || !dev_status) return HISPARSE_ERR_INVALID_ARG;
    *dev_status = h->d_status;
    return HISPARSE_OK;
}

int hisparse_status_clear(hisparse_t h, void *stream)
{
    if (!h) return HISPARSE_ERR_INVALID_ARG;
    if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(h->d_status, 0, sizeof(int32_t) * h->R, as_stream(stream)));
}

int hisparse_read_state(hisparse_t h, int32_t layer, int32_t *slot2tok, uint32_t *last_used,
                        int32_t *tok2slot, int32_t *lru_order, uint32_t *ticks, void *stream)
{
    if (!h) return HISPARSE_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->L || h->anchor[layer] >= 0) return HISPARSE_ERR_LAYER;
    const hs::HotState &st = h->state[layer];
    const size_t RD = (size_t)h->R * h->D;
    cudaError_t e = cudaStreamSynchronize(as_stream(stream));
    if (e == cudaSuccess && slot2tok) e = cudaMemcpy(slot2tok, st.slot2tok, RD * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && last_used) e = cudaMemcpy(last_used, st.last_used, RD * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && tok2slot)
        e = cudaMemcpy(tok2slot, st.tok2slot, (size_t)h->total_cap * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && lru_order) {
        std::vector<uint16_t> tmp(RD);
        e = cudaMemcpy(tmp.data(), st.lru, RD * 2, cudaMemcpyDeviceToHost);
        for (size_t i = 0; e == cudaSuccess && i < RD; ++i) lru_order[i] = tmp[i];
    }
    if (e == cudaSuccess && ticks) e = cudaMemcpy(ticks, st.tick, (size_t)h->R * 4, cudaMemcpyDeviceToHost);
    return cuda_status(e);
}

int hisparse_write_state(hisparse_t h, int32_t layer, const int32_t *slot2tok,
                         const uint32_t *last_used, const uint32_t *ticks, int32_t rebuild_rows,
                         void *stream)
{
    if (!h || !slot2tok || !last_used || !ticks) return HISPARSE_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->L || h->anchor[layer] >= 0) return HISPARSE_ERR_LAYER;
    if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
    const int R = h->R, D = h->D;
    const size_t RD = (size_t)R * D;
    // the token->slot map and the LRU order follow from slot->token and
    // the stamps; a token may sit in one slot only, and (paged pool, when
    // rows are rebuilt) must have a host row
    std::vector<int32_t> t2s((size_t)h->total_cap, -1);
    std::vector<uint16_t> lru(RD);
    std::vector<int32_t> plan;       // (host slot, slot) pairs for the rebuild, [R][D][2]
    std::vector<int32_t> counts(R, 0);
    if (rebuild_rows) plan.assign(RD * 2, -1);
    std::vector<int> order(D);
    for (int r = 0; r < R; ++r) {
        const int32_t *s2t = slot2tok + (size_t)r * D;
        const uint32_t *lu = last_used + (size_t)r * D;
        for (int sl = 0; sl < D; ++sl) {
            if (lu[sl] > ticks[r]) return HISPARSE_ERR_INVALID_ARG;   // a stamp from a later call
            const int32_t t = s2t[sl];
            if (t == -1) continue;
            if (t < 0 || t >= h->cap[r]) return HISPARSE_ERR_INVALID_ARG;
            int32_t &m = t2s[(size_t)h->off[r] + t];
            if (m != -1) return HISPARSE_ERR_INVALID_ARG;
            m = sl;
            if (rebuild_rows) {
                int64_t row = t;
                if (h->hb) {
                    const int32_t id = h->tbl[(size_t)tbl_row(h, r) + t / h->hb];
                    if (id < 0 || t / h->hb >= h->nblocks[r]) return HISPARSE_ERR_INVALID_ARG;
                    row = (int64_t)id * h->hb + t % h->hb;
                }
                int32_t *pr = &plan[((size_t)r * D + counts[r]++) * 2];
                pr[0] = (int32_t)row;
                pr[1] = sl;
            }
        }
        for (int i = 0; i < D; ++i) order[i] = i;
        std::sort(order.begin(), order.end(), [&](int a, int b) {
            return lu[a] != lu[b] ? lu[a] < lu[b] : a < b;
        });
        for (int i = 0; i < D; ++i) lru[(size_t)r * D + i] = (uint16_t)order[i];
    }
    const hs::HotState &st = h->state[layer];
    cudaError_t e = cudaStreamSynchronize(as_stream(stream));
    note_launch_all(h, as_stream(stream));
    if (e == cudaSuccess) e = cudaMemcpy(st.slot2tok, slot2tok, RD * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(st.last_used, last_used, RD * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(st.tok2slot, t2s.data(), t2s.size() * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && st.resbits) {
        std::vector<uint32_t> bits((size_t)R * st.res_words, 0u);
        for (int r = 0; r < R; ++r)
            for (int64_t t = 0; t < h->cap[r]; ++t)
                if (t2s[(size_t)h->off[r] + t] >= 0)
                    bits[(size_t)r * st.res_words + t / 32] |= 1u << (t % 32);
        e = cudaMemcpy(st.resbits, bits.data(), bits.size() * 4, cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaMemcpy(st.lru, lru.data(), RD * 2, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(st.tick, ticks, (size_t)R * 4, cudaMemcpyHostToDevice);
    if (e != cudaSuccess || !rebuild_rows) return cuda_status(e);
    // Rebuild the hot rows of this layer and of the layers that share its
    // slots: the replay kernel over a plan of every filled slot (k = D).
    int32_t *d_plan = nullptr, *d_counts = nullptr;
    e = cudaMalloc(reinterpret_cast<void **>(&d_plan), plan.size() * 4);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&d_counts), (size_t)R * 4);
    if (e == cudaErrorMemoryAllocation) {
        cudaGetLastError();
        cudaFree(d_plan);
        return HISPARSE_ERR_NO_MEMORY;
    }
    if (e == cudaSuccess) e = cudaMemcpy(d_plan, plan.data(), plan.size() * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(d_counts, counts.data(), (size_t)R * 4, cudaMemcpyHostToDevice);
    std::vector<int32_t> layers{layer};
    for (int l = 0; l < h->L; ++l)
        if (h->anchor[l] == layer) layers.push_back(l);
    for (size_t i0 = 0; e == cudaSuccess && i0 < layers.size(); i0 += hs::kMaxReplayLayers) {
        hs::ReplayLaunch c;
        c.num_layers = (int)std::min(layers.size() - i0, (size_t)hs::kMaxReplayLayers);
        for (int i = 0; i < c.num_layers; ++i) c.store[i] = layer_store(h, layers[i0 + i]);
        c.plan_rows = d_plan;
        c.plan_counts = d_counts;
        c.g = geometry(h);
        c.g.k = D;                     // plan rows of D pairs per request
        c.num_ctas = h->num_sms;
        c.programmatic = false;
        c.only_if = nullptr;
        note_launch_all(h, nullptr);
        e = hs::launch_replay(c, nullptr);
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    cudaFree(d_plan);
    cudaFree(d_counts);
    return cuda_status(e);
}

int hisparse_check_guards(hisparse_t h, int32_t *overwritten)
{
    if (!h || !overwritten) return HISPARSE_ERR_INVALID_ARG;
    if (!h->guards) return HISPARSE_ERR_UNSUPPORTED;
    if (cudaDeviceSynchronize() != cudaSuccess) return HISPARSE_ERR_CUDA;
    std::vector<unsigned char> band(kGuardBytes);
    int32_t bad = 0;
    // the pinned pool's bands, read on the host
    const size_t pool_bytes = (size_t)h->L * h->layer_rows() * h->B;
    for (const uint8_t *q : {h->host_pool - kGuardBytes, h->host_pool + pool_bytes})
        for (size_t i = 0; i < kGuardBytes; ++i)
            if (q[i] != kGuardByte) { ++bad; break; }
    for (const auto &g : h->guarded) {
        for (int side = 0; side < 2; ++side) {
            const uint8_t *src = side ? g.first + g.second : g.first - kGuardBytes;
            if (cudaMemcpy(band.data(), src, kGuardBytes, cudaMemcpyDeviceToHost) != cudaSuccess)
                return HISPARSE_ERR_CUDA;
            for (unsigned char b : band)
                if (b != kGuardByte) { ++bad; break; }
        }
    }
    *overwritten = bad;
    return HISPARSE_OK;
}

int hisparse_set_protected_calls(hisparse_t h, int32_t calls)
{
    if (!h || calls < 0) return HISPARSE_ERR_INVALID_ARG;
    h->protect_calls = calls;
    return HISPARSE_OK;
}

int hisparse_set_copy_ctas(hisparse_t h, int32_t ctas)
{
    if (!h || ctas < 1 || ctas > hs::kMaxCopyCtas) return HISPARSE_ERR_INVALID_ARG;
    if (ctas > 1) {
        // every cluster's CTAs must fit on the SMs of one GPC at once
        if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
        int n = 0;
        if (hs::resolve_max_clusters(h->k, ctas, resolve_smem(h), &n) != cudaSuccess) {
            cudaGetLastError();
            return HISPARSE_ERR_CUDA;
        }
        if (n < 1) return HISPARSE_ERR_UNSUPPORTED;
    }
    h->copy_ctas = ctas;
    return HISPARSE_OK;
}

int hisparse_get_copy_ctas(hisparse_t h, int32_t *ctas)
{
    if (!h || !ctas) return HISPARSE_ERR_INVALID_ARG;
    *ctas = h->copy_ctas;
    return HISPARSE_OK;
}

int hisparse_set_programmatic_launch(hisparse_t h, int32_t on)
{
    if (!h || (on != 0 && on != 1)) return HISPARSE_ERR_INVALID_ARG;
    h->programmatic = on == 1;
    return HISPARSE_OK;
}

int hisparse_set_stage_rows(hisparse_t h, int32_t rows)
{
    if (!h || rows < -1) return HISPARSE_ERR_INVALID_ARG;
    h->stage_rows = rows == -1 ? h->max_stage_rows : std::min(rows, h->max_stage_rows);
    return HISPARSE_OK;
}

int hisparse_set_copy_mode(hisparse_t h, int32_t mode)
{
    if (!h || (mode != HISPARSE_COPY_FUSED && mode != HISPARSE_COPY_SPLIT && mode != HISPARSE_COPY_AUTO))
        return HISPARSE_ERR_INVALID_ARG;
    h->copy_mode = mode;
    return HISPARSE_OK;
}

}  // extern "C"

extern "C" {

int hisparse_swap_in_noalloc(hisparse_t h, int32_t layer, const int32_t *topk_idx,
                             const int32_t *seq_lens, int32_t *out_slot_ids, void *stream)
{
    if (!h || !topk_idx || !seq_lens || !out_slot_ids) return HISPARSE_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->L || h->anchor[layer] >= 0) return HISPARSE_ERR_LAYER;
    if (!on_own_device(h)) return HISPARSE_ERR_INVALID_ARG;
    // the pairs of all requests plus one count per request must fit the array
    const int64_t need = ((int64_t)h->R * h->k * 2 + h->R) * 4;
    if (need > HISPARSE_NOALLOC_SCRATCH_BYTES) return HISPARSE_ERR_UNSUPPORTED;
    int32_t *scratch = h->noalloc_scratch;   // looked up by hisparse_create
    // Nothing needs clearing between calls: the resolve grid writes every
    // request's count, and the copy grid reads only the pairs those counts
    // cover.
    hs::ResolveLaunch a;
    a.topk = topk_idx;
    a.seq_lens = seq_lens;
    a.out = out_slot_ids;
    a.status = h->d_status;
    a.st = h->state[layer];
    a.store = layer_store(h, layer);
    a.g = geometry(h);
    a.max_cap = (int32_t)h->max_cap;
    a.fused_copy = false;
    a.stage_s2t = h->stage_s2t;
    a.lookup = h->lookup;
    a.resident = nullptr;
    a.res_max_blocks = 0;
    a.res_block_size = 0;
    a.deferred = nullptr;
    a.defer_bytes = 0;
    a.protect_calls = (uint32_t)h->protect_calls;
    a.stage_rows = 0;
    a.programmatic = h->programmatic;
    a.ncopy = 0;
    a.wait_late = false;
    a.aligned_rows = h->B < hs::kAlignedRowsBelow;
    a.plan_rows = scratch;
    a.plan_counts = scratch + (int64_t)h->R * h->k * 2;
    cudaError_t e = hs::launch_resolve(a, as_stream(stream));
    note_launch_layers(h, as_stream(stream), &layer, 1);
    if (e != cudaSuccess) return HISPARSE_ERR_CUDA;
    hs::ReplayLaunch c;
    c.plan_rows = a.plan_rows;
    c.plan_counts = a.plan_counts;
    c.store[0] = a.store;
    c.num_layers = 1;
    c.g = a.g;
    c.num_ctas = h->num_sms;
    c.programmatic = true;
    c.only_if = nullptr;
    return cuda_status(hs::launch_replay(c, as_stream(stream)));
}

// ---- measurement kernels ---------------------------------------------------

int hisparse_synthetic_compute(void *buf, int64_t bytes, int32_t passes, int32_t ctas_per_sm,
                               void *stream)
{
    if (!buf || bytes <= 0 || bytes % 16 != 0 || passes < 0 || ctas_per_sm < 1)
        return HISPARSE_ERR_INVALID_ARG;
    if (!aligned16(buf)) return HISPARSE_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return HISPARSE_ERR_CUDA;
    return cuda_status(hs::launch_synthetic_compute(buf, bytes, passes, sms * ctas_per_sm,
                                                    as_stream(stream)));
}

int hisparse_link_probe(const void *src, void *dst, int64_t bytes, int32_t num_ctas, void *stream)
{
    if (!src || !dst || bytes < 0 || bytes % 16 != 0 || num_ctas < 0) return HISPARSE_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return HISPARSE_ERR_ALIGNMENT;
    if (bytes == 0) return HISPARSE_OK;
    int ctas = num_ctas;
    if (ctas == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&ctas, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return HISPARSE_ERR_CUDA;
    }
    return cuda_status(hs::launch_link_probe(src, dst, bytes, ctas, as_stream(stream)));
}

int hisparse_link_gather(const void *src, int64_t row_bytes, const int64_t *rows, int64_t n,
                         void *dst, int32_t num_ctas, void *stream)
{
    if (!src || !dst || !rows || n < 0 || row_bytes <= 0 || row_bytes % 16 != 0 ||
        row_bytes / 16 > INT32_MAX || num_ctas < 0)
        return HISPARSE_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return HISPARSE_ERR_ALIGNMENT;
    if (n == 0) return HISPARSE_OK;
    int ctas = num_ctas;
    if (ctas == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&ctas, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return HISPARSE_ERR_CUDA;
    }
    return cuda_status(hs::launch_link_gather(src, row_bytes, rows, n, dst, ctas, as_stream(stream)));
}

}  // extern "C"
