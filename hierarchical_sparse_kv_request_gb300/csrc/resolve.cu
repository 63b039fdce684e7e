// resolve.cu -- the swap-in resolver kernel.
//
// One CTA of 1024 threads resolves one request's top-k for one call
// ([Guide] "HiSparse: Hierarchical Sparse Attention", Decode Workflow: fast
// path for short sequences; otherwise hit detection -> LRU reorder -> miss
// handling with a host-to-device copy; [Arch] "HiSparse local KV offload
// architecture", Hot lookup and LRU: a hot row is used in place and
// refreshes the GPU LRU, a miss takes the LRU victim and copies the pinned
// host row into it).  With copier CTAs the launch is a thread-block cluster
// per request: rank 0 resolves, the other ranks only copy.
//
// The miss copies cross the host link and dominate the call, so everything
// else is arranged around starting them as early as possible and keeping
// them going:
//   1. the slot->token row and the LRU list (and, where kept, the
//      request's resident-token bitmap row) are staged into shared memory
//      with asynchronous copies issued at kernel start, under the first
//      global round trip; when it fits, the staged row also yields an inverse
//      token->slot table in shared memory, so the hit lookup needs no gather
//      of the token->slot map after the top-k row arrives;
//   2. a miss is known as soon as its lookup returns (with the bitmap, as
//      soon as its bit is read), long before its victim slot is: at
//      classification every miss takes an arrival index (warp ballots and
//      one barrier) and its host row goes on a list.  Right after
//      classification the first chunks of that list are loaded into
//      registers (or, optionally, the first `stage_rows` rows are fetched
//      into shared memory by the bulk-copy engine).  With copier CTAs the
//      copiers load the list instead: with the bitmap they stage the same
//      rows and classify for themselves, in the same arrival order;
//      otherwise the list goes to them (distributed shared memory, released
//      by a cluster barrier) and they load it at once;
//   3. then the block scans give each miss its rank in token order and its
//      victim, and each victim is filed under its miss's arrival index (in
//      the copiers' shared memory, released by a cluster barrier; copiers
//      that classify for themselves get their victims before the resolver
//      writes the hot state); all state writes are plain stores (the
//      slot->token row is staged, so no write waits on a load of its own);
//   4. finally the rows are stored to their victims while a rolling window
//      of 8 loads per thread keeps the link busy to the end.  Rows under
//      1 KB are copied in 64-byte-aligned spans of one row per warp load.
//      Each thread walks its items with cursors (no division per item): all
//      warps issue their first loads at once, so the issue slots spent
//      before them are on the critical path, and for the same reason the
//      host lays out the shared memory once per launch.
// Only the bytes' route differs from a copy in rank order; where each row
// lands is fixed by its rank, so the results are the same.
//
// With a paged host pool ([Arch] Ownership: tokens map to logical host
// blocks), the request's host block table row is staged as well, under the
// token->slot round trip; a miss whose block is not reserved stops the call
// for that request (status NO_HOST_ROW, and nothing is fetched for it), and
// miss rows are addressed, and recorded in the plan, by their row in the
// layer's pool.
//
// Exact LRU without sorting.  The request's slots are kept in a list `lru`
// ordered by (last_used, slot).  One call stamps every selected slot (hits and
// refilled victims) with a new, larger tick, so afterwards the list is
//     [unselected slots, in their old order] ++ [selected slots, by slot].
// The victims are the first m non-hit entries of the old list, in list order,
// which is exactly ascending (last_used, slot) among non-hit slots.  Both the
// victim ranks and the rewritten list come from one block prefix sum over the
// non-hit flags of the list, plus a popcount prefix over the selected-slot
// bitmap.  Misses are ranked by token with a bitmap over [0, seq_len) and a
// popcount prefix, which yields ascending token order without a sort.
#include "hs_common.cuh"

namespace hs {
namespace {

constexpr int NT = 1024;       // threads per CTA
// Host chunks in flight per thread.  The copy keeps a window of COPY_WINDOW
// loads per thread: storing a chunk frees its register for the load of the
// chunk COPY_WINDOW steps ahead, so the link's queue never drains between
// batches.  The first EARLY_LOADS<KT> chunks of the window are loaded right
// after classification, before the victims are known (KT: top-k entries per
// thread; these registers stay live through the block scans).
constexpr int COPY_WINDOW = 8;
template <int KT> __host__ __device__ constexpr int early_loads() { return KT == 8 ? 2 : 4; }
// How long a CTA waits for its staged rows before it gives up on them (2 s
// of the GPU's global timer): far beyond any copy that completes (a call
// moves at most a few MB per CTA), so reaching it means a fault of the copy,
// which is recorded (status COPY_TIMEOUT) instead of waited for forever.
constexpr uint64_t kWaitNs = 2000000000ull;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct SmemPlan {
    size_t hit, sel, miss, lru, s2t, inv, res, dup, tbl, chunk, vict, lrow, avict, bar, cnt, stage,
        total;
};

// Shared memory of the CTA: bitmaps over slots and tokens, the staged LRU
// list, optionally the staged slot->token row (and, with it, an inverse
// token->slot table over [0, max_cap)) and host block table row, victims by
// miss rank and by arrival index, the leftover host rows, the staging
// mbarrier and arrival counter, and `stage_rows` rows of B bytes staged by
// the bulk-copy engine.
inline SmemPlan plan_smem(int k, int D, int max_cap, bool stage_s2t, int lookup,
                                              int tbl_stride, int stage_rows, int64_t B)
{
    SmemPlan p;
    const size_t DW = (size_t)(D + 31) / 32, MW = (size_t)(max_cap + 31) / 32;
    size_t o = 32 * 4;             // warp totals
    p.hit = o;   o += DW * 4;
    p.sel = o;   o += DW * 4;
    p.miss = o;  o += MW * 4;
    p.lru = align_up(o, 16); o = p.lru + align_up((size_t)D * 2, 16);
    p.s2t = o;   o += stage_s2t ? align_up((size_t)D * 4, 16) : 0;
    p.inv = o;   o += (stage_s2t && lookup >= kLookupInverse) ? align_up((size_t)max_cap * 2, 16) : 0;
    // with the inverse table: the staged resident-token bitmap row (16-byte
    // rows) and a token bitmap that catches duplicates
    const bool res = stage_s2t && lookup >= kLookupResident;
    p.res = o;   o += res ? align_up((size_t)MW * 4, 16) : 0;
    p.dup = o;   o += res ? align_up(MW * 4, 16) : 0;   // the block table row
                                                                      // after it is staged in
                                                                      // 16-byte copies
    p.tbl = o;   o += (size_t)tbl_stride * 4;   // a multiple of 16
    p.chunk = o; o = align_up(o + (size_t)NT * 2, 4);
    p.vict = o;  o = align_up(o + (size_t)k * 2, 16);
    p.lrow = o;  o += align_up((size_t)k * 4, 16);   // 16-byte rows: copied to copiers
    p.avict = o; o += align_up((size_t)k * 2, 16);
    p.bar = o;   o += 8;
    p.cnt = o;   o += 16;
    p.stage = align_up(o, 128);
    o = p.stage + (size_t)stage_rows * (size_t)B;
    p.total = align_up(o, 16);
    return p;
}

struct Smem {
    uint32_t *warp_tot;  // [32]
    uint32_t *hitbits;   // [DW]  slots hit by this call
    uint32_t *selbits;   // [DW]  slots chosen as victims
    uint32_t *missbits;  // [MW]  miss tokens (and, on the fast path, all tokens)
    uint16_t *lru_s;     // [D]   staged LRU list
    int32_t *s2t_s;      // [D]   staged slot->token row (null when not staged)
    uint16_t *inv;       // [max_cap] slot of each token, built from s2t_s (null: the
                         //       token->slot map in global memory is gathered instead)
    uint32_t *res_s;     // [MW]  staged resident-token bitmap row (null: not kept)
    uint32_t *dupbits;   // [MW]  tokens of this call, to catch duplicates (with res_s)
    int32_t *tbl_s;      // [tbl_stride] staged host block table row (null: no paged pool)
    uint16_t *chunk_pre; // [NT]  misses before each thread's chunk of missbits
    uint16_t *victims;   // [k]   victim slot of miss rank i
    int32_t *left_row;   // [k]   host row of leftover q = arrival SR + q (token, or pool
                         //       row when paged)
    uint16_t *arr_vict;  // [k]   victim slot of the miss with arrival index j
    uint64_t *bar;       //       mbarrier of the staged rows
    uint32_t *arrived;   //       misses that took an arrival index
    uint32_t *flags;     //       error flags of the CTA's classification (kFlag*)
    uint32_t *pub;       // [2]   in a copier CTA: the misses to load (written by the
                         //       resolver before the first cluster barrier) and to
                         //       store (before the second)
    uint8_t *stage;      // [stage_rows][B] rows fetched by the bulk-copy engine
};

// KT small signed indices (each in [-1, 32767]) packed two to a register.
template <int KT>
struct PackedIdx {
    uint32_t w[(KT + 1) / 2];
    __device__ __forceinline__ int32_t get(int i) const
    {
        return (int32_t)(int16_t)(uint16_t)(w[i >> 1] >> ((i & 1) * 16));
    }
    __device__ __forceinline__ void set(int i, int32_t v)
    {
        const int sh = (i & 1) * 16;
        w[i >> 1] = (w[i >> 1] & ~(0xFFFFu << sh)) | ((uint32_t)(uint16_t)v << sh);
    }
};

// Classification outcomes, OR-ed over the CTA in one barrier.
constexpr uint32_t kFlagBad = 1, kFlagDup = 2, kFlagBadRes = 4, kFlagNoHost = 8;

// OR of `f` over the CTA: one warp reduction, one shared atomic per warp
// and one barrier.  *word must be 0 and published by an earlier barrier.
__device__ __forceinline__ uint32_t block_or(uint32_t f, uint32_t *word)
{
    f = __reduce_or_sync(0xffffffffu, f);
    if ((threadIdx.x & 31) == 0 && f) atomicOr(word, f);
    __syncthreads();
    return *word;
}

// The status a call's flags give (BAD_INDEX, then DUPLICATE, BAD_RESIDENT
// and NO_HOST_ROW), or OK.
__device__ __forceinline__ int status_of(uint32_t flags)
{
    return (flags & kFlagBad) ? kStatusBadIndex
           : (flags & kFlagDup) ? kStatusDuplicate
           : (flags & kFlagBadRes) ? kStatusBadResident
           : (flags & kFlagNoHost) ? kStatusNoHostRow : kStatusOk;
}

__device__ __forceinline__ bool test_bit(const uint32_t *bits, int i)
{
    return (bits[i >> 5] >> (i & 31)) & 1u;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// all but this thread's most recent group (two groups) of asynchronous copies
// have landed
__device__ __forceinline__ void cp_async_wait_but_last() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_but_last2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// ---- bulk-copy engine (TMA, non-tensor form) and its mbarrier --------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t arrivals)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(arrivals)
                 : "memory");
    // make the initialised barrier visible to the bulk-copy engine
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One arrival of this thread, announcing `bytes` more to be delivered.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait for phase 0 of the staging barrier; false after kWaitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar)
{
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, 0))
        if (global_ns() - t0 > kWaitNs) return false;
    return true;
}
// Wait for the staged rows of request r.  If they do not all land within
// the bound, record COPY_TIMEOUT and wait once more (bounded as well) so
// that no copy is still writing this CTA's shared memory when it exits.
__device__ __forceinline__ bool staged_rows_landed(uint64_t *bar, int32_t *status, int r)
{
    if (mbar_wait_bounded(bar)) return true;
    record_status(status, r, kStatusCopyTimeout);
    mbar_wait_bounded(bar);
    return false;
}
// gmem (here pinned host memory through its device address) -> smem, `bytes`
// a multiple of 16 from 16-byte aligned addresses; completes on `bar`.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// smem -> gmem; tracked in the issuing thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk stores have read their shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- thread-block clusters: one resolver CTA and its copier CTAs ----------
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of the cluster arrives once per phase, then waits for the
// phase; arrive releases this thread's earlier writes (shared memory of
// other CTAs included) and wait acquires everyone's.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// Store to the same shared-memory location in CTA `rank` of the cluster
// (every CTA of the launch has the same shared-memory layout).
__device__ __forceinline__ uint32_t remote_addr(const void *local, uint32_t rank)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    return a;
}
__device__ __forceinline__ void st_remote_u32(const uint32_t *local, uint32_t rank, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote_addr(local, rank)), "r"(v) : "memory");
}
__device__ __forceinline__ void st_remote_v4(const void *local, uint32_t rank, uint4 v)
{
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(remote_addr(local, rank)),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// Copy `bytes` (a multiple of 16; 16-byte aligned) of this CTA's shared
// memory to the same place in every copier CTA, one 16-byte store per thread
// and copier.
__device__ __forceinline__ void copy_to_copiers(const void *local, uint32_t bytes, int ncopy)
{
    const uint4 *src = reinterpret_cast<const uint4 *>(local);
    for (uint32_t v = threadIdx.x; v < bytes / 16; v += blockDim.x) {
        const uint4 x = src[v];
        for (int q = 1; q <= ncopy; ++q) st_remote_v4(src + v, (uint32_t)q, x);
    }
}

// Which 16-byte chunk of the leftover list a thread's n-th copy moves.
//  - flat: chunk e = first + n * stride of the list, chunk e % CH of
//    leftover e / CH (consecutive lanes take consecutive chunks);
//  - unit-aligned: a warp's n-th task is e = first + n * stride; task e is
//    the (e % H)-th 512 bytes of the 64-byte-aligned span around leftover
//    e / H's host row, one 16-byte piece per lane, and lanes whose piece lies
//    outside the row move nothing.  No 64-byte unit of host memory is then
//    split between two warp loads.  Measured on GB300 (gathers of random
//    pinned rows): 656-byte rows 1.7-4% faster this way, 1152-byte rows 1-3%
//    slower.
// A thread walks its items with cursors (leftover q, and x: the chunk, or
// the task within the row's span), stepping by the stride's quotient and
// remainder: the one division is at construction.  The walk is issue-bound
// where it matters (all warps of a CTA issue their first loads at once), and
// a division per item cost ~1.5 us there on decode-sized calls.
struct CopyCursor {
    int q, x;
};

struct CopyWalk {
    int rows, CH, X, dq, dx, lane;
    bool aligned;
    uint32_t base_lo;   // low bits of the host rows' base: alignment only
    uint32_t B;
    CopyCursor start;
    __device__ __forceinline__ CopyWalk(bool al, int rows_, int ch, int first, int stride,
                                        const uint8_t *hrow0, int64_t B_)
        : rows(rows_), CH(ch), X(al ? (ch + 3 + 31) / 32 : ch), lane((int)(threadIdx.x & 31)),
          aligned(al), base_lo((uint32_t)reinterpret_cast<uintptr_t>(hrow0)), B((uint32_t)B_)
    {
        dq = div_small(stride, X);
        dx = stride - dq * X;
        start.q = div_small(first, X);
        start.x = first - start.q * X;
    }
    // v / X for v >= 0; the spans of rows under 1 KB take X <= 3 tasks, those
    // of 480- to 976-byte rows 2 (a shift instead of a division sequence)
    static __device__ __forceinline__ int div_small(int v, int X)
    {
        return X == 1 ? v : X == 2 ? (v >> 1) : v / X;
    }
    __device__ __forceinline__ void next(CopyCursor &k) const
    {
        k.q += dq;
        k.x += dx;
        if (k.x >= X) {
            k.x -= X;
            ++k.q;
        }
    }
    // chunk c of leftover k.q (whose host row is *hr) for cursor k; false
    // if the item moves nothing
    __device__ __forceinline__ bool at(const CopyCursor &k, const int32_t *left_row, int32_t &hr,
                                       int &c) const
    {
        if (k.q >= rows) return false;
        hr = left_row[k.q];
        if (!aligned) {
            c = k.x;
            return true;
        }
        const int delta = (int)(((base_lo + (uint32_t)hr * B) >> 4) & 3u);
        c = k.x * 32 + lane - delta;
        return c >= 0 && c < CH;
    }
    __device__ __forceinline__ bool done(const CopyCursor &k) const { return k.q >= rows; }
};

// Resident row of position t from its block id `id` (-1: not resident), or
// -2 when the id is malformed (below -1, or rows reaching the flag bit).
__device__ __forceinline__ int32_t resident_row(int32_t id, int32_t t, int32_t bs)
{
    if (id == -1) return -1;
    if (id < -1 || (int64_t)id * bs + bs > kResidentFlag) return -2;
    return id * bs + t % bs;
}

// With a late wait (ResolveLaunch::wait_late) the grid reads its inputs and
// this layer's state before the previous kernel of the stream has completed,
// and waits for it (griddepcontrol.wait) only before its first write to
// global memory; only then may the next launch start early.
__device__ __forceinline__ void late_grid_wait(const ResolveLaunch &a)
{
    if (a.wait_late) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
}

// Final writes of a request whose call ends without touching its state; on
// success (the fast path) each position resolves to its resident row or to
// slot = position.
template <int KT>
__device__ __forceinline__ void finish_untouched(const ResolveLaunch &a, int r,
                                                 const int32_t (&t)[KT], const int32_t (&rid)[KT],
                                                 int status, uint32_t tick)
{
    const int k = a.g.k;
    cp_async_wait_all();  // staged rows may still be landing in shared memory
    late_grid_wait(a);
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int j = threadIdx.x + i * NT;
        if (j >= k) continue;
        int32_t v = -1;
        if (status == kStatusOk) {
            const int32_t row = t[i] >= 0 ? resident_row(rid[i], t[i], a.res_block_size) : -1;
            v = row >= 0 ? (kResidentFlag | row) : t[i];
        }
        a.out[(int64_t)r * k + j] = v;
    }
    if (threadIdx.x == 0) {
        if (status != kStatusOk) record_status(a.status, r, status);
        if (a.plan_counts) a.plan_counts[r] = 0;
        if (a.deferred) a.deferred[r] = 0;
        a.st.tick[r] = tick;
    }
}

// A copier's share of the leftover rows: the first COPY_WINDOW loads go out
// at once; once the cluster barrier has released the victims (filed under
// the leftovers' indices in arr_vict; *go == 0: nothing to store after all),
// each stored chunk's register takes the load COPY_WINDOW items ahead.
__device__ __forceinline__ void copier_rows(const CopyWalk &walk, const int32_t *lrow,
                                            const uint16_t *arr_vict, const uint8_t *hrow0,
                                            uint8_t *drow0, int64_t B, const uint32_t *go)
{
    uint4 pv[COPY_WINDOW];
    CopyCursor ld = walk.start, st = walk.start;
#pragma unroll
    for (int u = 0; u < COPY_WINDOW; ++u) {
        int32_t hr;
        int cc;
        if (walk.at(ld, lrow, hr, cc)) pv[u] = ld_host_v4(hrow0 + (int64_t)hr * B + cc * 16);
        walk.next(ld);
    }
    cluster_wait();                       // the victims are in (or no copy)
    if (*go == 0) return;
    while (!walk.done(st)) {
#pragma unroll
        for (int u = 0; u < COPY_WINDOW; ++u) {
            int32_t hr;
            int cc;
            if (walk.at(st, lrow, hr, cc)) st_v4(drow0 + (int64_t)arr_vict[st.q] * B + cc * 16, pv[u]);
            walk.next(st);
            if (walk.at(ld, lrow, hr, cc)) pv[u] = ld_host_v4(hrow0 + (int64_t)hr * B + cc * 16);
            walk.next(ld);
        }
    }
}

// A copier CTA (rank c >= 1 of request r's cluster of 1 + ncopy CTAs).  It
// resolves nothing and touches no hot state: it loads the miss rows the
// resolver (rank 0) lists in this CTA's shared memory at classification, and
// stores them into the victim slots the resolver files there once the block
// scans have chosen them.  Its SM issues host loads and nothing else, so
// they queue behind nothing, and the resolver's own stores to the hot state
// queue behind no host loads.  Copier c takes the rounds n of the list with
// n % ncopy == c - 1: rounds of NT chunks (flat mapping) or of 32 warp tasks
// (aligned spans).
__device__ __forceinline__ void copier_main(const ResolveLaunch &a, const Smem &sm, int r, int c,
                                            int ncopy)
{
    const int tid = threadIdx.x;
    const int D = a.g.D, CH = a.g.chunks;
    const int64_t B = a.g.B;
    const int32_t S = a.seq_lens[r];
    const int64_t cap = a.g.host_cap[r];
    // the resolver takes its paths without a copy (a malformed length, the
    // fast path) on the same test, and then never reaches a cluster barrier
    if (S < 0 || (int64_t)S > cap || S <= D) return;
    const uint8_t *hrow0 = a.store.host + (a.g.hb ? 0 : a.g.host_off[r]) * B;
    uint8_t *drow0 = a.store.dev + (int64_t)r * D * B;
    cluster_arrive();
    cluster_wait();                       // phase 1: the leftover list is in
    if (sm.pub[0] == 0) return;           // an error, or no miss: no phase 2
    // Arrive for phase 2 before loading: the phase then ends as soon as the
    // resolver has filed the victims, not when this CTA's last thread has
    // got its loads out (host loads in flight hold up the issue of more).
    cluster_arrive();
    const int rows = (int)sm.pub[0];
    const CopyWalk walk = a.aligned_rows
                              ? CopyWalk(true, rows, CH, (c - 1) * (NT / 32) + (tid >> 5), ncopy * (NT / 32), hrow0, B)
                              : CopyWalk(false, rows, CH, (c - 1) * NT + tid, ncopy * NT, hrow0, B);
    copier_rows(walk, sm.left_row, sm.arr_vict, hrow0, drow0, B, &sm.pub[1]);
}

// Misses and their arrival indices, from the staged resident-token bitmap
// row: entry i of this thread (top-k entry tid + i NT) is a miss when it is a
// valid position, not a resident page, its bit is clear and it has a host row.
// The indices run over [0, m) in (warp, entry, lane) order: warp ballots place
// each miss within its warp, one barrier publishes the warps' counts (and
// error flags) through warp_tot, and each warp scans them for its base.  A
// self-classifying copier numbers its misses in the same order from the same
// inputs (without the flags and packed indices), so both build the same list.
template <int KT>
__device__ __forceinline__ void number_misses(uint32_t miss, uint32_t f, uint32_t *warp_tot,
                                              PackedIdx<KT> &arr, uint32_t &flags, uint32_t &m_all)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t in_warp = 0;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const bool mine = (miss >> i) & 1u;
        const unsigned mask = __ballot_sync(0xffffffffu, mine);
        arr.set(i, mine ? (int32_t)(in_warp + __popc(mask & ((1u << lane) - 1u))) : -1);
        in_warp += (uint32_t)__popc(mask);
    }
    const uint32_t wf = __reduce_or_sync(0xffffffffu, f);
    if (lane == 0) warp_tot[warp] = (wf << 16) | in_warp;   // in_warp <= 32 KT
    __syncthreads();
    static_assert(NT == 32 * 32, "one count per lane");
    const uint32_t v = warp_tot[lane];
    flags = __reduce_or_sync(0xffffffffu, v >> 16);
    uint32_t incl = v & 0xFFFFu;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    m_all = __shfl_sync(0xffffffffu, incl, 31);
    const uint32_t before = __shfl_sync(0xffffffffu, incl, (warp + 31) & 31);
    const uint32_t base = warp ? before : 0u;
#pragma unroll
    for (int i = 0; i < KT; ++i)
        if (arr.get(i) >= 0) arr.set(i, (int32_t)base + arr.get(i));
}

// A self-classifying copier CTA (with the resident-token bitmap): it stages
// the request's bitmap row itself, classifies the top-k row as the resolver
// does and numbers the misses the same way, so it has the list of host rows
// without a message, and starts its loads as soon as its own classification
// is done.  One cluster barrier follows: the resolver arrives once it has
// filed the victims in this CTA's shared memory (or found that nothing is to
// be copied) and set sm.pub[1]; this CTA arrives at once and waits for it
// before it stores, and always before it leaves, since the resolver writes
// into its shared memory on every path.
template <int KT>
__device__ __forceinline__ void copier_self(const ResolveLaunch &a, const Smem &sm, int r, int c,
                                            int ncopy)
{
    const int tid = threadIdx.x;
    const int k = a.g.k, D = a.g.D, CH = a.g.chunks;
    const int64_t B = a.g.B;
    const int32_t hb = a.g.hb;
    const int32_t S = a.seq_lens[r];
    const int64_t off = a.g.host_off[r];
    const int64_t cap = a.g.host_cap[r];
    int32_t t[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int j = tid + i * NT;
        t[i] = j < k ? a.topk[(int64_t)r * k + j] : -1;
    }
    const uint32_t *rb = a.st.resbits + (int64_t)r * a.st.res_words;
    for (int i = tid; i < (a.st.res_words >> 2); i += NT) cp_async16(sm.res_s + i * 4, rb + i * 4);
    cp_async_commit();
    int32_t rid[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        rid[i] = -1;
        if (a.resident && t[i] >= 0 && t[i] < S && t[i] <= cap) {
            const int32_t b = t[i] / a.res_block_size;
            if (b < a.res_max_blocks) rid[i] = a.resident[(int64_t)r * a.res_max_blocks + b];
        }
    }
    // the resolver's paths without a copy (a malformed length, the fast
    // path), taken by it on the same test, reach no cluster barrier
    if (S < 0 || (int64_t)S > cap || S <= D) {
        cp_async_wait_all();
        return;
    }
    if (hb) {
        const int32_t *tbl = a.g.host_tbl + (int64_t)r * a.g.tbl_stride;
        const int nq = (int)(((int64_t)S + 4LL * hb - 1) / (4LL * hb));
        for (int i = tid; i < nq; i += NT) cp_async16(sm.tbl_s + i * 4, tbl + i * 4);
        cp_async_commit();
    }
    cluster_arrive();
    cp_async_wait_all();
    __syncthreads();
    uint32_t miss = 0;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int32_t x = t[i];
        if (x < 0 || x >= S) continue;
        const int32_t row = resident_row(rid[i], x, a.res_block_size);
        if (row != -1 || (sm.res_s[x >> 5] >> (x & 31)) & 1u) continue;
        if (hb && sm.tbl_s[x / hb] < 0) continue;
        miss |= 1u << i;
    }
    // The list in arrival order, numbered as number_misses numbers it (warp,
    // entry slot, lane), without its packed indices and error flags: the
    // copier files each miss's host row at once.
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t below = (1u << lane) - 1u;
    uint32_t wmask[KT];
    uint32_t in_warp = 0;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        wmask[i] = __ballot_sync(0xffffffffu, (miss >> i) & 1u);
        in_warp += (uint32_t)__popc(wmask[i]);
    }
    if (lane == 0) sm.warp_tot[warp] = in_warp;
    __syncthreads();
    uint32_t incl = sm.warp_tot[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    const uint32_t m_all = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t pos = __shfl_sync(0xffffffffu, incl, (warp + 31) & 31);
    if (warp == 0) pos = 0;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        if ((miss >> i) & 1u)
            sm.left_row[pos + __popc(wmask[i] & below)] = hb ? sm.tbl_s[t[i] / hb] * hb + t[i] % hb : t[i];
        pos += (uint32_t)__popc(wmask[i]);
    }
    __syncthreads();
    const uint8_t *hrow0 = a.store.host + (hb ? 0 : off) * B;
    uint8_t *drow0 = a.store.dev + (int64_t)r * D * B;
    const int rows = (int)m_all;
    const CopyWalk walk = a.aligned_rows
                              ? CopyWalk(true, rows, CH, (c - 1) * (NT / 32) + (tid >> 5), ncopy * (NT / 32), hrow0, B)
                              : CopyWalk(false, rows, CH, (c - 1) * NT + tid, ncopy * NT, hrow0, B);
    copier_rows(walk, sm.left_row, sm.arr_vict, hrow0, drow0, B, &sm.pub[1]);
}

template <int KT>
__global__ void __launch_bounds__(NT, 1) resolve_kernel(ResolveLaunch a)
{
    constexpr int EARLY = early_loads<KT>();
    static_assert(EARLY <= COPY_WINDOW, "the early loads are the first of the window");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // With copier CTAs (a cluster launch of 1 + ncopy CTAs per request) this
    // CTA resolves request r if it is rank 0 of its cluster, else copies.
    const int ncopy = a.ncopy;
    const int r = blockIdx.x / (ncopy + 1);
    const int tid = threadIdx.x;
    const int k = a.g.k, D = a.g.D;
    const int DW = (D + 31) >> 5;
    const int64_t B = a.g.B;
    const int CH = a.g.chunks;
    const int SR = a.stage_rows;   // rows the bulk-copy engine may stage (0: none)

    const int32_t hb = a.g.hb;
    const ResolveSmem &sp = a.smem;   // the layout of plan_smem, laid out by the host
    Smem sm;
    sm.warp_tot = reinterpret_cast<uint32_t *>(smem_raw);
    sm.hitbits = reinterpret_cast<uint32_t *>(smem_raw + sp.hit);
    sm.selbits = reinterpret_cast<uint32_t *>(smem_raw + sp.sel);
    sm.missbits = reinterpret_cast<uint32_t *>(smem_raw + sp.miss);
    sm.lru_s = reinterpret_cast<uint16_t *>(smem_raw + sp.lru);
    sm.s2t_s = a.stage_s2t ? reinterpret_cast<int32_t *>(smem_raw + sp.s2t) : nullptr;
    sm.inv = (a.stage_s2t && a.lookup >= kLookupInverse) ? reinterpret_cast<uint16_t *>(smem_raw + sp.inv)
                                                         : nullptr;
    const bool early_classify = sm.inv && a.lookup >= kLookupResident && a.st.resbits;
    sm.res_s = early_classify ? reinterpret_cast<uint32_t *>(smem_raw + sp.res) : nullptr;
    sm.dupbits = early_classify ? reinterpret_cast<uint32_t *>(smem_raw + sp.dup) : nullptr;
    sm.tbl_s = hb ? reinterpret_cast<int32_t *>(smem_raw + sp.tbl) : nullptr;
    sm.chunk_pre = reinterpret_cast<uint16_t *>(smem_raw + sp.chunk);
    sm.victims = reinterpret_cast<uint16_t *>(smem_raw + sp.vict);
    sm.left_row = reinterpret_cast<int32_t *>(smem_raw + sp.lrow);
    sm.arr_vict = reinterpret_cast<uint16_t *>(smem_raw + sp.avict);
    sm.bar = reinterpret_cast<uint64_t *>(smem_raw + sp.bar);
    sm.arrived = reinterpret_cast<uint32_t *>(smem_raw + sp.cnt);
    sm.flags = sm.arrived + 1;
    sm.pub = sm.arrived + 2;
    sm.stage = smem_raw + sp.stage;

    // Launched behind another kernel with a programmatic dependency, this
    // grid may start while that one still runs (its CTAs are placed and set
    // up under the other's tail).  Normally nothing from global memory is
    // read before the other grid has completed and its writes are visible
    // (without such a dependency the wait returns at once); only then may the
    // next launch start early, so a swap-in that follows never reads hot
    // state that an older call is still writing.  (A copy grid launched
    // behind this one still waits for this grid before reading the plan.)
    // With wait_late the host has checked that the previous launch wrote
    // nothing this call reads (see late_grid_wait).
    if (!a.wait_late) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (ncopy) {
        const int rank = (int)cluster_rank();
        if (rank != 0) {
            // A copier's reads (host rows) follow its resolver's list, and its
            // stores the resolver's wait (phase 2); it never holds up the next
            // launch, which its resolver's later signal gates.
            if (a.wait_late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            if (early_classify) copier_self<KT>(a, sm, r, rank, ncopy);
            else copier_main(a, sm, r, rank, ncopy);
            return;
        }
    }

    // ---- loads that do not depend on each other --------------------------
    const int32_t S = a.seq_lens[r];
    const int64_t off = a.g.host_off[r];
    const int64_t cap = a.g.host_cap[r];
    const uint32_t tick = a.st.tick[r] + 1u;
    int32_t t[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int j = tid + i * NT;
        t[i] = j < k ? a.topk[(int64_t)r * k + j] : -1;
    }
    // Stage the resident-token bitmap row (if kept), the slot->token row and
    // the LRU list with asynchronous copies (three groups); they land under
    // the round trips above.  (16-byte rows need D % 8 == 0.)
    const uint16_t *lru = a.st.lru + (int64_t)r * D;
    int32_t *slot2tok = a.st.slot2tok + (int64_t)r * D;
    const bool staged_async = (D & 7) == 0;
    if (sm.res_s) {   // the resident-token bitmap row first: classification needs it first
        const uint32_t *rb = a.st.resbits + (int64_t)r * a.st.res_words;
        for (int i = tid; i < (a.st.res_words >> 2); i += NT) cp_async16(sm.res_s + i * 4, rb + i * 4);
    }
    cp_async_commit();
    if (staged_async && sm.s2t_s)
        for (int i = tid; i < (D >> 2); i += NT) cp_async16(sm.s2t_s + i * 4, slot2tok + i * 4);
    cp_async_commit();
    if (staged_async)
        for (int i = tid; i < (D >> 3); i += NT) cp_async16(sm.lru_s + i * 8, lru + i * 8);
    cp_async_commit();
    // Resident pages first ([Arch] Resident device pages; Hot lookup and
    // LRU): gather the block id of every position's block (-1 when there is
    // no table or the block lies past its end).
    int32_t rid[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        rid[i] = -1;
        if (a.resident && t[i] >= 0 && t[i] < S && t[i] <= cap) {
            const int32_t b = t[i] / a.res_block_size;
            if (b < a.res_max_blocks) rid[i] = a.resident[(int64_t)r * a.res_max_blocks + b];
        }
    }

    if (S < 0 || (int64_t)S > cap) {  // uniform across the CTA
        finish_untouched<KT>(a, r, t, rid, kStatusBadSeqLen, tick);
        return;
    }

    // ---- fast path: every token is already at slot = token ---------------
    if (S <= D) {
        const int mw = (S + 31) >> 5;
        for (int w = tid; w < mw; w += NT) sm.missbits[w] = 0u;
        if (tid == 0) *sm.flags = 0u;
        __syncthreads();
        uint32_t f = 0;
#pragma unroll
        for (int i = 0; i < KT; ++i) {
            const int32_t x = t[i];
            if (x == -1) continue;
            if (x < 0 || x >= S) { f |= kFlagBad; continue; }
            if (resident_row(rid[i], x, a.res_block_size) == -2) f |= kFlagBadRes;
            const uint32_t bit = 1u << (x & 31);
            if (atomicOr(&sm.missbits[x >> 5], bit) & bit) f |= kFlagDup;
        }
        finish_untouched<KT>(a, r, t, rid, status_of(block_or(f, sm.flags)), tick);
        return;
    }

    // ---- slow path: hit detection ----------------------------------------
    if (hb) {
        // the host block ids of tokens [0, S): 16-byte rows of the table
        // (the stride is a multiple of 4 entries and covers the capacity)
        const int32_t *tbl = a.g.host_tbl + (int64_t)r * a.g.tbl_stride;
        const int nq = (int)(((int64_t)S + 4LL * hb - 1) / (4LL * hb));
        for (int i = tid; i < nq; i += NT) cp_async16(sm.tbl_s + i * 4, tbl + i * 4);
        cp_async_commit();
    }
    // host row of token x: its position in the request's region, or its row
    // in the layer's pool
    auto host_slot = [&](int32_t x) -> int32_t {
        return hb ? sm.tbl_s[x / hb] * hb + x % hb : x;
    };
    // Hit lookup: the slot of each top-k token, or -1.  Without the inverse
    // table, a gather of the token->slot map (a round trip to global memory
    // that starts only once the top-k row is in).
    int32_t *tok2slot = a.st.tok2slot + off;
    int32_t s[KT];
    if (!sm.inv) {
#pragma unroll
        for (int i = 0; i < KT; ++i) {
            s[i] = (t[i] >= 0 && t[i] < S) ? tok2slot[t[i]] : -1;
            if (s[i] >= D) s[i] = -1;  // never true for state this library wrote
        }
    }
    const int mw = (S + 31) >> 5;
    for (int w = tid; w < mw; w += NT) sm.missbits[w] = 0u;
    if (sm.dupbits)
        for (int w = tid; w < mw; w += NT) sm.dupbits[w] = 0u;
    for (int w = tid; w < DW; w += NT) { sm.hitbits[w] = 0u; sm.selbits[w] = 0u; }
    if (!staged_async) {
        for (int i = tid; i < D; i += NT) sm.lru_s[i] = lru[i];
        if (sm.s2t_s)
            for (int i = tid; i < D; i += NT) sm.s2t_s[i] = slot2tok[i];
    }
    if (tid == 0) {
        *sm.arrived = 0u;
        *sm.flags = 0u;
        if (SR) mbar_init(sm.bar, NT);   // every thread arrives once
    }
    if (sm.res_s) {
        // Misses first: the staged resident-token bitmap tells a miss from a
        // hit before any slot is known; the hits' slots come from the inverse
        // table once the miss list is out (below).
        if (hb) cp_async_wait_all();   // the block table row is needed too
        else cp_async_wait_but_last2();  // the slot->token row and LRU list may still land
        __syncthreads();
#pragma unroll
        for (int i = 0; i < KT; ++i) s[i] = -1;
    } else if (sm.inv) {
        // With the inverse table the lookup needs only the staged
        // slot->token row, whose copy was issued at the start: every slot
        // files itself under its token, and a token's entry counts only if
        // that slot still holds the token (so entries of tokens that no slot
        // holds, never written, are harmless: the maps are mutual inverses).
        if (hb) cp_async_wait_all();   // the block table row is needed too
        else cp_async_wait_but_last();  // the LRU list may still be landing
        __syncthreads();
        for (int sl = tid; sl < D; sl += NT) {
            const int32_t x = sm.s2t_s[sl];
            if (x >= 0 && x < a.max_cap) sm.inv[x] = (uint16_t)sl;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < KT; ++i) {
            s[i] = -1;
            if (t[i] >= 0 && t[i] < S) {
                const int v = sm.inv[t[i]];
                if (v < D && sm.s2t_s[v] == t[i]) s[i] = v;
            }
        }
    } else {
        cp_async_wait_all();
        __syncthreads();
    }

    // Classify.  A resident position is marked in the token bitmap only to
    // catch duplicates; its bit is cleared again before the misses are
    // ranked, and it never touches the hot state.  A miss with a host row is
    // also marked for the early fetch below.
    uint32_t f = 0;       // kFlag* of this thread's entries
    uint32_t miss = 0;    // bit i: entry i is a miss with a host row
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int32_t x = t[i];
        if (x == -1) continue;
        if (x < 0 || x >= S) { f |= kFlagBad; continue; }
        rid[i] = resident_row(rid[i], x, a.res_block_size);   // now the row
        if (rid[i] == -2) f |= kFlagBadRes;
        const uint32_t bit = 1u << (x & 31);
        if (sm.res_s) {
            // duplicates by token; a miss is a non-resident token without a slot
            if (atomicOr(&sm.dupbits[x >> 5], bit) & bit) f |= kFlagDup;
            if (rid[i] == -1 && !(sm.res_s[x >> 5] & bit)) {
                if (hb && sm.tbl_s[x / hb] < 0) {
                    f |= kFlagNoHost;
                } else {
                    miss |= 1u << i;
                    atomicOr(&sm.missbits[x >> 5], bit);
                }
            }
            continue;
        }
        if (rid[i] == -1 && s[i] < 0) {
            if (hb && sm.tbl_s[x / hb] < 0) f |= kFlagNoHost;
            else miss |= 1u << i;
        }
        if (rid[i] < 0 && s[i] >= 0) {
            const uint32_t sbit = 1u << (s[i] & 31);
            if (atomicOr(&sm.hitbits[s[i] >> 5], sbit) & sbit) f |= kFlagDup;
        } else {
            if (atomicOr(&sm.missbits[x >> 5], bit) & bit) f |= kFlagDup;
        }
    }

    // Arrival indices (warp-aggregated), and the early fetch: arrival j <
    // SR stages the row in shared memory row j by the bulk-copy engine; the
    // others become leftover j - SR.  The host row is known now; only the
    // victim slot waits for the scans below.
    const uint8_t *hrow0 = a.store.host + (hb ? 0 : off) * B;
    uint8_t *drow0 = a.store.dev + (int64_t)r * D * B;
    PackedIdx<KT> arr;    // arrival index of entry i (a miss), else -1
    uint32_t staged_bytes = 0;
    uint32_t flags, m_all;
    if (!sm.res_s) cp_async_wait_all();   // the LRU list, published by the next barrier
    number_misses<KT>(miss, f, sm.warp_tot, arr, flags, m_all);
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int32_t j = arr.get(i);
        if (j < 0) continue;
        if (j < SR) staged_bytes += (uint32_t)B;
        else sm.left_row[j - SR] = host_slot(t[i]);
    }
    if (SR) {
        mbar_arrive_expect_tx(sm.bar, staged_bytes);
#pragma unroll
        for (int i = 0; i < KT; ++i) {
            const int32_t j = arr.get(i);
            if (j >= 0 && j < SR)
                bulk_load(sm.stage + (int64_t)j * B, hrow0 + (int64_t)host_slot(t[i]) * B,
                          (uint32_t)B, sm.bar);
        }
    }
    // Copiers: the list goes out now (count 0 on an error: nothing to copy).
    // Phase 2 follows only if the count is nonzero (`copying`); a copier
    // that reads 0 leaves after phase 1.
    // The leftover rows are in shared memory (for the early loads below),
    // and with copiers they go out now: 16 bytes a thread, then the count (0
    // on an error: nothing to copy), released by the first cluster barrier.
    // Phase 2 follows only if the count is nonzero (`copying`); a copier that
    // reads 0 leaves after phase 1.
    __syncthreads();
    const bool copying = ncopy && !flags && m_all > 0u;
    // With the resident-token bitmap the copiers classify for themselves and
    // build the same list (self_list): one cluster barrier, at which this
    // CTA arrives once it has filed the victims and set sm.pub[1] (0: no
    // copy) in their shared memory, on every path.  Otherwise the list goes
    // to them here, with two barriers.
    const bool self_list = ncopy && sm.res_s;
    if (ncopy && !self_list) {
        if (copying) copy_to_copiers(sm.left_row, (m_all * 4u + 15u) / 16u * 16u, ncopy);
        if (tid == 0)
            for (int q = 1; q <= ncopy; ++q) st_remote_u32(&sm.pub[0], q, flags ? 0u : m_all);
        cluster_arrive();
    }
    if (flags) {
        // staged rows may still be landing in shared memory
        if (SR) staged_rows_landed(sm.bar, a.status, r);
#pragma unroll
        for (int i = 0; i < KT; ++i) rid[i] = -1;
        finish_untouched<KT>(a, r, t, rid, status_of(flags), tick);
        if (self_list) {
            if (tid == 0)
                for (int q = 1; q <= ncopy; ++q) st_remote_u32(&sm.pub[1], q, 0u);
            cluster_arrive();
        } else if (ncopy) {
            cluster_wait();
        }
        return;
    }

    // Leftover chunks: chunk e is chunk e % CH of leftover e / CH.  Thread
    // tid copies chunks tid, tid + NT, tid + 2 NT, ...; the first EARLY of
    // them are loaded now and stored after the state writes below.  In a
    // call without errors every miss took one arrival index, so the count is
    // the call's miss count m.  (A request with many misses can leave its
    // copies to a full-GPU copy grid launched behind this kernel.)
    const int m_arr = (int)m_all;
    const bool defer = a.deferred && (int64_t)m_arr * B > a.defer_bytes;
    const int nleft = (a.fused_copy && !defer && !ncopy) ? max(m_arr - SR, 0) : 0;
    const CopyWalk walk = a.aligned_rows ? CopyWalk(true, nleft, CH, tid >> 5, NT / 32, hrow0, B)
                                         : CopyWalk(false, nleft, CH, tid, NT, hrow0, B);
    const int32_t *lrow = sm.left_row;
    uint4 pv[COPY_WINDOW];
    CopyCursor cur_ld = walk.start;
#pragma unroll
    for (int u = 0; u < EARLY; ++u) {
        int32_t hr;
        int c;
        if (walk.at(cur_ld, lrow, hr, c)) pv[u] = ld_host_v4(hrow0 + (int64_t)hr * B + c * 16);
        walk.next(cur_ld);
    }
    late_grid_wait(a);   // the first global writes follow

    if (sm.res_s) {
        // The hits' slots, from the inverse table of the staged slot->token
        // row (landed by now, with the LRU list): every slot files itself
        // under its token; a hit's entry is the slot that holds it.
        cp_async_wait_all();
        __syncthreads();
        for (int sl = tid; sl < D; sl += NT) {
            const int32_t x = sm.s2t_s[sl];
            if (x >= 0 && x < a.max_cap) sm.inv[x] = (uint16_t)sl;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < KT; ++i) {
            if (t[i] < 0 || t[i] >= S || rid[i] != -1 || ((miss >> i) & 1u)) continue;
            const int v = sm.inv[t[i]];
            if (v < D && sm.s2t_s[v] == t[i]) {
                s[i] = v;
                atomicOr(&sm.hitbits[v >> 5], 1u << (v & 31));
            }
        }
        __syncthreads();   // the hit bitmap is complete
    }

    if (a.resident) {
#pragma unroll
        for (int i = 0; i < KT; ++i)
            if (t[i] >= 0 && rid[i] >= 0) atomicAnd(&sm.missbits[t[i] >> 5], ~(1u << (t[i] & 31)));
        __syncthreads();
    }
    // resident positions, hits and padding resolve now
    int32_t *out = a.out + (int64_t)r * k;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int j = tid + i * NT;
        if (j >= k) continue;
        if (t[i] < 0) out[j] = -1;
        else if (rid[i] >= 0) out[j] = kResidentFlag | rid[i];
        else if (s[i] >= 0) out[j] = s[i];
    }

    // One prefix sum gives both (a) the misses before each thread's chunk of
    // miss-bitmap words and (b) the non-hit list entries before each
    // thread's chunk of the LRU list.
    const int C = (D + NT - 1) / NT;
    const int e0 = min(tid * C, D), e1 = min(e0 + C, D);
    const int WC = (mw + NT - 1) / NT;
    const int w0 = min(tid * WC, mw), w1 = min(w0 + WC, mw);
    uint32_t nh = 0, mc = 0;
    for (int e = e0; e < e1; ++e) nh += !test_bit(sm.hitbits, sm.lru_s[e]);
    for (int w = w0; w < w1; ++w) mc += __popc(sm.missbits[w]);
    uint32_t tot;
    const uint32_t pre = block_exclusive_scan<NT>((mc << 16) | nh, sm.warp_tot, tot);
    const int m = (int)(tot >> 16);
    const int h = D - (int)(tot & 0xFFFFu);
    sm.chunk_pre[tid] = (uint16_t)(pre >> 16);

    // Protected slots ([Arch] Resident device pages: a later verification
    // step may not reuse a hot row before an earlier step has consumed it):
    // with P > 0, victims need a stamp below max(1, tick - P).  The list is
    // sorted by stamp, so it is enough that the last victim, the m-th non-hit
    // entry, has one; its owner looks the stamp up and tells the CTA.
    if (a.protect_calls && m > 0) {
        const uint32_t thr = tick > a.protect_calls ? tick - a.protect_calls : 1u;
        uint32_t q = pre & 0xFFFFu;
        __syncthreads();   // the scan's total is read; warp_tot[0] is free again
        for (int e = e0; e < e1; ++e) {
            const int sl = sm.lru_s[e];
            if (test_bit(sm.hitbits, sl)) continue;
            if ((int)q == m - 1)
                sm.warp_tot[0] = a.st.last_used[(int64_t)r * D + sl] >= thr ? 1u : 0u;
            ++q;
        }
        __syncthreads();
        if (sm.warp_tot[0]) {
            if (SR) staged_rows_landed(sm.bar, a.status, r);
            finish_untouched<KT>(a, r, t, rid, kStatusCapacity, tick);
            if (self_list) {   // no copy after all
                if (tid == 0)
                    for (int q = 1; q <= ncopy; ++q) st_remote_u32(&sm.pub[1], q, 0u);
                cluster_arrive();
            } else if (ncopy) {
                cluster_wait();
                if (copying) {   // the copiers wait in phase 2: no copy after all
                    if (tid == 0)
                        for (int q = 1; q <= ncopy; ++q) st_remote_u32(&sm.pub[1], q, 0u);
                    cluster_arrive();
                    cluster_wait();
                }
            }
            return;
        }
    }

    // Victims = the first m non-hit list entries; the rest keep their order
    // at the front of the new list.
    uint16_t *lru_w = a.st.lru + (int64_t)r * D;
    {
        uint32_t q = pre & 0xFFFFu;
        for (int e = e0; e < e1; ++e) {
            const int sl = sm.lru_s[e];
            if (test_bit(sm.hitbits, sl)) continue;
            if ((int)q < m) {
                sm.victims[q] = (uint16_t)sl;
                atomicOr(&sm.selbits[sl >> 5], 1u << (sl & 31));
            } else {
                lru_w[q - m] = (uint16_t)sl;
            }
            ++q;
        }
    }
    __syncthreads();

    // Each miss's victim: misses take victims by ascending token rank, and
    // each victim is also filed under the miss's arrival index, where the
    // copies look it up.  With self-classifying copiers the victims go out
    // before this CTA's global state writes, so the copiers' stores wait for
    // nothing else.
    int32_t vict[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        vict[i] = -1;
        const int j = tid + i * NT;
        const int32_t x = t[i];
        if (j >= k || x < 0 || rid[i] >= 0 || s[i] >= 0) continue;
        const int w = x >> 5;
        const int owner = w / WC;
        uint32_t rank = sm.chunk_pre[owner];
        for (int q = owner * WC; q < w; ++q) rank += __popc(sm.missbits[q]);
        rank += __popc(sm.missbits[w] & ((1u << (x & 31)) - 1u));
        const int v = sm.victims[rank];
        sm.arr_vict[arr.get(i)] = (uint16_t)v;
        vict[i] = v | (int32_t)(rank << 16);   // slot (< 65536) and rank (< k)
    }
    if (self_list) {
        if (copying) {
            __syncthreads();
            copy_to_copiers(sm.arr_vict, (m_all * 2u + 15u) / 16u * 16u, ncopy);
        }
        if (tid == 0)
            for (int q = 1; q <= ncopy; ++q) st_remote_u32(&sm.pub[1], q, copying ? 1u : 0u);
        cluster_arrive();
    }
    // The resident-token bitmap row in global memory, if kept: evicted tokens
    // leave it, misses enter it (atomics: threads share its words).
    uint32_t *resg = a.st.resbits ? a.st.resbits + (int64_t)r * a.st.res_words : nullptr;
    // State writes (stores only: no load of their own to wait for).
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        if (vict[i] < 0) continue;
        const int j = tid + i * NT;
        const int32_t x = t[i];
        const int v = vict[i] & 0xFFFF;
        const uint32_t rank = (uint32_t)vict[i] >> 16;
        const int32_t old = sm.s2t_s ? sm.s2t_s[v] : slot2tok[v];
        if (old >= 0 && (int64_t)old < cap) {
            tok2slot[old] = -1;
            if (resg) atomicAnd(&resg[old >> 5], ~(1u << (old & 31)));
        }
        slot2tok[v] = x;
        tok2slot[x] = v;
        if (resg) atomicOr(&resg[x >> 5], 1u << (x & 31));
        out[j] = v;
        if (a.plan_rows) {
            int32_t *pr = a.plan_rows + ((int64_t)r * k + rank) * 2;
            pr[0] = host_slot(x);
            pr[1] = v;
        }
    }
    // Message protocol: the copiers may store their rows now (phase 2).
    if (!self_list && ncopy) {
        cluster_wait();
        if (copying) {
            __syncthreads();
            copy_to_copiers(sm.arr_vict, (m_all * 2u + 15u) / 16u * 16u, ncopy);
            if (tid == 0)
                for (int q = 1; q <= ncopy; ++q) st_remote_u32(&sm.pub[1], q, 1u);
            cluster_arrive();
        }
    }
    // Selected slots (hits and victims) go to the back of the list in slot
    // order and are stamped with the tick.  (The scan's barriers also publish
    // the leftover victims written above.)
    {
        uint32_t *last_used = a.st.last_used + (int64_t)r * D;
        const uint32_t w = tid < DW ? (sm.hitbits[tid] | sm.selbits[tid]) : 0u;
        uint32_t tot2;
        uint32_t pos = (uint32_t)(D - h - m) + block_exclusive_scan<NT>(__popc(w), sm.warp_tot, tot2);
        uint32_t bits = w;
        while (bits) {
            const int b = __ffs(bits) - 1;
            bits &= bits - 1u;
            const int sl = tid * 32 + b;
            lru_w[pos++] = (uint16_t)sl;
            last_used[sl] = tick;
        }
    }
    if (tid == 0) {
        if (a.plan_counts) a.plan_counts[r] = m;
        if (a.deferred) a.deferred[r] = defer ? 1 : 0;
        a.st.tick[r] = tick;
    }
    if (copying && !self_list) cluster_wait();

    // ---- miss copies: pinned host rows -> victim slots ---------------------
    // The leftovers through a window of COPY_WINDOW loads per thread: the
    // rest of the window is loaded now; then each stored chunk's register
    // takes the load of the thread's chunk COPY_WINDOW steps ahead.  Loads
    // return in about the order they were issued, so every thread keeps
    // COPY_WINDOW loads in flight until its last ones.
#pragma unroll
    for (int u = EARLY; u < COPY_WINDOW; ++u) {
        int32_t hr;
        int c;
        if (walk.at(cur_ld, lrow, hr, c)) pv[u] = ld_host_v4(hrow0 + (int64_t)hr * B + c * 16);
        walk.next(cur_ld);
    }
    CopyCursor cur_st = walk.start;
    while (!walk.done(cur_st)) {
#pragma unroll
        for (int u = 0; u < COPY_WINDOW; ++u) {
            int32_t hr;
            int c;
            if (walk.at(cur_st, lrow, hr, c))
                st_v4(drow0 + (int64_t)sm.arr_vict[SR + cur_st.q] * B + c * 16, pv[u]);
            walk.next(cur_st);
            if (walk.at(cur_ld, lrow, hr, c)) pv[u] = ld_host_v4(hrow0 + (int64_t)hr * B + c * 16);
            walk.next(cur_ld);
        }
    }
    // the staged rows, once they have all landed, one bulk store per row
    if (SR) {
        if (!staged_rows_landed(sm.bar, a.status, r)) return;
        const int nstaged = min(m_arr, SR);
        if (tid < nstaged) {
            fence_proxy_async();
            for (int j = tid; j < nstaged; j += NT)
                bulk_store(drow0 + (int64_t)sm.arr_vict[j] * B, sm.stage + (int64_t)j * B,
                           (uint32_t)B);
            bulk_commit();
            bulk_wait_read();
        }
    }
}

template <int KT>
cudaError_t launch_kt(const ResolveLaunch &a, cudaStream_t s, size_t smem)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.g.R * (1 + a.ncopy));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (a.programmatic) {
        // programmatic dependency on the previous kernel of the stream: this
        // grid may be placed before that one ends and waits for it on the
        // device (griddepcontrol.wait at the kernel's start)
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (a.ncopy) {
        // one cluster per request: the resolver and its copiers
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 1 + a.ncopy;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, resolve_kernel<KT>, a);
}

template <int KT>
cudaError_t prepare_kt(size_t smem)
{
    return cudaFuncSetAttribute(resolve_kernel<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
}

}  // namespace

size_t resolve_smem_bytes(int k, int D, int max_cap, bool stage_s2t, int lookup, int tbl_stride,
                          int stage_rows, int64_t B)
{
    return plan_smem(k, D, max_cap, stage_s2t, lookup, tbl_stride, stage_rows, B).total;
}

int resolve_stage_rows(int k, int D, int max_cap, bool stage_s2t, int lookup, int tbl_stride,
                       int64_t B, size_t max_smem)
{
    const size_t base = resolve_smem_bytes(k, D, max_cap, stage_s2t, lookup, tbl_stride, 0, B);
    const size_t room = align_up(base, 128) + 16 <= max_smem ? max_smem - align_up(base, 128) - 16 : 0;
    const int64_t rows = (int64_t)(room / (size_t)B);
    return (int)(rows < k ? rows : k);
}

int resolve_threads() { return NT; }

cudaError_t resolve_prepare(size_t smem)
{
    cudaError_t e = prepare_kt<1>(smem);
    if (e == cudaSuccess) e = prepare_kt<2>(smem);
    if (e == cudaSuccess) e = prepare_kt<4>(smem);
    if (e == cudaSuccess) e = prepare_kt<8>(smem);
    return e;
}

template <int KT>
cudaError_t max_clusters_kt(int ctas, size_t smem, int *clusters)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, resolve_kernel<KT>, &cfg);
}

cudaError_t resolve_max_clusters(int k, int ctas, size_t smem, int *clusters)
{
    const int kt = (k + NT - 1) / NT;
    if (kt <= 1) return max_clusters_kt<1>(ctas, smem, clusters);
    if (kt <= 2) return max_clusters_kt<2>(ctas, smem, clusters);
    if (kt <= 4) return max_clusters_kt<4>(ctas, smem, clusters);
    return max_clusters_kt<8>(ctas, smem, clusters);
}

cudaError_t launch_resolve(const ResolveLaunch &a_in, cudaStream_t s)
{
    const SmemPlan p = plan_smem(a_in.g.k, a_in.g.D, a_in.max_cap, a_in.stage_s2t, a_in.lookup,
                                 a_in.g.hb ? a_in.g.tbl_stride : 0, a_in.stage_rows, a_in.g.B);
    if (p.total > (size_t)UINT32_MAX) return cudaErrorInvalidValue;
    ResolveLaunch a = a_in;
    a.smem = ResolveSmem{(uint32_t)p.hit,  (uint32_t)p.sel,   (uint32_t)p.miss, (uint32_t)p.lru,
                         (uint32_t)p.s2t,  (uint32_t)p.inv,   (uint32_t)p.res,  (uint32_t)p.dup,
                         (uint32_t)p.tbl,  (uint32_t)p.chunk, (uint32_t)p.vict, (uint32_t)p.lrow,
                         (uint32_t)p.avict, (uint32_t)p.bar,  (uint32_t)p.cnt,  (uint32_t)p.stage};
    const int kt = (a.g.k + NT - 1) / NT;
    if (kt <= 1) return launch_kt<1>(a, s, p.total);
    if (kt <= 2) return launch_kt<2>(a, s, p.total);
    if (kt <= 4) return launch_kt<4>(a, s, p.total);
    return launch_kt<8>(a, s, p.total);
}

}  // namespace hs
