// resolve.cu -- the swap-in resolver kernel.
//
// One CTA of 1024 threads resolves one request's top-k for one call
// ([Guide] "HiSparse: Hierarchical Sparse Attention", Decode Workflow: fast
// path for short sequences; otherwise hit detection -> LRU reorder -> miss
// handling with a host-to-device copy; [Arch] "HiSparse local KV offload
// architecture", Hot lookup and LRU: a hot row is used in place and
// refreshes the GPU LRU, a miss takes the LRU victim and copies the pinned
// host row into it).
//
// The miss copies cross the host link and dominate the call, so everything
// else is arranged around starting them early and keeping them going:
//   1. the LRU list is staged into shared memory with asynchronous copies
//      issued at kernel start, under the first global round trips;
//   2. once the sorted miss list exists, every thread loads its first host
//      chunks into registers, and those loads are in flight while the
//      victims are chosen;
//   3. the slot->token row is staged too, so once the victims are known all
//      state writes are plain stores with no loads of their own (they still
//      queue behind the thread's host loads in flight, which keep the link
//      busy meanwhile); they are issued before the prefetched rows are
//      consumed, then every thread streams the rest of the rows.
//
// With a paged host pool ([Arch] Ownership: tokens map to logical host
// blocks), the request's host block table row is staged as well, under the
// token->slot round trip; a miss whose block is not reserved stops the call
// for that request (status NO_HOST_ROW), and miss rows are addressed, and
// recorded in the plan, by their row in the layer's pool.
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
// Host chunks per thread loaded before the victims are chosen, by the number
// of top-k entries per thread.  Deeper is faster (decode_40k, measured: 4
// -> 8 took a step from 54.1 to 52.3 us), as far as the 64 registers of a
// 1024-thread CTA hold them without spilling.
template <int KT> __host__ __device__ constexpr int prefetch_depth() { return KT == 2 ? 8 : 4; }
// Host chunks in flight per thread in the copy loop.  Measured on decode_40k
// (32 CTAs): 4 ends the launch ~1.3 us sooner than 8; 2 and 6 gain less, and
// with 128 or 256 CTAs the depth makes no difference.
constexpr int COPY_UNROLL = 4;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct SmemPlan {
    size_t hit, sel, miss, lru, s2t, tbl, chunk, vict, mtok, total;
};

// Shared memory of the CTA: bitmaps over slots and tokens, the staged LRU
// list, optionally the staged slot->token row and host block table row, and
// miss rows and victims by miss rank.
__host__ __device__ inline SmemPlan plan_smem(int k, int D, int max_cap, bool stage_s2t,
                                              int tbl_stride)
{
    SmemPlan p;
    const size_t DW = (size_t)(D + 31) / 32, MW = (size_t)(max_cap + 31) / 32;
    size_t o = 32 * 4;             // warp totals
    p.hit = o;   o += DW * 4;
    p.sel = o;   o += DW * 4;
    p.miss = o;  o += MW * 4;
    p.lru = align_up(o, 16); o = p.lru + align_up((size_t)D * 2, 16);
    p.s2t = o;   o += stage_s2t ? align_up((size_t)D * 4, 16) : 0;
    p.tbl = o;   o += (size_t)tbl_stride * 4;   // a multiple of 16
    p.chunk = o; o = align_up(o + (size_t)NT * 2, 4);
    p.vict = o;  o = align_up(o + (size_t)k * 2, 4);
    p.mtok = o;  o += (size_t)k * 4;
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
    int32_t *tbl_s;      // [tbl_stride] staged host block table row (null: no paged pool)
    uint16_t *chunk_pre; // [NT]  misses before each thread's chunk of missbits
    uint16_t *victims;   // [k]   victim slot of miss rank i
    int32_t *misstok;    // [k]   host row of miss rank i (token, or pool row when paged)
};

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

// Resident row of position t from its block id `id` (-1: not resident), or
// -2 when the id is malformed (below -1, or rows reaching the flag bit).
__device__ __forceinline__ int32_t resident_row(int32_t id, int32_t t, int32_t bs)
{
    if (id == -1) return -1;
    if (id < -1 || (int64_t)id * bs + bs > kResidentFlag) return -2;
    return id * bs + t % bs;
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

template <int KT>
__global__ void __launch_bounds__(NT, 1) resolve_kernel(ResolveLaunch a)
{
    constexpr int PREFETCH = prefetch_depth<KT>();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int k = a.g.k, D = a.g.D;
    const int DW = (D + 31) >> 5;

    const int32_t hb = a.g.hb;
    const SmemPlan sp = plan_smem(k, D, a.max_cap, a.stage_s2t, hb ? a.g.tbl_stride : 0);
    Smem sm;
    sm.warp_tot = reinterpret_cast<uint32_t *>(smem_raw);
    sm.hitbits = reinterpret_cast<uint32_t *>(smem_raw + sp.hit);
    sm.selbits = reinterpret_cast<uint32_t *>(smem_raw + sp.sel);
    sm.missbits = reinterpret_cast<uint32_t *>(smem_raw + sp.miss);
    sm.lru_s = reinterpret_cast<uint16_t *>(smem_raw + sp.lru);
    sm.s2t_s = a.stage_s2t ? reinterpret_cast<int32_t *>(smem_raw + sp.s2t) : nullptr;
    sm.tbl_s = hb ? reinterpret_cast<int32_t *>(smem_raw + sp.tbl) : nullptr;
    sm.chunk_pre = reinterpret_cast<uint16_t *>(smem_raw + sp.chunk);
    sm.victims = reinterpret_cast<uint16_t *>(smem_raw + sp.vict);
    sm.misstok = reinterpret_cast<int32_t *>(smem_raw + sp.mtok);

    // A copy grid launched with a programmatic dependency may be scheduled
    // now; it still waits for this grid to finish before reading the plan.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

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
    // Stage the LRU list and the slot->token row with asynchronous copies;
    // they land under the round trips above.  (16-byte rows need D % 8 == 0.)
    const uint16_t *lru = a.st.lru + (int64_t)r * D;
    int32_t *slot2tok = a.st.slot2tok + (int64_t)r * D;
    const bool staged_async = (D & 7) == 0;
    if (staged_async) {
        for (int i = tid; i < (D >> 3); i += NT) cp_async16(sm.lru_s + i * 8, lru + i * 8);
        if (sm.s2t_s)
            for (int i = tid; i < (D >> 2); i += NT) cp_async16(sm.s2t_s + i * 4, slot2tok + i * 4);
    }
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
        __syncthreads();
        bool bad = false, dup = false, badres = false;
#pragma unroll
        for (int i = 0; i < KT; ++i) {
            const int32_t x = t[i];
            if (x == -1) continue;
            if (x < 0 || x >= S) { bad = true; continue; }
            badres |= resident_row(rid[i], x, a.res_block_size) == -2;
            const uint32_t bit = 1u << (x & 31);
            dup |= (atomicOr(&sm.missbits[x >> 5], bit) & bit) != 0u;
        }
        bad = __syncthreads_or(bad);
        dup = __syncthreads_or(dup);
        badres = __syncthreads_or(badres);
        finish_untouched<KT>(a, r, t, rid,
                             bad ? kStatusBadIndex
                                 : (dup ? kStatusDuplicate : (badres ? kStatusBadResident : kStatusOk)),
                             tick);
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
    int32_t *tok2slot = a.st.tok2slot + off;
    int32_t s[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        s[i] = (t[i] >= 0 && t[i] < S) ? tok2slot[t[i]] : -1;
        if (s[i] >= D) s[i] = -1;  // never true for state this library wrote
    }
    const int mw = (S + 31) >> 5;
    for (int w = tid; w < mw; w += NT) sm.missbits[w] = 0u;
    for (int w = tid; w < DW; w += NT) { sm.hitbits[w] = 0u; sm.selbits[w] = 0u; }
    if (!staged_async) {
        for (int i = tid; i < D; i += NT) sm.lru_s[i] = lru[i];
        if (sm.s2t_s)
            for (int i = tid; i < D; i += NT) sm.s2t_s[i] = slot2tok[i];
    }
    cp_async_wait_all();
    __syncthreads();

    // Classify.  A resident position is marked in the token bitmap only to
    // catch duplicates; its bit is cleared again before the misses are
    // ranked, and it never touches the hot state.
    bool bad = false, dup = false, badres = false, nohost = false;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int32_t x = t[i];
        if (x == -1) continue;
        if (x < 0 || x >= S) { bad = true; continue; }
        rid[i] = resident_row(rid[i], x, a.res_block_size);   // now the row
        badres |= rid[i] == -2;
        if (rid[i] == -1 && s[i] < 0 && hb) nohost |= sm.tbl_s[x / hb] < 0;
        if (rid[i] < 0 && s[i] >= 0) {
            const uint32_t bit = 1u << (s[i] & 31);
            dup |= (atomicOr(&sm.hitbits[s[i] >> 5], bit) & bit) != 0u;
        } else {
            const uint32_t bit = 1u << (x & 31);
            dup |= (atomicOr(&sm.missbits[x >> 5], bit) & bit) != 0u;
        }
    }
    bad = __syncthreads_or(bad);
    dup = __syncthreads_or(dup);
    badres = __syncthreads_or(badres);
    nohost = __syncthreads_or(nohost);
    if (bad || dup || badres || nohost) {
#pragma unroll
        for (int i = 0; i < KT; ++i) rid[i] = -1;
        finish_untouched<KT>(a, r, t, rid,
                             bad ? kStatusBadIndex
                                 : (dup ? kStatusDuplicate
                                        : (badres ? kStatusBadResident : kStatusNoHostRow)),
                             tick);
        return;
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
    {   // the sorted miss list: enumerate this thread's words in order
        uint32_t rank = pre >> 16;
        for (int w = w0; w < w1; ++w) {
            uint32_t bits = sm.missbits[w];
            while (bits) {
                const int b = __ffs(bits) - 1;
                bits &= bits - 1u;
                sm.misstok[rank++] = host_slot(w * 32 + b);
            }
        }
    }
    __syncthreads();

    // Protected slots ([Arch] Resident device pages: a later verification
    // step may not reuse a hot row before an earlier step has consumed it):
    // with P > 0, victims need a stamp below max(1, tick - P).  The list is
    // sorted by stamp, so it is enough that the last victim, the m-th non-hit
    // entry, has one; its owner looks the stamp up and tells the CTA.
    if (a.protect_calls && m > 0) {
        const uint32_t thr = tick > a.protect_calls ? tick - a.protect_calls : 1u;
        uint32_t q = pre & 0xFFFFu;
        for (int e = e0; e < e1; ++e) {
            const int sl = sm.lru_s[e];
            if (test_bit(sm.hitbits, sl)) continue;
            if ((int)q == m - 1)
                sm.warp_tot[0] = a.st.last_used[(int64_t)r * D + sl] >= thr ? 1u : 0u;
            ++q;
        }
        __syncthreads();
        if (sm.warp_tot[0]) {
            finish_untouched<KT>(a, r, t, rid, kStatusCapacity, tick);
            return;
        }
    }

    // First host chunks: loaded now, stored after the state writes below.
    const int64_t B = a.g.B;
    const int CH = a.g.chunks;
    // A request with many misses can leave its copies to a full-GPU copy
    // grid launched behind this kernel: one SM alone moves them slowly.
    const bool defer = a.deferred && (int64_t)m * B > a.defer_bytes;
    const int total = (a.fused_copy && !defer) ? m * CH : 0;
    const uint8_t *hrow0 = a.store.host + (hb ? 0 : off) * B;
    uint8_t *drow0 = a.store.dev + (int64_t)r * D * B;
    uint4 pv[PREFETCH];
#pragma unroll
    for (int u = 0; u < PREFETCH; ++u) {
        const int e = tid + u * NT;
        if (e < total) {
            const int i = e / CH, c = e - i * CH;
            pv[u] = ld_host_v4(hrow0 + (int64_t)sm.misstok[i] * B + c * 16);
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

    // State writes (stores only: no load of their own to wait for).  Misses
    // take victims by ascending token rank.
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int j = tid + i * NT;
        const int32_t x = t[i];
        if (j >= k || x < 0 || rid[i] >= 0 || s[i] >= 0) continue;
        const int w = x >> 5;
        const int owner = w / WC;
        uint32_t rank = sm.chunk_pre[owner];
        for (int q = owner * WC; q < w; ++q) rank += __popc(sm.missbits[q]);
        rank += __popc(sm.missbits[w] & ((1u << (x & 31)) - 1u));
        const int v = sm.victims[rank];
        const int32_t old = sm.s2t_s ? sm.s2t_s[v] : slot2tok[v];
        if (old >= 0 && (int64_t)old < cap) tok2slot[old] = -1;
        slot2tok[v] = x;
        tok2slot[x] = v;
        out[j] = v;
        if (a.plan_rows) {
            int32_t *pr = a.plan_rows + ((int64_t)r * k + rank) * 2;
            pr[0] = host_slot(x);
            pr[1] = v;
        }
    }
    // Selected slots (hits and victims) go to the back of the list in slot
    // order and are stamped with the tick.
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

    // ---- miss copies: pinned host rows -> victim slots ---------------------
#pragma unroll
    for (int u = 0; u < PREFETCH; ++u) {
        const int e = tid + u * NT;
        if (e < total) {
            const int i = e / CH, c = e - i * CH;
            st_v4(drow0 + (int64_t)sm.victims[i] * B + c * 16, pv[u]);
        }
    }
    for (int e = PREFETCH * NT + tid; e < total; e += NT * COPY_UNROLL) {
        uint4 v[COPY_UNROLL];
        uint8_t *dst[COPY_UNROLL];
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
            const int ee = e + u * NT;
            dst[u] = nullptr;
            if (ee < total) {
                const int i = ee / CH, c = ee - i * CH;
                v[u] = ld_host_v4(hrow0 + (int64_t)sm.misstok[i] * B + c * 16);
                dst[u] = drow0 + (int64_t)sm.victims[i] * B + c * 16;
            }
        }
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u)
            if (dst[u]) st_v4(dst[u], v[u]);
    }
}

template <int KT>
cudaError_t launch_kt(const ResolveLaunch &a, cudaStream_t s, size_t smem)
{
    resolve_kernel<KT><<<a.g.R, NT, smem, s>>>(a);
    return cudaGetLastError();
}

template <int KT>
cudaError_t prepare_kt(size_t smem)
{
    return cudaFuncSetAttribute(resolve_kernel<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
}

}  // namespace

size_t resolve_smem_bytes(int k, int D, int max_cap, bool stage_s2t, int tbl_stride)
{
    return plan_smem(k, D, max_cap, stage_s2t, tbl_stride).total;
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

cudaError_t launch_resolve(const ResolveLaunch &a, cudaStream_t s)
{
    const size_t smem = resolve_smem_bytes(a.g.k, a.g.D, a.max_cap, a.stage_s2t,
                                           a.g.hb ? a.g.tbl_stride : 0);
    const int kt = (a.g.k + NT - 1) / NT;
    if (kt <= 1) return launch_kt<1>(a, s, smem);
    if (kt <= 2) return launch_kt<2>(a, s, smem);
    if (kt <= 4) return launch_kt<4>(a, s, smem);
    return launch_kt<8>(a, s, smem);
}

}  // namespace hs
