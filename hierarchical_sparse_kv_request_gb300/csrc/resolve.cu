// resolve.cu -- the swap-in resolver kernel.
//
// One CTA resolves one request's top-k for one call ([Guide] "HiSparse:
// Hierarchical Sparse Attention", Decode Workflow: fast path for short
// sequences; otherwise hit detection -> LRU reorder -> miss handling with a
// host-to-device copy; [Arch] "HiSparse local KV offload architecture", Hot
// lookup and LRU: a hot row is used in place and refreshes the GPU LRU, a
// miss takes the LRU victim and copies the pinned host row into it).
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
//
// Every global access below is a coalesced row/array access or a single
// gather of the token->slot map; there are no loops over keys.
#include "hs_common.cuh"

namespace hs {
namespace {

constexpr int NT = 1024;       // threads per CTA
constexpr int COPY_UNROLL = 8;  // 16-byte host loads in flight per thread

struct Smem {
    uint32_t *warp_tot;  // [32]
    uint32_t *hitbits;   // [DW]  slots hit by this call
    uint32_t *selbits;   // [DW]  slots chosen as victims
    uint32_t *missbits;  // [MW]  miss tokens (and, on the fast path, all tokens)
    uint16_t *lru_s;     // [D]   staged LRU list
    uint16_t *chunk_pre; // [NT]  misses before each thread's chunk of missbits
    uint16_t *victims;   // [k]   victim slot of miss rank i
    int32_t *misstok;    // [k]   token of miss rank i
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct SmemPlan {
    size_t hit, sel, miss, lru, chunk, vict, mtok, total;
};

__host__ __device__ inline SmemPlan plan_smem(int k, int D, int max_cap)
{
    SmemPlan p;
    const size_t DW = (size_t)(D + 31) / 32, MW = (size_t)(max_cap + 31) / 32;
    size_t o = 32 * 4;
    p.hit = o;   o += DW * 4;
    p.sel = o;   o += DW * 4;
    p.miss = o;  o += MW * 4;
    p.lru = o;   o = align_up(o + (size_t)D * 2, 4);
    p.chunk = o; o = align_up(o + (size_t)NT * 2, 4);
    p.vict = o;  o = align_up(o + (size_t)k * 2, 4);
    p.mtok = o;  o += (size_t)k * 4;
    p.total = align_up(o, 16);
    return p;
}

__device__ __forceinline__ bool test_bit(const uint32_t *bits, int i)
{
    return (bits[i >> 5] >> (i & 31)) & 1u;
}

// Final writes of a request whose call ends without touching its state.
template <int KT>
__device__ __forceinline__ void finish_untouched(const ResolveLaunch &a, int r,
                                                 const int32_t (&t)[KT], int status,
                                                 uint32_t tick)
{
    const int k = a.g.k;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int j = threadIdx.x + i * NT;
        if (j < k) a.out[(int64_t)r * k + j] = status == kStatusOk ? t[i] : -1;
    }
    if (threadIdx.x == 0) {
        a.status[r] = status;
        if (a.plan_counts) a.plan_counts[r] = 0;
        a.st.tick[r] = tick;
    }
}

template <int KT>
__global__ void __launch_bounds__(NT, 1) resolve_kernel(ResolveLaunch a)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int k = a.g.k, D = a.g.D;
    const int DW = (D + 31) >> 5;

    const SmemPlan sp = plan_smem(k, D, a.max_cap);
    Smem sm;
    sm.warp_tot = reinterpret_cast<uint32_t *>(smem_raw);
    sm.hitbits = reinterpret_cast<uint32_t *>(smem_raw + sp.hit);
    sm.selbits = reinterpret_cast<uint32_t *>(smem_raw + sp.sel);
    sm.missbits = reinterpret_cast<uint32_t *>(smem_raw + sp.miss);
    sm.lru_s = reinterpret_cast<uint16_t *>(smem_raw + sp.lru);
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

    if (S < 0 || (int64_t)S > cap) {  // uniform across the CTA
        finish_untouched<KT>(a, r, t, kStatusBadSeqLen, tick);
        return;
    }

    // ---- fast path: every token is already at slot = token ---------------
    if (S <= D) {
        const int mw = (S + 31) >> 5;
        for (int w = tid; w < mw; w += NT) sm.missbits[w] = 0u;
        __syncthreads();
        bool bad = false, dup = false;
#pragma unroll
        for (int i = 0; i < KT; ++i) {
            const int32_t x = t[i];
            if (x == -1) continue;
            if (x < 0 || x >= S) { bad = true; continue; }
            const uint32_t bit = 1u << (x & 31);
            dup |= (atomicOr(&sm.missbits[x >> 5], bit) & bit) != 0u;
        }
        bad = __syncthreads_or(bad);
        dup = __syncthreads_or(dup);
        finish_untouched<KT>(a, r, t,
                             bad ? kStatusBadIndex : (dup ? kStatusDuplicate : kStatusOk), tick);
        return;
    }

    // ---- slow path --------------------------------------------------------
    int32_t *tok2slot = a.st.tok2slot + off;
    int32_t *slot2tok = a.st.slot2tok + (int64_t)r * D;
    uint32_t *last_used = a.st.last_used + (int64_t)r * D;
    uint16_t *lru = a.st.lru + (int64_t)r * D;

    // Hit detection: gather the token->slot map (issued before the barrier
    // so its latency overlaps the shared-memory clears and the list staging).
    int32_t s[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        s[i] = (t[i] >= 0 && t[i] < S) ? tok2slot[t[i]] : -1;
        if (s[i] >= D) s[i] = -1;  // never true for state this library wrote
    }

    const int mw = (S + 31) >> 5;
    for (int w = tid; w < mw; w += NT) sm.missbits[w] = 0u;
    for (int w = tid; w < DW; w += NT) { sm.hitbits[w] = 0u; sm.selbits[w] = 0u; }
    // stage the LRU list (pairs of slots when D is even, so rows stay 4-byte aligned)
    if ((D & 1) == 0) {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(lru);
        uint32_t *dst = reinterpret_cast<uint32_t *>(sm.lru_s);
        for (int i = tid; i < (D >> 1); i += NT) dst[i] = src[i];
    } else {
        for (int i = tid; i < D; i += NT) sm.lru_s[i] = lru[i];
    }
    __syncthreads();

    bool bad = false, dup = false;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int32_t x = t[i];
        if (x == -1) continue;
        if (x < 0 || x >= S) { bad = true; continue; }
        if (s[i] >= 0) {
            const uint32_t bit = 1u << (s[i] & 31);
            dup |= (atomicOr(&sm.hitbits[s[i] >> 5], bit) & bit) != 0u;
        } else {
            const uint32_t bit = 1u << (x & 31);
            dup |= (atomicOr(&sm.missbits[x >> 5], bit) & bit) != 0u;
        }
    }
    bad = __syncthreads_or(bad);
    dup = __syncthreads_or(dup);
    if (bad || dup) {
        finish_untouched<KT>(a, r, t, bad ? kStatusBadIndex : kStatusDuplicate, tick);
        return;
    }

    // One prefix sum gives both (a) the number of misses before each
    // thread's chunk of miss-bitmap words and (b) the number of non-hit list
    // entries before each thread's chunk of the LRU list.
    const int C = (D + NT - 1) / NT;   // list entries per thread
    const int e0 = min(tid * C, D), e1 = min(e0 + C, D);
    const int WC = (mw + NT - 1) / NT; // miss-bitmap words per thread
    const int w0 = min(tid * WC, mw), w1 = min(w0 + WC, mw);
    uint32_t nh = 0, mc = 0;
    for (int e = e0; e < e1; ++e) nh += !test_bit(sm.hitbits, sm.lru_s[e]);
    for (int w = w0; w < w1; ++w) mc += __popc(sm.missbits[w]);
    uint32_t tot;
    const uint32_t pre = block_exclusive_scan<NT>((mc << 16) | nh, sm.warp_tot, tot);
    const int m = (int)(tot >> 16);
    const int nonhit = (int)(tot & 0xFFFFu);
    const int h = D - nonhit;
    sm.chunk_pre[tid] = (uint16_t)(pre >> 16);

    // Victims = the first m non-hit list entries; the rest keep their order
    // at the front of the new list.
    {
        uint32_t q = pre & 0xFFFFu;
        for (int e = e0; e < e1; ++e) {
            const int sl = sm.lru_s[e];
            if (test_bit(sm.hitbits, sl)) continue;
            if ((int)q < m) {
                sm.victims[q] = (uint16_t)sl;
                atomicOr(&sm.selbits[sl >> 5], 1u << (sl & 31));
            } else {
                lru[q - m] = (uint16_t)sl;
            }
            ++q;
        }
    }
    __syncthreads();

    // Selected slots (hits and victims) go to the back of the list in slot
    // order and are stamped with the tick.
    {
        const uint32_t w = tid < DW ? (sm.hitbits[tid] | sm.selbits[tid]) : 0u;
        uint32_t tot2;
        uint32_t pos = (uint32_t)(D - h - m) + block_exclusive_scan<NT>(__popc(w), sm.warp_tot, tot2);
        uint32_t bits = w;
        while (bits) {
            const int b = __ffs(bits) - 1;
            bits &= bits - 1u;
            const int sl = tid * 32 + b;
            lru[pos++] = (uint16_t)sl;
            last_used[sl] = tick;
        }
    }

    // Outputs in input order; misses take victims by ascending token rank.
    int32_t *out = a.out + (int64_t)r * k;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        const int j = tid + i * NT;
        if (j >= k) continue;
        const int32_t x = t[i];
        if (x < 0) { out[j] = -1; continue; }
        if (s[i] >= 0) { out[j] = s[i]; continue; }
        const int w = x >> 5;
        const int owner = w / WC;
        uint32_t rank = sm.chunk_pre[owner];
        for (int q = owner * WC; q < w; ++q) rank += __popc(sm.missbits[q]);
        rank += __popc(sm.missbits[w] & ((1u << (x & 31)) - 1u));
        const int v = sm.victims[rank];
        const int32_t old = slot2tok[v];
        if (old >= 0 && (int64_t)old < cap) tok2slot[old] = -1;
        slot2tok[v] = x;
        tok2slot[x] = v;
        out[j] = v;
        sm.misstok[rank] = x;
        if (a.plan_rows) {
            int32_t *pr = a.plan_rows + ((int64_t)r * k + rank) * 2;
            pr[0] = x;
            pr[1] = v;
        }
    }
    if (tid == 0) {
        a.status[r] = kStatusOk;
        if (a.plan_counts) a.plan_counts[r] = m;
        a.st.tick[r] = tick;
    }
    if (!a.fused_copy || m == 0) return;

    // ---- fused miss copy: pinned host rows -> freed device slots ---------
    __syncthreads();
    const int64_t B = a.g.B;
    const int CH = a.g.chunks;
    const int total = m * CH;
    const uint8_t *hrow0 = a.store.host + off * B;
    uint8_t *drow0 = a.store.dev + (int64_t)r * D * B;
    for (int e = tid; e < total; e += NT * COPY_UNROLL) {
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
    cudaError_t e = cudaFuncSetAttribute(resolve_kernel<KT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    resolve_kernel<KT><<<a.g.R, NT, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t resolve_smem_bytes(int k, int D, int max_cap) { return plan_smem(k, D, max_cap).total; }
int resolve_threads() { return NT; }

cudaError_t launch_resolve(const ResolveLaunch &a, cudaStream_t s)
{
    const size_t smem = resolve_smem_bytes(a.g.k, a.g.D, a.max_cap);
    const int kt = (a.g.k + NT - 1) / NT;
    if (kt <= 1) return launch_kt<1>(a, s, smem);
    if (kt <= 2) return launch_kt<2>(a, s, smem);
    if (kt <= 4) return launch_kt<4>(a, s, smem);
    return launch_kt<8>(a, s, smem);
}

}  // namespace hs
