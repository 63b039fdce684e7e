// copy.cu -- plan replay, eager backup and prefill kernels.
//
// Sources: [Guide] "HiSparse: Hierarchical Sparse Attention" -- Shared-index
// prefetch (skip layers replay the anchor's miss plan with a copy-only kernel
// on a small fixed grid) and Decode Workflow (eager backup of the newest
// token's KV to host; short sequences keep every token in the buffer).
#include "hs_common.cuh"

namespace hs {
namespace {

constexpr int REPLAY_NT = 512;
constexpr int REPLAY_ROWS = 8;     // plan rows a warp takes at a time
constexpr int REPLAY_UNROLL = 11;  // host chunks in flight per lane (8 rows of 656 B: one pass)

// Copy every (host slot -> device slot) pair of a plan, host row -> device
// slot, for each of a list of layers.  A host slot is a token position in the
// request's region, or, with a paged host pool, a row of the layer's pool.
// Work units are plan rows, numbered layer by layer over the concatenation of
// all requests' plan rows.  Each CTA first builds the prefix sum of plan
// counts in shared memory (clamped to [0, k]); then each warp takes
// REPLAY_ROWS rows at a time.  One launch covers all the skip layers of an
// anchor, so its few CTAs are placed once, ahead of the compute they overlap,
// and stay until every layer is copied.  Pairs whose host slot or device slot
// is out of range are skipped.
__global__ void __launch_bounds__(REPLAY_NT) replay_kernel(ReplayLaunch a)
{
    extern __shared__ __align__(16) uint32_t rows_before[];  // [R + 1]
    __shared__ uint32_t warp_tot[32];
    if (a.programmatic) {
        // wait for the resolve grid that writes the plan (griddepcontrol.wait)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    const int R = a.g.R, k = a.g.k, D = a.g.D;
    const int tid = threadIdx.x;

    // exclusive prefix of counts over requests (R <= 8192: 16 per thread)
    const int per = (R + REPLAY_NT - 1) / REPLAY_NT;
    const int r0 = min(tid * per, R), r1 = min(r0 + per, R);
    auto rows_of = [&](int r) -> uint32_t {
        if (a.only_if && a.only_if[r] == 0) return 0u;
        return (uint32_t)min(max(a.plan_counts[r], 0), k);
    };
    uint32_t local = 0;
    for (int r = r0; r < r1; ++r) local += rows_of(r);
    uint32_t total_rows;
    uint32_t run = block_exclusive_scan<REPLAY_NT>(local, warp_tot, total_rows);
    for (int r = r0; r < r1; ++r) {
        rows_before[r] = run;
        run += rows_of(r);
    }
    if (tid == 0) rows_before[R] = total_rows;
    __syncthreads();

    // Each warp takes REPLAY_ROWS plan rows at a time: lanes 0..REPLAY_ROWS-1
    // resolve one row each (its request by binary search over the prefix,
    // its plan pair, the two row addresses) into shared memory, then the
    // warp streams the chunks of all its rows with REPLAY_UNROLL host loads in
    // flight per lane.  Plan pairs are read once per row, not per chunk.
    __shared__ const uint8_t *row_src[REPLAY_NT / 32][REPLAY_ROWS];
    __shared__ uint8_t *row_dst[REPLAY_NT / 32][REPLAY_ROWS];
    const int CH = a.g.chunks;
    const int64_t B = a.g.B;
    const int lane = tid & 31, warp = tid >> 5;
    const uint64_t per_layer = total_rows;
    const uint64_t units = per_layer * (uint64_t)a.num_layers;
    const uint64_t wstride = (uint64_t)gridDim.x * (REPLAY_NT / 32);
    const int elems = REPLAY_ROWS * CH;
    for (uint64_t u0 = (uint64_t)blockIdx.x * (REPLAY_NT / 32) + warp; u0 < units;
         u0 += wstride * REPLAY_ROWS) {
        if (lane < REPLAY_ROWS) {
            const uint8_t *src = nullptr;
            uint8_t *dst = nullptr;
            const uint64_t u = u0 + (uint64_t)lane * wstride;
            if (u < units) {
                const int layer = (int)(u / per_layer);
                const uint32_t row = (uint32_t)(u - (uint64_t)layer * per_layer);
                int lo = 0, hi = R;  // last r with rows_before[r] <= row
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (rows_before[mid] <= row) lo = mid; else hi = mid;
                }
                const int r = lo;
                const int32_t *pr = a.plan_rows + ((int64_t)r * k + (row - rows_before[r])) * 2;
                const int32_t hslot = pr[0], slot = pr[1];
                const int64_t limit = a.g.hb ? a.g.pool_rows : a.g.host_cap[r];
                if (hslot >= 0 && (int64_t)hslot < limit && slot >= 0 && slot < D) {
                    const int64_t hrow = a.g.hb ? (int64_t)hslot : a.g.host_off[r] + hslot;
                    src = a.store[layer].host + hrow * B;
                    dst = a.store[layer].dev + ((int64_t)r * D + slot) * B;
                }
            }
            row_src[warp][lane] = src;
            row_dst[warp][lane] = dst;
        }
        __syncwarp();
        for (int e = lane; e < elems; e += 32 * REPLAY_UNROLL) {
            uint4 v[REPLAY_UNROLL];
            uint8_t *dst[REPLAY_UNROLL];
#pragma unroll
            for (int q = 0; q < REPLAY_UNROLL; ++q) {
                dst[q] = nullptr;
                const int ee = e + q * 32;
                if (ee >= elems) continue;
                const int j = ee / CH, c = ee - j * CH;
                const uint8_t *sp = row_src[warp][j];
                if (!sp) continue;
                v[q] = ld_host_v4(sp + c * 16);
                dst[q] = row_dst[warp][j] + c * 16;
            }
#pragma unroll
            for (int q = 0; q < REPLAY_UNROLL; ++q)
                if (dst[q]) st_v4(dst[q], v[q]);
        }
        __syncwarp();
    }
}

// Backup: one thread per 16-byte chunk of each request's new row; the thread
// writes that chunk in every listed layer.  Latency is all there is to this
// launch (R x B bytes a layer), so the chunk loads of the first layers go out
// together with the position lookup, and each group of BACKUP_GROUP layers
// has all its loads in flight before any of its stores.  The layers share the
// positions, so a bad position or a missing host row sets one status bit for
// all of them.
constexpr int BACKUP_GROUP = 4;

__global__ void __launch_bounds__(256) backup_kernel(BackupLaunch a)
{
    // with a programmatic launch (see launch_backup) this grid may start
    // before the previous kernel of the stream ends: wait for it before
    // reading anything (without one the wait returns at once)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int CH = a.g.chunks;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (int64_t)a.g.R * CH) return;
    const int r = (int)(e / CH), c = (int)(e - (int64_t)r * CH);
    const int64_t B = a.g.B;
    const int D = a.g.D;
    const int L = a.num_layers;
    uint4 v[BACKUP_GROUP];
#pragma unroll
    for (int u = 0; u < BACKUP_GROUP; ++u)
        if (u < L) v[u] = ld_dev_v4(a.layer[u].rows + (int64_t)r * B + c * 16);
    const int32_t p = a.positions[r];
    if (p == -1) return;
    const int64_t cap = a.g.host_cap[r];
    if (p < 0 || (int64_t)p >= cap) {
        if (c == 0) record_status(a.status, r, kStatusBadPosition);
        return;
    }
    // with a paged host pool the position's block must be reserved
    const int64_t row = host_row_of(a.g, r, p);
    if (row < 0) {
        if (c == 0) record_status(a.status, r, kStatusNoHostRow);
        return;
    }
    for (int l0 = 0; l0 < L; l0 += BACKUP_GROUP) {
        if (l0 > 0) {
#pragma unroll
            for (int u = 0; u < BACKUP_GROUP; ++u)
                if (l0 + u < L) v[u] = ld_dev_v4(a.layer[l0 + u].rows + (int64_t)r * B + c * 16);
        }
#pragma unroll
        for (int u = 0; u < BACKUP_GROUP; ++u) {
            if (l0 + u >= L) continue;
            const BackupLayer &Ly = a.layer[l0 + u];
            st_v4(Ly.host + row * B + c * 16, v[u]);
            if (p < D) st_v4(Ly.dev + ((int64_t)r * D + p) * B + c * 16, v[u]);
        }
    }
    // a short request (p < D) holds every token at slot = token: pair slot
    // p with token p in the maps of the layers that own state
    if (p < D && c == 0) {
        for (int li = 0; li < L; ++li) {
            const BackupLayer &Ly = a.layer[li];
            if (!Ly.st.tok2slot) continue;
            int32_t *t2s = Ly.st.tok2slot + a.g.host_off[r];
            int32_t *s2t = Ly.st.slot2tok + (int64_t)r * D;
            const int32_t old_tok = s2t[p], old_slot = t2s[p];
            if (old_tok >= 0 && old_tok != p) t2s[old_tok] = -1;
            if (old_slot >= 0 && old_slot != p) s2t[old_slot] = -1;
            s2t[p] = p;
            t2s[p] = p;
            if (Ly.st.resbits) {   // token old_tok leaves the buffer, token p is in it
                uint32_t *rb = Ly.st.resbits + (int64_t)r * Ly.st.res_words;
                if (old_tok >= 0 && old_tok != p) atomicAnd(&rb[old_tok >> 5], ~(1u << (old_tok & 31)));
                atomicOr(&rb[p >> 5], 1u << (p & 31));
            }
        }
    }
}

// Prefill: grid (blocks per request, R, L).  For request r, n = min(S, D):
// slot i <- token S-n+i.  Every map entry is written with its final value,
// so blocks never race.  With a paged host pool every block of tokens
// [S-n, S) must be reserved; each CTA checks that itself, so either all of a
// request's CTAs write or none does.
__global__ void __launch_bounds__(256) prefill_kernel(const int32_t *seq_lens,
                                                      const LayerDescDev *layers, Geometry g,
                                                      int32_t *status)
{
    const int r = blockIdx.y, l = blockIdx.z;
    const int32_t S = seq_lens[r];
    if (S == -1) return;
    const int64_t cap = g.host_cap[r];
    if (S < 0 || (int64_t)S > cap) {
        if (l == 0 && blockIdx.x == 0 && threadIdx.x == 0) record_status(status, r, kStatusBadSeqLen);
        return;
    }
    const int D = g.D;
    const int32_t n = S < D ? S : D;
    if (g.hb) {
        bool missing = false;
        if (n > 0) {
            const int32_t b0 = (S - n) / g.hb, b1 = (S - 1) / g.hb;
            for (int32_t b = b0 + (int32_t)threadIdx.x; b <= b1; b += blockDim.x)
                missing |= g.host_tbl[(int64_t)r * g.tbl_stride + b] < 0;
        }
        if (__syncthreads_or(missing)) {
            if (l == 0 && blockIdx.x == 0 && threadIdx.x == 0) record_status(status, r, kStatusNoHostRow);
            return;
        }
    }
    const LayerDescDev L = layers[l];
    const int64_t off = g.host_off[r];
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t gs = (int64_t)gridDim.x * blockDim.x;
    if (L.st.tok2slot) {
        int32_t *t2s = L.st.tok2slot + off;
        for (int64_t t = gt; t < cap; t += gs)
            t2s[t] = (t >= S - n && t < S) ? (int32_t)(t - (S - n)) : -1;
        int32_t *s2t = L.st.slot2tok + (int64_t)r * D;
        uint32_t *lu = L.st.last_used + (int64_t)r * D;
        uint16_t *lru = L.st.lru + (int64_t)r * D;
        for (int64_t s = gt; s < D; s += gs) {
            s2t[s] = s < n ? (int32_t)(S - n + s) : -1;
            lu[s] = 0u;
            lru[s] = (uint16_t)s;
        }
        if (gt == 0) L.st.tick[r] = 0u;
        if (L.st.resbits) {   // tokens [S - n, S) have slots
            uint32_t *rb = L.st.resbits + (int64_t)r * L.st.res_words;
            const int64_t lo = S - n, hi = S;
            for (int64_t w = gt; w < L.st.res_words; w += gs) {
                const int64_t t0 = w * 32;
                const int64_t a = lo > t0 ? lo - t0 : 0, b = hi < t0 + 32 ? hi - t0 : 32;
                uint32_t word = 0u;
                if (b > a) word = (b - a == 32) ? ~0u : (((1u << (b - a)) - 1u) << a);
                rb[w] = word;
            }
        }
    }
    const int CH = g.chunks;
    const int64_t B = g.B;
    const int64_t total = (int64_t)n * CH;
    for (int64_t e = gt; e < total; e += gs) {
        const int64_t i = e / CH;
        const int c = (int)(e - i * CH);
        const uint4 v = ld_host_v4(L.host + host_row_of(g, r, S - n + i) * B + c * 16);
        st_v4(L.dev + ((int64_t)r * D + i) * B + c * 16, v);
    }
}

// Host block table edits: one CTA per run.
__global__ void __launch_bounds__(128) table_runs_kernel(int32_t *table, TableRuns runs)
{
    const int i = blockIdx.x;
    if (i >= runs.n) return;
    const int32_t first = runs.first[i], value = runs.value[i], len = runs.len[i];
    for (int32_t j = threadIdx.x; j < len; j += blockDim.x)
        table[first + j] = value < 0 ? -1 : value + j;
}

}  // namespace

size_t replay_smem_bytes(int R) { return (size_t)(R + 1) * 4; }

cudaError_t copy_prepare()
{
    // Load these kernels now.  With lazy module loading (the CUDA default) a
    // kernel is loaded at its first launch, on the launching thread, and the
    // stream waits meanwhile: the first backup of a process measured 0.77 s
    // instead of microseconds.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, replay_kernel);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&attr, backup_kernel);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&attr, prefill_kernel);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&attr, table_runs_kernel);
    return e;
}

cudaError_t launch_table_runs(int32_t *table, const TableRuns &runs, cudaStream_t s)
{
    if (runs.n <= 0) return cudaSuccess;
    table_runs_kernel<<<runs.n, 128, 0, s>>>(table, runs);
    return cudaGetLastError();
}

cudaError_t launch_replay(const ReplayLaunch &a, cudaStream_t s)
{
    const size_t smem = replay_smem_bytes(a.g.R);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_ctas);
    cfg.blockDim = dim3(REPLAY_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (a.programmatic) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, replay_kernel, a);
}

cudaError_t launch_backup(const BackupLaunch &a, cudaStream_t s)
{
    const int64_t n = (int64_t)a.g.R * a.g.chunks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (a.programmatic) {
        // a backup usually follows the step's last swap-in: placed under its
        // tail, it waits for it on the device (griddepcontrol.wait)
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, backup_kernel, a);
}

cudaError_t launch_prefill(const int32_t *seq_lens, const LayerDescDev *layers, int num_layers,
                           const Geometry &g, int32_t *status, cudaStream_t s)
{
    dim3 grid(8, g.R, num_layers);
    prefill_kernel<<<grid, 256, 0, s>>>(seq_lens, layers, g, status);
    return cudaGetLastError();
}

}  // namespace hs
