/*
 * hisparse_oracle.c -- plain, slow, single-threaded CPU oracle of the HiSparse
 * decode-time swap-in resolver.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg load this file's library.  The product
 * path (the CUDA library) never calls it, and this file shares no code,
 * header, table or helper with it.
 *
 * Citations name the two pages the method is taken from:
 *   [Arch]  "HiSparse local KV offload architecture" (vLLM design doc)
 *   [Guide] "HiSparse: Hierarchical Sparse Attention" (SGLang user guide)
 *
 * The method is an exact data-structure algorithm (no floating point): each
 * function below writes out its definition step by step, in the order the
 * pages give, and uses the C library's qsort as the only "library step".
 *
 * Points the pages leave open, and the reading taken here:
 *   - fast path iff seq_len <= device_buffer_size ([Guide] Decode Workflow);
 *     it changes no map, LRU entry or plan;
 *   - misses are handled in ascending token order, victims are the non-hit
 *     slots in ascending (last_used, slot) order, miss i goes to victim i;
 *   - the LRU clock ("tick") of a hot state advances by one on every swap-in
 *     call, starting at 1; prefill stamps 0; every slot selected by a call
 *     (hit or refilled) gets last_used = tick;
 *   - top-k entries are -1 (padding, resolves to -1) or distinct positions in
 *     [0, seq_len); anything else sets a per-request status, leaves that
 *     request's state untouched and writes -1 to all its outputs;
 *   - resident pages come first ([Arch] Resident device pages; Hot lookup and
 *     LRU): with a resident block table, a position whose block is resident
 *     resolves to RESIDENT_FLAG | (block * block_size + position % block_size)
 *     and touches no hot state -- no stamp, no map, no plan entry, no miss;
 *   - the tick is kept per request (a prefill restarts one request's clock);
 *   - paged host pool ([Arch] Ownership: the coordinator maps tokens to
 *     logical host blocks and owns their allocation; the pool budget is
 *     rounded down to whole host blocks): each layer's pool holds
 *     floor(ratio * R * D / hb) blocks of hb token rows; a request's tokens
 *     [b*hb, (b+1)*hb) live in the block its table names at entry b.
 *     Reservation hands out the lowest free block ids, one at a time, in the
 *     order asked.  A miss, a backup or a prefill that needs a row of a block
 *     not reserved sets status NO_HOST_ROW and leaves the request untouched.
 *     A plan then records the host row in the layer's pool (block * hb +
 *     token % hb), the "host slot" a replay reads;
 *   - per-request status word ([Arch] Performance invariants: no device
 *     readback on the decode path, so an error has to stay recorded on the
 *     device until the caller reads it, even when later calls of the same
 *     step -- other layers, later sub-steps, backups -- succeed): besides each
 *     call's own status code, every request keeps a word of error bits; a
 *     call that ends with code c != OK for the request ORs bit c (1 << c) into
 *     it -- swap-ins, prefills and backups alike, on any layer -- and a
 *     successful call leaves it alone.  Only an explicit clear resets it;
 *   - optional protection ([Arch] Resident device pages: speculative
 *     verification steps share the hot state, and a later step may not reuse
 *     a hot row before an earlier step has consumed it): with P > 0, a slot
 *     selected by one of the request's last P calls (last_used >= tick - P,
 *     prefill stamps excluded) is not a victim; a call whose misses outnumber
 *     the other non-hit slots sets status CAPACITY and leaves the request
 *     untouched.  P = 0 (the default) relies on stream order alone.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define HSO_OK 0
#define HSO_BAD_INDEX 1     /* an entry outside {-1} U [0, seq_len) */
#define HSO_DUPLICATE 2     /* a position selected twice            */
#define HSO_BAD_SEQ_LEN 3   /* seq_len outside [0, host capacity]   */
#define HSO_BAD_POSITION 4  /* backup position outside [0, capacity) */
#define HSO_BAD_RESIDENT 5  /* a resident block id outside [-1, 2^30 / block_size) */
#define HSO_NO_HOST_ROW 6   /* a needed host row lies in a block not reserved */
#define HSO_CAPACITY 7      /* protected slots leave too few victims for the misses */

/* A resident hit resolves to this flag OR'd with its row in the resident pool. */
#define HSO_RESIDENT_FLAG 0x40000000

typedef struct hs_oracle {
    int R, L, k, D;
    int64_t B;
    int track_bytes;
    int *anchor;          /* [L]; -1 = the layer owns its hot state          */
    int64_t *cap;         /* [R]; host token capacity per request           */
    int64_t *host_off;    /* [R]; first host token row of each request      */
    int64_t total_cap;
    /* hot state, allocated only for layers with anchor == -1 */
    int32_t **tok2slot;   /* [L] -> [total_cap]  token -> slot or -1        */
    int32_t **slot2tok;   /* [L] -> [R*D]        slot -> token or -1        */
    uint32_t **last_used; /* [L] -> [R*D]        LRU stamp of each slot     */
    uint32_t **tick;      /* [L] -> [R]          stamp of the latest call   */
    /* paged host pool (hb > 0); hb == 0: request r owns host rows
     * [host_off[r], host_off[r] + cap[r]) of each layer */
    int32_t hb;           /* token rows per host block                       */
    int32_t pool_blocks;  /* host blocks per layer                           */
    int32_t **blocks;     /* [R] -> [ceil(cap[r] / hb)] block id or -1       */
    int32_t *nblocks;     /* [R] reserved blocks, always a prefix of the table */
    char *in_use;         /* [pool_blocks]                                    */
    int64_t host_rows;    /* rows of one layer's pool                        */
    int32_t protect_calls; /* P: slots stamped by the last P calls are kept   */
    int32_t *status_word; /* [R] OR of (1 << code) over the errors since clear */
    /* bytes (only with track_bytes) */
    uint8_t **host;       /* [L] -> [host_rows * B]  pinned host pool       */
    uint8_t **dev;        /* [L] -> [R * D * B]      device hot buffer      */
} hs_oracle;

static void hso_free(hs_oracle *o)
{
    if (!o) return;
    for (int l = 0; l < o->L; ++l) {
        if (o->tok2slot) free(o->tok2slot[l]);
        if (o->slot2tok) free(o->slot2tok[l]);
        if (o->last_used) free(o->last_used[l]);
        if (o->tick) free(o->tick[l]);
        if (o->host) free(o->host[l]);
        if (o->dev) free(o->dev[l]);
    }
    if (o->blocks)
        for (int r = 0; r < o->R; ++r) free(o->blocks[r]);
    free(o->tok2slot); free(o->slot2tok); free(o->last_used); free(o->tick);
    free(o->host); free(o->dev);
    free(o->blocks); free(o->nblocks); free(o->in_use);
    free(o->anchor); free(o->cap); free(o->host_off); free(o->status_word);
    free(o);
}

void hso_destroy(hs_oracle *o) { hso_free(o); }

static hs_oracle *create(int R, int L, int64_t B, int k, int D,
                         const int *anchor_of_layer, const int64_t *host_capacity,
                         int32_t hb, int64_t pool_blocks, int track_bytes)
{
    if (R <= 0 || L <= 0 || B <= 0 || k <= 0 || D <= 0 || k > D) return NULL;
    hs_oracle *o = (hs_oracle *)calloc(1, sizeof(hs_oracle));
    if (!o) return NULL;
    o->R = R; o->L = L; o->B = B; o->k = k; o->D = D;
    o->track_bytes = track_bytes;
    o->anchor = (int *)malloc(sizeof(int) * (size_t)L);
    o->cap = (int64_t *)malloc(sizeof(int64_t) * (size_t)R);
    o->host_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)R);
    o->status_word = (int32_t *)calloc((size_t)R, sizeof(int32_t));
    o->tok2slot = (int32_t **)calloc((size_t)L, sizeof(int32_t *));
    o->slot2tok = (int32_t **)calloc((size_t)L, sizeof(int32_t *));
    o->last_used = (uint32_t **)calloc((size_t)L, sizeof(uint32_t *));
    o->tick = (uint32_t **)calloc((size_t)L, sizeof(uint32_t *));
    o->host = (uint8_t **)calloc((size_t)L, sizeof(uint8_t *));
    o->dev = (uint8_t **)calloc((size_t)L, sizeof(uint8_t *));
    if (!o->anchor || !o->cap || !o->host_off || !o->status_word || !o->tok2slot || !o->slot2tok ||
        !o->last_used || !o->tick || !o->host || !o->dev) { hso_free(o); return NULL; }
    int64_t off = 0;
    for (int r = 0; r < R; ++r) {
        if (host_capacity[r] < 0) { hso_free(o); return NULL; }
        o->cap[r] = host_capacity[r];
        o->host_off[r] = off;
        off += host_capacity[r];
    }
    o->total_cap = off;
    o->hb = hb;
    o->host_rows = off;
    if (hb > 0) {
        /* [Arch] Ownership: a pool of whole host blocks, and one block table
         * per request naming the block of each hb tokens. */
        if (pool_blocks < 1 || pool_blocks * hb > INT32_MAX) { hso_free(o); return NULL; }
        o->pool_blocks = (int32_t)pool_blocks;
        o->host_rows = pool_blocks * hb;
        o->blocks = (int32_t **)calloc((size_t)R, sizeof(int32_t *));
        o->nblocks = (int32_t *)calloc((size_t)R, sizeof(int32_t));
        o->in_use = (char *)calloc((size_t)pool_blocks, 1);
        if (!o->blocks || !o->nblocks || !o->in_use) { hso_free(o); return NULL; }
        for (int r = 0; r < R; ++r) {
            int64_t nb = (o->cap[r] + hb - 1) / hb;
            o->blocks[r] = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nb > 0 ? nb : 1));
            if (!o->blocks[r]) { hso_free(o); return NULL; }
            for (int64_t b = 0; b < nb; ++b) o->blocks[r][b] = -1;
        }
    }
    for (int l = 0; l < L; ++l) {
        o->anchor[l] = anchor_of_layer ? anchor_of_layer[l] : -1;
        if (o->anchor[l] >= L || o->anchor[l] == l) { hso_free(o); return NULL; }
        if (o->anchor[l] < 0) {
            /* [Arch] Ownership: the hot-row map and LRU belong to the
             * per-cache runtime; index-sharing followers hold none
             * ([Arch] Performance invariants). */
            o->tok2slot[l] = (int32_t *)malloc(sizeof(int32_t) * (size_t)(o->total_cap > 0 ? o->total_cap : 1));
            o->slot2tok[l] = (int32_t *)malloc(sizeof(int32_t) * (size_t)R * D);
            o->last_used[l] = (uint32_t *)calloc((size_t)R * D, sizeof(uint32_t));
            o->tick[l] = (uint32_t *)calloc((size_t)R, sizeof(uint32_t));
            if (!o->tok2slot[l] || !o->slot2tok[l] || !o->last_used[l] || !o->tick[l]) {
                hso_free(o);
                return NULL;
            }
            for (int64_t i = 0; i < o->total_cap; ++i) o->tok2slot[l][i] = -1;
            for (int64_t i = 0; i < (int64_t)R * D; ++i) o->slot2tok[l][i] = -1;
        }
        if (track_bytes) {
            o->host[l] = (uint8_t *)calloc((size_t)(o->host_rows * B), 1);
            o->dev[l] = (uint8_t *)calloc((size_t)((int64_t)R * D * B), 1);
            if (!o->host[l] || !o->dev[l]) { hso_free(o); return NULL; }
        }
    }
    return o;
}

/* Every request owns host_capacity[r] contiguous token rows of each layer. */
hs_oracle *hso_create(int R, int L, int64_t B, int k, int D,
                      const int *anchor_of_layer, const int64_t *host_capacity,
                      int track_bytes)
{
    return create(R, L, B, k, D, anchor_of_layer, host_capacity, 0, 0, track_bytes);
}

/*
 * Paged host pool: host_capacity[r] is only the longest request r may grow
 * to; the rows themselves come from a pool of floor(ratio * R * D / hb)
 * blocks of hb rows per layer ([Guide] HiSparse Config Parameters: the
 * host_to_device_ratio sizes the logical pool against the device pool;
 * [Arch] the budget is rounded down to whole host blocks).
 */
hs_oracle *hso_create_paged(int R, int L, int64_t B, int k, int D,
                            const int *anchor_of_layer, const int64_t *host_capacity,
                            int ratio, int32_t hb, int track_bytes)
{
    if (ratio < 1 || hb < 1) return NULL;
    int64_t pool_blocks = (int64_t)ratio * R * D / hb;
    return create(R, L, B, k, D, anchor_of_layer, host_capacity, hb, pool_blocks, track_bytes);
}

int32_t hso_pool_blocks(const hs_oracle *o) { return o->pool_blocks; }

/* Protect the slots selected by each request's last `calls` swap-in calls
 * (0 = no protection).  Returns -1 for a negative count. */
int hso_set_protected_calls(hs_oracle *o, int32_t calls)
{
    if (calls < 0) return -1;
    o->protect_calls = calls;
    return 0;
}

int32_t hso_free_blocks(const hs_oracle *o)
{
    int32_t n = 0;
    for (int32_t b = 0; b < o->pool_blocks; ++b) n += !o->in_use[b];
    return n;
}

/* Record a call's status code for request r in its status word: an error
 * (code != OK) sets bit `code`; OK changes nothing. */
static void note_status(hs_oracle *o, int r, int32_t code)
{
    if (code != HSO_OK) o->status_word[r] |= (int32_t)1 << code;
}

/* Copy out the R status words. */
void hso_status_word(const hs_oracle *o, int32_t *words)
{
    memcpy(words, o->status_word, sizeof(int32_t) * (size_t)o->R);
}

/* Reset every request's status word to 0 (no error recorded). */
void hso_status_clear(hs_oracle *o)
{
    memset(o->status_word, 0, sizeof(int32_t) * (size_t)o->R);
}

/* Host row (in the layer's pool) of token t of request r; -1 when the
 * token's block is not reserved. */
static int64_t host_row_of(const hs_oracle *o, int r, int64_t t)
{
    if (o->hb == 0) return o->host_off[r] + t;
    int32_t id = o->blocks[r][t / o->hb];
    if (id < 0) return -1;
    return (int64_t)id * o->hb + t % o->hb;
}

/* The plan's "host slot" of token t: its position within the request's
 * region, or, with a paged pool, its row in the layer's pool. */
static int32_t plan_host_slot(const hs_oracle *o, int r, int32_t t)
{
    return o->hb == 0 ? t : (int32_t)host_row_of(o, r, t);
}

/*
 * Reserve host blocks ([Arch] Ownership: logical host block allocation
 * belongs to the coordinator): for each i in order, request reqs[i] gets
 * blocks until its table covers tokens [0, ntok[i]); each new table entry,
 * in block order, takes the lowest-numbered free block.  All or nothing:
 * returns -1 (bad request or length, nothing changed), -2 (too few free
 * blocks, nothing changed) or 0.
 */
int hso_reserve(hs_oracle *o, int n, const int32_t *reqs, const int64_t *ntok)
{
    if (o->hb == 0 || n < 0) return -1;
    int64_t *want = (int64_t *)calloc((size_t)o->R, sizeof(int64_t));
    for (int r = 0; r < o->R; ++r) want[r] = o->nblocks[r];
    for (int i = 0; i < n; ++i) {
        if (reqs[i] < 0 || reqs[i] >= o->R || ntok[i] < 0 || ntok[i] > o->cap[reqs[i]]) {
            free(want);
            return -1;
        }
        int64_t nb = (ntok[i] + o->hb - 1) / o->hb;
        if (nb > want[reqs[i]]) want[reqs[i]] = nb;
    }
    int64_t need = 0;
    for (int r = 0; r < o->R; ++r) need += want[r] - o->nblocks[r];
    free(want);
    if (need > hso_free_blocks(o)) return -2;
    for (int i = 0; i < n; ++i) {
        int r = reqs[i];
        int64_t nb = (ntok[i] + o->hb - 1) / o->hb;
        while (o->nblocks[r] < nb) {
            int32_t id = 0;
            while (o->in_use[id]) ++id;
            o->in_use[id] = 1;
            o->blocks[r][o->nblocks[r]++] = id;
        }
    }
    return 0;
}

/* Release every host block of each listed request; their table entries
 * become -1.  The request's hot state is left as it is.  Returns -1 (bad
 * request, nothing changed) or 0. */
int hso_release(hs_oracle *o, int n, const int32_t *reqs)
{
    if (o->hb == 0 || n < 0) return -1;
    for (int i = 0; i < n; ++i)
        if (reqs[i] < 0 || reqs[i] >= o->R) return -1;
    for (int i = 0; i < n; ++i) {
        int r = reqs[i];
        for (int32_t b = 0; b < o->nblocks[r]; ++b) {
            o->in_use[o->blocks[r][b]] = 0;
            o->blocks[r][b] = -1;
        }
        o->nblocks[r] = 0;
    }
    return 0;
}

/* Copy out request r's reserved block ids; returns how many there are. */
int32_t hso_block_table(const hs_oracle *o, int r, int32_t *ids)
{
    if (o->hb == 0 || r < 0 || r >= o->R) return -1;
    if (ids) memcpy(ids, o->blocks[r], sizeof(int32_t) * (size_t)o->nblocks[r]);
    return o->nblocks[r];
}

/* Rows [hb][B] of host block `id` of a layer's paged pool. */
uint8_t *hso_block_rows(hs_oracle *o, int layer, int32_t id)
{
    if (!o->track_bytes || o->hb == 0 || id < 0 || id >= o->pool_blocks) return NULL;
    return o->host[layer] + (int64_t)id * o->hb * o->B;
}

/* Host row of token t of request r in a layer's pool (NULL when not
 * tracking bytes, or when the token's host block is not reserved). */
uint8_t *hso_host_row(hs_oracle *o, int layer, int r, int64_t t)
{
    if (!o->track_bytes) return NULL;
    int64_t row = host_row_of(o, r, t);
    return row < 0 ? NULL : o->host[layer] + row * o->B;
}

uint8_t *hso_dev_row(hs_oracle *o, int layer, int r, int64_t s)
{
    if (!o->track_bytes) return NULL;
    return o->dev[layer] + ((int64_t)r * o->D + s) * o->B;
}

/* Copy host row t of request r into device slot s of the same layer. */
static void copy_row(hs_oracle *o, int layer, int r, int32_t t, int32_t s)
{
    if (!o->track_bytes) return;
    memcpy(hso_dev_row(o, layer, r, s), hso_host_row(o, layer, r, t), (size_t)o->B);
}

/*
 * Prefill: the hot buffer of every request starts with the most recent
 * n = min(S, D) tokens, slot i holding token S - n + i, all stamped 0, and
 * the request's tick restarts at 0.  ([Guide] Decode Workflow: for S <= D
 * "all KV is already in the buffer", which fixes slot = token in that
 * case.)  S = -1 leaves request r alone; S outside [0, capacity] sets
 * BAD_SEQ_LEN and a row of the newest n tokens in a host block not reserved
 * sets NO_HOST_ROW, both leaving the request untouched.  status may be NULL.
 */
int hso_prefill(hs_oracle *o, const int32_t *seq_lens, int32_t *status)
{
    for (int r = 0; r < o->R; ++r) {
        int32_t S = seq_lens[r];
        if (S == -1) continue;
        int32_t st = HSO_OK;
        int32_t n = S < o->D ? S : o->D;
        if (S < 0 || S > o->cap[r]) st = HSO_BAD_SEQ_LEN;
        else
            for (int32_t i = 0; i < n; ++i)
                if (host_row_of(o, r, S - n + i) < 0) { st = HSO_NO_HOST_ROW; break; }
        if (status) status[r] = st;
        note_status(o, r, st);
        if (st != HSO_OK) continue;
        for (int l = 0; l < o->L; ++l) {
            if (o->anchor[l] < 0) {
                int32_t *t2s = o->tok2slot[l] + o->host_off[r];
                int32_t *s2t = o->slot2tok[l] + (int64_t)r * o->D;
                uint32_t *lu = o->last_used[l] + (int64_t)r * o->D;
                for (int64_t t = 0; t < o->cap[r]; ++t) t2s[t] = -1;
                for (int32_t s = 0; s < o->D; ++s) { s2t[s] = -1; lu[s] = 0; }
                for (int32_t i = 0; i < n; ++i) {
                    s2t[i] = S - n + i;
                    t2s[S - n + i] = i;
                }
                o->tick[l][r] = 0;
            }
            for (int32_t i = 0; i < n; ++i) copy_row(o, l, r, S - n + i, i);
        }
    }
    return 0;
}

/* Sort keys for the misses (ascending token). */
static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Sort keys for LRU candidates: ascending (last_used, slot). */
typedef struct { uint32_t last_used; int32_t slot; } lru_key;
static int cmp_lru(const void *a, const void *b)
{
    const lru_key *x = (const lru_key *)a, *y = (const lru_key *)b;
    if (x->last_used != y->last_used) return x->last_used < y->last_used ? -1 : 1;
    return (x->slot > y->slot) - (x->slot < y->slot);
}

/* Validate one request's top-k row; returns a status code. */
static int32_t validate(const int32_t *topk, int k, int32_t S)
{
    int32_t *v = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    int n = 0, bad = 0;
    for (int j = 0; j < k; ++j) {
        if (topk[j] == -1) continue;
        if (topk[j] < 0 || topk[j] >= S) { bad = 1; continue; }
        v[n++] = topk[j];
    }
    int32_t st = HSO_OK;
    if (bad) st = HSO_BAD_INDEX;
    else {
        qsort(v, (size_t)n, sizeof(int32_t), cmp_i32);
        for (int i = 1; i < n; ++i)
            if (v[i] == v[i - 1]) { st = HSO_DUPLICATE; break; }
    }
    free(v);
    return st;
}

/* Resident block table of one request ([Arch] Resident device pages: the
 * attention-facing handle's block table).  NULL blocks = no resident tier. */
typedef struct {
    const int32_t *blocks;  /* [max_blocks]: resident block id or -1 */
    int32_t max_blocks;
    int32_t block_size;
} resident_table;

/* Row of token t in the resident pool, or -1 when its block is not resident
 * (a block past the end of the table is not resident). */
static int64_t resident_row(const resident_table *rt, int32_t t)
{
    if (!rt->blocks) return -1;
    int32_t b = t / rt->block_size;
    if (b >= rt->max_blocks || rt->blocks[b] < 0) return -1;
    return (int64_t)rt->blocks[b] * rt->block_size + t % rt->block_size;
}

/* Every looked-up block id must be -1 or name rows below the flag bit. */
static int32_t validate_resident(const resident_table *rt, const int32_t *topk, int k)
{
    if (!rt->blocks) return HSO_OK;
    for (int j = 0; j < k; ++j) {
        if (topk[j] < 0) continue;
        int32_t b = topk[j] / rt->block_size;
        if (b >= rt->max_blocks) continue;
        int32_t id = rt->blocks[b];
        if (id < -1 || (int64_t)id * rt->block_size + rt->block_size > HSO_RESIDENT_FLAG)
            return HSO_BAD_RESIDENT;
    }
    return HSO_OK;
}

/*
 * One request of one swap-in call on hot-state layer `a`
 * ([Guide] Decode Workflow, swap-in step; [Arch] Hot lookup and LRU).
 */
static void swap_in_request(hs_oracle *o, int a, int r, const int32_t *topk,
                            int32_t S, uint32_t tick, const resident_table *rt,
                            int32_t *out, int32_t *plan, int32_t *count, int32_t *status)
{
    const int k = o->k, D = o->D;
    *count = 0;
    if (S < 0 || S > o->cap[r]) *status = HSO_BAD_SEQ_LEN;
    else *status = validate(topk, k, S);
    if (*status == HSO_OK) *status = validate_resident(rt, topk, k);
    if (*status != HSO_OK) {
        for (int j = 0; j < k; ++j) out[j] = -1;
        return;
    }

    /* Resident pages first: a resident position resolves to its resident row
     * and is done. */
    char *done = (char *)calloc((size_t)k, 1);
    for (int j = 0; j < k; ++j) {
        if (topk[j] < 0) continue;
        int64_t row = resident_row(rt, topk[j]);
        if (row >= 0) {
            out[j] = (int32_t)(HSO_RESIDENT_FLAG | row);
            done[j] = 1;
        }
    }

    /* Short sequence: every KV row is already in the buffer, slot = token. */
    if (S <= D) {
        for (int j = 0; j < k; ++j)
            if (!done[j]) out[j] = topk[j];
        free(done);
        return;
    }

    int32_t *t2s = o->tok2slot[a] + o->host_off[r];
    int32_t *s2t = o->slot2tok[a] + (int64_t)r * D;
    uint32_t *lu = o->last_used[a] + (int64_t)r * D;

    /* Hit detection: a token is hot iff the token->slot map holds a slot. */
    char *is_hit_slot = (char *)calloc((size_t)D, 1);
    int32_t *miss = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    int m = 0;
    for (int j = 0; j < k; ++j) {
        int32_t t = topk[j];
        if (t < 0 || done[j]) continue;
        if (t2s[t] >= 0) is_hit_slot[t2s[t]] = 1;
        else miss[m++] = t;
    }
    /* Every miss needs its host row; with a paged pool its block must be
     * reserved, else the request is left untouched. */
    for (int i = 0; i < m; ++i)
        if (host_row_of(o, r, miss[i]) < 0) {
            *status = HSO_NO_HOST_ROW;
            for (int j = 0; j < k; ++j) out[j] = -1;
            free(done); free(is_hit_slot); free(miss);
            return;
        }
    /* Misses are handled in ascending token order. */
    qsort(miss, (size_t)m, sizeof(int32_t), cmp_i32);

    /* LRU victims: the m non-hit slots with the smallest (last_used, slot). */
    lru_key *cand = (lru_key *)malloc(sizeof(lru_key) * (size_t)D);
    int nc = 0;
    for (int32_t s = 0; s < D; ++s)
        if (!is_hit_slot[s]) { cand[nc].last_used = lu[s]; cand[nc].slot = s; ++nc; }
    qsort(cand, (size_t)nc, sizeof(lru_key), cmp_lru);
    /* k <= D and every hit uses one slot, so m <= k - hits <= D - hits = nc. */

    /* Protected slots are not victims.  The candidates are sorted by
     * last_used, so the first m are all unprotected exactly when at least m
     * candidates are. */
    if (o->protect_calls > 0) {
        uint32_t p = (uint32_t)o->protect_calls;
        uint32_t thr = tick > p ? tick - p : 1u;
        int unprotected = 0;
        for (int i = 0; i < nc; ++i) unprotected += cand[i].last_used < thr;
        if (m > unprotected) {
            *status = HSO_CAPACITY;
            for (int j = 0; j < k; ++j) out[j] = -1;
            free(done); free(is_hit_slot); free(miss); free(cand);
            return;
        }
    }

    /* Refill: miss i evicts victim i and is copied from pinned host memory. */
    for (int i = 0; i < m; ++i) {
        int32_t v = cand[i].slot, t = miss[i];
        if (s2t[v] >= 0) t2s[s2t[v]] = -1;
        s2t[v] = t;
        t2s[t] = v;
        plan[2 * i] = plan_host_slot(o, r, t);
        plan[2 * i + 1] = v;
        copy_row(o, a, r, t, v);
    }
    *count = m;

    /* Outputs in input order; every selected slot is stamped with the tick. */
    for (int j = 0; j < k; ++j) {
        int32_t t = topk[j];
        if (done[j]) continue;
        if (t < 0) { out[j] = -1; continue; }
        out[j] = t2s[t];
        lu[t2s[t]] = tick;
    }
    free(done); free(is_hit_slot); free(miss); free(cand);
}

/*
 * hso_swap_in: resolve one call's top-k rows for every request.
 *   topk   [R][k] int32     out    [R][k] int32
 *   plan   [R][k][2] int32  (token, slot) pairs, first count[r] valid
 *   count  [R] int32        status [R] int32
 * Returns -1 if `layer` holds no hot state of its own.
 */
int hso_swap_in_resident(hs_oracle *o, int layer, const int32_t *topk, const int32_t *seq_lens,
                         const int32_t *resident_blocks, int32_t max_blocks, int32_t block_size,
                         int32_t *out, int32_t *plan, int32_t *count, int32_t *status)
{
    if (layer < 0 || layer >= o->L || o->anchor[layer] >= 0) return -1;
    if (resident_blocks && (max_blocks < 1 || block_size < 1)) return -1;
    for (int r = 0; r < o->R; ++r) {
        uint32_t tick = ++o->tick[layer][r];
        resident_table rt;
        rt.blocks = resident_blocks ? resident_blocks + (int64_t)r * max_blocks : NULL;
        rt.max_blocks = max_blocks;
        rt.block_size = block_size;
        swap_in_request(o, layer, r, topk + (int64_t)r * o->k, seq_lens[r], tick, &rt,
                        out + (int64_t)r * o->k, plan + (int64_t)r * o->k * 2,
                        count + r, status + r);
        note_status(o, r, status[r]);
    }
    return 0;
}

int hso_swap_in(hs_oracle *o, int layer, const int32_t *topk, const int32_t *seq_lens,
                int32_t *out, int32_t *plan, int32_t *count, int32_t *status)
{
    return hso_swap_in_resident(o, layer, topk, seq_lens, NULL, 0, 0, out, plan, count, status);
}

/*
 * Replay a recorded miss plan on another layer's KV storage
 * ([Guide] Shared-index prefetch): for every (host slot, device slot) pair,
 * copy that layer's host row into that layer's device slot.  No map or LRU
 * changes.  A pair naming a row or slot out of range is skipped.
 */
int hso_replay(hs_oracle *o, const int32_t *plan, const int32_t *count, int layer)
{
    if (layer < 0 || layer >= o->L) return -1;
    if (!o->track_bytes) return 0;
    for (int r = 0; r < o->R; ++r) {
        int32_t c = count[r] < 0 ? 0 : (count[r] > o->k ? o->k : count[r]);
        for (int i = 0; i < c; ++i) {
            int32_t h = plan[((int64_t)r * o->k + i) * 2];
            int32_t v = plan[((int64_t)r * o->k + i) * 2 + 1];
            int64_t limit = o->hb == 0 ? o->cap[r] : o->host_rows;
            if (h < 0 || h >= limit || v < 0 || v >= o->D) continue;
            int64_t row = o->hb == 0 ? o->host_off[r] + h : h;
            memcpy(hso_dev_row(o, layer, r, v), o->host[layer] + row * o->B, (size_t)o->B);
        }
    }
    return 0;
}

/*
 * Eager backup ([Guide] Decode Workflow): each request's newest KV row goes
 * to host position positions[r] (-1 skips the request); the position is the
 * request's current seq_len.  A position inside the device buffer (< D)
 * belongs to a short sequence, whose buffer holds every token at
 * slot = token, so device slot p is written as well and, for a layer with
 * hot state, the maps pair slot p with token p (their stamps are left as
 * they are).
 */
int hso_backup(hs_oracle *o, int layer, const uint8_t *rows, const int32_t *positions,
               int32_t *status)
{
    if (layer < 0 || layer >= o->L) return -1;
    for (int r = 0; r < o->R; ++r) {
        int32_t p = positions[r];
        status[r] = HSO_OK;
        if (p == -1) continue;
        if (p < 0 || p >= o->cap[r]) {
            status[r] = HSO_BAD_POSITION;
            note_status(o, r, status[r]);
            continue;
        }
        if (host_row_of(o, r, p) < 0) {
            status[r] = HSO_NO_HOST_ROW;
            note_status(o, r, status[r]);
            continue;
        }
        if (o->track_bytes)
            memcpy(hso_host_row(o, layer, r, p), rows + (int64_t)r * o->B, (size_t)o->B);
        if (p < o->D) {
            if (o->track_bytes)
                memcpy(hso_dev_row(o, layer, r, p), rows + (int64_t)r * o->B, (size_t)o->B);
            if (o->anchor[layer] < 0) {
                int32_t *t2s = o->tok2slot[layer] + o->host_off[r];
                int32_t *s2t = o->slot2tok[layer] + (int64_t)r * o->D;
                /* unlink whatever slot p and token p were paired with */
                if (s2t[p] >= 0 && s2t[p] != p) t2s[s2t[p]] = -1;
                if (t2s[p] >= 0 && t2s[p] != p) s2t[t2s[p]] = -1;
                s2t[p] = p;
                t2s[p] = p;
            }
        }
    }
    return 0;
}

/* Copy out a hot-state layer's maps, LRU stamps and per-request ticks. */
int hso_state(hs_oracle *o, int layer, int32_t *slot2tok, uint32_t *last_used,
              int32_t *tok2slot, uint32_t *tick)
{
    if (layer < 0 || layer >= o->L || o->anchor[layer] >= 0) return -1;
    size_t nd = (size_t)o->R * o->D;
    if (slot2tok) memcpy(slot2tok, o->slot2tok[layer], nd * sizeof(int32_t));
    if (last_used) memcpy(last_used, o->last_used[layer], nd * sizeof(uint32_t));
    if (tok2slot) memcpy(tok2slot, o->tok2slot[layer], (size_t)o->total_cap * sizeof(int32_t));
    if (tick) memcpy(tick, o->tick[layer], (size_t)o->R * sizeof(uint32_t));
    return 0;
}

int64_t hso_total_capacity(const hs_oracle *o) { return o->total_cap; }
