/*
 * hisparse.h -- C ABI of the HiSparse decode-time swap-in resolver for
 * NVIDIA GB300 (sm_103a).
 *
 * Each decode step, for every request and every sparse layer that owns an
 * indexer, the resolver takes the top-k token positions chosen by the
 * indexer and turns them into physical row IDs of a small per-request
 * device ("hot") buffer, copying the rows that are not hot from pinned host
 * memory, where the full KV of every request lives.
 *
 * Sources (cited by page title and section):
 *   [Guide] "HiSparse: Hierarchical Sparse Attention" (SGLang user guide):
 *           Decode Workflow; HiSparse Config Parameters; Shared-index
 *           prefetch.
 *   [Arch]  "HiSparse local KV offload architecture" (vLLM design doc):
 *           Ownership; Resident device pages; Hot lookup and LRU;
 *           Performance invariants.
 *
 * Conventions for every entry point:
 *   - Return value: HISPARSE_OK (0) or a negative HISPARSE_ERR_* code.  Host
 *     checks run before any GPU work; on error nothing is enqueued.
 *   - Pointers documented as "device" must be device memory (cudaMalloc or
 *     torch CUDA tensors) of the handle's device; "host" means ordinary host
 *     memory.  "Device-addressable" accepts both device memory and pinned
 *     host memory the device can address (cudaHostAlloc, cudaHostRegister;
 *     with unified addressing, as on GB300, the host pointer itself): the
 *     kernels then read or write it over the host link directly (zero-copy,
 *     NVLink-C2C on GB300).  No entry point keeps a caller pointer after it
 *     returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  The decode-path calls that take a stream (prefill, the
 *     swap-ins, replays, backups, host block reservation and release) are
 *     asynchronous and stream-ordered: they never synchronise and never read
 *     device data back to the host ([Arch] Performance invariants: no device
 *     scalar readback, no CPU/device metadata round trip), and they launch
 *     one kernel ([Arch]: no extra launch) -- two for a swap-in in the split
 *     and auto copy modes, one per 128 table runs for a reservation -- so
 *     they can be captured in a CUDA graph.  hisparse_read_state and
 *     hisparse_write_state synchronise `stream`; they are not for the
 *     decode path.
 *   - Problems in the *data* (a bad top-k index, a duplicate, a bad
 *     position) are recorded per request in a device status word that keeps
 *     them until cleared (see hisparse_status); the affected request's state
 *     is left untouched.
 *   - A handle is not thread-safe; calls on one handle must be ordered by
 *     the caller (one stream, or events between streams).
 *   - A handle belongs to the device current at hisparse_create; calls that
 *     launch work return HISPARSE_ERR_INVALID_ARG unless that device is
 *     current.
 */
#ifndef HISPARSE_H
#define HISPARSE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes (host) ---------------------------------------------- */
#define HISPARSE_OK 0
#define HISPARSE_ERR_INVALID_ARG (-1)  /* null pointer, bad index, bad handle */
#define HISPARSE_ERR_LAYOUT (-2)       /* inconsistent layout                 */
#define HISPARSE_ERR_CAPACITY (-3)     /* host capacity beyond the ratio, or
                                          too few free host blocks           */
#define HISPARSE_ERR_LAYER (-4)        /* layer out of range / has no state   */
#define HISPARSE_ERR_CUDA (-5)         /* a CUDA runtime call failed          */
#define HISPARSE_ERR_NO_MEMORY (-6)    /* pinned or device allocation failed  */
#define HISPARSE_ERR_UNSUPPORTED (-7)  /* beyond this library's size limits   */
#define HISPARSE_ERR_ALIGNMENT (-8)    /* pointer not 16-byte aligned         */

/* ---- per-request status codes (see hisparse_status: the device array
 * holds, per request, a word with bit HISPARSE_STATUS_BIT(code) set for every
 * error code met since the last hisparse_status_clear) ------------------ */
#define HISPARSE_STATUS_OK 0
#define HISPARSE_STATUS_BAD_INDEX 1    /* entry outside {-1} U [0, seq_len)   */
#define HISPARSE_STATUS_DUPLICATE 2    /* a position selected twice           */
#define HISPARSE_STATUS_BAD_SEQ_LEN 3  /* seq_len outside [0, host_capacity]  */
#define HISPARSE_STATUS_BAD_POSITION 4 /* backup position outside [0, cap)    */
#define HISPARSE_STATUS_BAD_RESIDENT 5 /* resident block id < -1 or too large */
#define HISPARSE_STATUS_NO_HOST_ROW 6  /* paged pool: a needed host row lies in
                                          a block the request has not reserved */
#define HISPARSE_STATUS_CAPACITY 7     /* protected slots leave too few victims
                                          for the misses                      */
#define HISPARSE_STATUS_COPY_TIMEOUT 8 /* rows staged by the bulk-copy engine
                                          did not all arrive within the wait
                                          bound (not expected; the request's
                                          new slots may hold stale bytes)      */

#define HISPARSE_STATUS_BIT(code) (1 << (code))

/* A slot ID with this bit set names a row of the caller's resident pool
 * (see hisparse_swap_in_resident); hot slots are below D. */
#define HISPARSE_RESIDENT_FLAG (1 << 30)

/* ---- size limits ------------------------------------------------------- */
#define HISPARSE_MAX_TOP_K 8192
#define HISPARSE_MAX_DEVICE_BUFFER 32768
#define HISPARSE_MAX_HOST_CAPACITY (1 << 20) /* tokens per request          */
#define HISPARSE_MAX_REQUESTS 8192
/* Also: top_k * row_bytes / 16 (a call's 16-byte miss chunks per request)
 * at most 2^31 - 1, else create returns UNSUPPORTED. */
#define HISPARSE_MAX_HOST_BLOCK_TOKENS 65536

/* Copy strategy of hisparse_swap_in (see hisparse_set_copy_mode). */
#define HISPARSE_COPY_FUSED 1  /* the resolving CTA copies its own misses     */
#define HISPARSE_COPY_SPLIT 2  /* a second, wide grid copies all misses       */
#define HISPARSE_COPY_AUTO 3   /* fused; in batches below 8 requests, requests
                                  with > 256 KB of misses leave them to a
                                  second, wide grid                          */

typedef struct hisparse_handle *hisparse_t;

/*
 * Layout of one handle ([Guide] HiSparse Config Parameters; [Arch] Resident
 * device pages, Ownership).
 *   num_requests          R: request rows of the batch (the attention
 *                         metadata's graph-stable request index; row r of
 *                         every per-request array below).
 *   num_layers            L: sparse layers sharing this handle.
 *   row_bytes             B: bytes of one token's KV row in one layer, a
 *                         multiple of 16 (656 for fp8 MLA rows, 1152 for bf16).
 *   top_k                 k: indices per request per call, 1 <= k <= D.
 *   device_buffer_size    D: hot slots per request per layer.
 *   host_to_device_ratio  host token capacity, summed over requests, may not
 *                         exceed ratio * R * D ("host_to_device_ratio").
 *   swap_in_block_size    accepted for compatibility with the guide's
 *                         config ("swap_in_block_size", default 960); a hint
 *                         only, the kernels pick their own block shapes.
 *   anchor_of_layer       host [L] or NULL: -1 = the layer has its own
 *                         indexer and hot state (maps + LRU); a value a >= 0
 *                         marks a "skip" layer that reuses layer a's top-k
 *                         and owns KV storage only ([Guide] Shared-index
 *                         prefetch; [Arch] Performance invariants: index-
 *                         sharing followers drop their private LRU state).
 *                         NULL = every layer owns its state.
 *   host_capacity         host [R]: token rows of host storage per request,
 *                         at least its longest seq_len including growth by
 *                         backups.
 * The arrays are copied by hisparse_create.
 */
typedef struct hisparse_layout {
    int32_t num_requests;
    int32_t num_layers;
    int64_t row_bytes;
    int32_t top_k;
    int32_t device_buffer_size;
    int32_t host_to_device_ratio;
    int32_t swap_in_block_size;
    const int32_t *anchor_of_layer;
    const int64_t *host_capacity;
} hisparse_layout;

/*
 * A miss plan ([Guide] Shared-index prefetch: the anchor's swap-in records
 * which host slot goes to which device buffer slot).  Caller-owned device
 * memory:
 *   rows    device-addressable int32 [R][k][2]: (host slot, device slot) pairs of
 *           request r, ascending by token; only the first counts[r] pairs
 *           are written.  The host slot is the token position within the
 *           request's host region, or, with a paged host pool, the token's
 *           row in the layer's pool (block id * host_block_tokens + token %
 *           host_block_tokens).
 *   counts  device-addressable int32 [R]: misses of request r in the
 *           recording call.
 * Speculative verification ([Arch] Resident device pages: every
 * verification step gets its own replayable plan row) uses one plan per
 * sub-step.
 */
typedef struct hisparse_plan {
    int32_t *rows;
    int32_t *counts;
} hisparse_plan;

/*
 * hisparse_create: validate `layout`, allocate the pinned host pool
 * ([L][sum of host_capacity][B] bytes, mapped into the device address
 * space), the device hot buffers ([L][R][D][B] bytes), and, for every layer
 * that owns state, the token->slot map (int32 per host token), slot->token
 * map and LRU stamps (int32/uint32 [R][D]), the LRU order ([R][D] slots)
 * and one LRU tick per request ([Arch] Ownership: the per-cache runtime owns
 * the host/hot storage, the hot-row map and the LRU).  The handle belongs to
 * the device current at the call.  Pinned memory is zeroed; the hot state
 * starts empty until hisparse_prefill.
 * Errors: INVALID_ARG (null), LAYOUT (a field out of range, top_k > D,
 * row_bytes % 16, an anchor that owns no state), CAPACITY (ratio exceeded),
 * UNSUPPORTED (limits above), NO_MEMORY, CUDA.  *out is NULL on error.
 */
int hisparse_create(const hisparse_layout *layout, hisparse_t *out);

/*
 * hisparse_create_paged: hisparse_create with a paged host pool ([Arch]
 * Ownership: the coordinator maps each request's tokens to logical host
 * blocks and owns their allocation, from a CPU block pool with its own
 * lifecycle; the configured budget is rounded down to whole host blocks.
 * [Guide] HiSparse Config Parameters: host_to_device_ratio sizes the logical
 * pool against the device pool).
 *   host_block_tokens  hb >= 1: token rows per host block.
 * Each layer's pinned pool holds floor(ratio * R * D / hb) blocks of hb
 * rows, [pool_blocks * hb][B] bytes; block ids are the same in every layer.
 * host_capacity[r] is now only the longest request r may grow to (it sizes
 * the token->slot map and the block table; the sum may exceed the pool).
 * Request r's token t lives in row  table[r][t / hb] * hb + t % hb  of the
 * layer's pool; its table starts empty (see hisparse_host_reserve).
 * Errors: as hisparse_create, plus LAYOUT (hb < 1), CAPACITY (the budget is
 * less than one block), UNSUPPORTED (hb > HISPARSE_MAX_HOST_BLOCK_TOKENS,
 * more than 2^31 - 1 rows per layer, or a block table row that does not fit
 * in the resolve kernel's shared memory).
 */
int hisparse_create_paged(const hisparse_layout *layout, int32_t host_block_tokens,
                          hisparse_t *out);

/*
 * hisparse_host_reserve: grow requests' host block tables.  For each i in
 * order, request requests[i] (host int32 [n]) gets blocks until its table
 * covers tokens [0, num_tokens[i]) (host int64 [n], 0 <= num_tokens[i] <=
 * host_capacity); each new entry, in block order, takes the lowest-numbered
 * free block.  All or nothing: too few free blocks for the whole batch
 * returns CAPACITY and changes nothing; a bad request or length returns
 * INVALID_ARG.  The host copy of the tables (hisparse_host_block_table) is
 * updated at once; the device copy that the kernels read is updated by
 * stream-ordered launches on `stream` (one per 128 runs of consecutive
 * ids), so order the calls that use the new blocks after it.  Capturable.
 * The caller writes the rows of new blocks (hisparse_host_block_rows) before
 * the swap-in, backup or prefill that reads them.  CUDA (a launch failed):
 * the host copy is rolled back, but the device copy may hold part of the
 * change; only hisparse_destroy is safe on the handle after that.
 */
int hisparse_host_reserve(hisparse_t h, int32_t n, const int32_t *requests,
                          const int64_t *num_tokens, void *stream);

/*
 * hisparse_host_release: return every host block of each listed request
 * (host int32 [n]) to the pool; their table entries become -1 (device copy:
 * stream-ordered on `stream`).  The requests' hot state is left as it is:
 * restart a request with hisparse_prefill before its next swap-in.  A
 * released block may be handed out by the next reservation: the caller
 * must not write its rows for a new owner until the GPU work that reads the
 * old owner's rows has completed ([Arch] Spill transaction: host pages are
 * republished only after the copy event is observed).  INVALID_ARG for a
 * bad request, nothing released.  CUDA: as for hisparse_host_reserve.
 */
int hisparse_host_release(hisparse_t h, int32_t n, const int32_t *requests, void *stream);

/* Host copy of request `request`'s block table: *count = reserved blocks;
 * the first min(max_ids, count) ids go to `ids` (host).  No GPU work. */
int hisparse_host_block_table(hisparse_t h, int32_t request, int32_t *ids, int32_t max_ids,
                              int32_t *count);

/* Host block size, pool size and free blocks (all 0 without a paged pool);
 * any pointer may be NULL.  No GPU work. */
int hisparse_host_pool_info(hisparse_t h, int32_t *block_tokens, int32_t *pool_blocks,
                            int32_t *free_blocks);

/* Host pointer to the hb rows (B bytes each, contiguous) of pool block
 * `block` of layer `layer`.  Valid until hisparse_destroy. */
int hisparse_host_block_rows(hisparse_t h, int32_t layer, int32_t block, void **host_ptr);

/* Free everything the handle owns.  The caller must have synchronised all
 * streams that used it.  NULL is accepted. */
int hisparse_destroy(hisparse_t h);

/*
 * hisparse_host_rows: host pointer to token row 0 of (layer, request) in the
 * pinned pool; rows are contiguous, B bytes each, host_capacity[request] of
 * them.  The caller writes the request's prefix KV there (the role of the
 * direct-to-host import in [Guide] PD Disaggregation Integration) before
 * hisparse_prefill.  Valid until hisparse_destroy.  A handle with a paged
 * host pool has no per-request region: INVALID_ARG (use
 * hisparse_host_block_rows).
 */
int hisparse_host_rows(hisparse_t h, int32_t layer, int32_t request, void **host_ptr);

/*
 * hisparse_device_buffer: device pointer to layer `layer`'s hot buffer,
 * [R][D][B] bytes, request-major; slot s of request r is the row at byte
 * offset (r * D + s) * B.  This is what sparse attention reads with the
 * slot IDs from hisparse_swap_in ([Arch] Ownership: the attention backend
 * consumes the device cache and physical row IDs).
 */
int hisparse_device_buffer(hisparse_t h, int32_t layer, void **dev_ptr);

/*
 * hisparse_prefill: (re)start requests.  seq_lens: device int32 [R]; an
 * entry of -1 leaves that request untouched, any other value must lie in
 * [0, host_capacity[r]] (else status BAD_SEQ_LEN).  For every layer, the
 * newest n = min(S, D) token rows are copied from the host pool into slots
 * 0..n-1 (slot i <- token S-n+i), and for state-owning layers the maps are
 * set to match, every stamp and the tick are reset to 0 and the LRU order
 * becomes slot order.  A request with S <= D therefore holds every token at
 * slot = token ([Guide] Decode Workflow, fast path).  With a paged host pool
 * the blocks of tokens [S-n, S) must be reserved, else status NO_HOST_ROW
 * and the request is left untouched.  One launch.
 */
int hisparse_prefill(hisparse_t h, const int32_t *seq_lens, void *stream);

/*
 * hisparse_swap_in: resolve one call's top-k for every request on a layer
 * that owns state ([Guide] Decode Workflow, swap-in; [Arch] Hot lookup and
 * LRU), in one launch.
 *   topk_idx      device-addressable int32 [R][k]: token positions; -1 =
 *                 padding.
 *   seq_lens      device-addressable int32 [R]: current length S of each
 *                 request.
 *   out_slot_ids  device-addressable int32 [R][k]: output, the hot slot
 *                 holding each input position (-1 for padding), in input
 *                 order.
 *   out_plan      NULL, or a plan (both pointers non-NULL) to record the
 *                 misses into.
 * Per request: the tick advances by one (a uint32: a request must be
 * restarted with hisparse_prefill, which resets its tick, before 2^32 - 1
 * calls, or stamps stop ordering).  If S <= D the fast path applies:
 * out = topk, nothing else changes.  Otherwise each position is looked up
 * in the token->slot map; hits keep their slot; misses, in ascending token
 * order, take the non-hit slots with the smallest (last_used, slot) in that
 * order, the evicted tokens are unmapped, and each miss's row is copied from
 * the pinned host pool into its slot; every selected slot is stamped with
 * the tick.  A malformed row (see status codes) leaves the request's state
 * untouched and writes -1 to its outputs and 0 to its plan count; so does,
 * with a paged host pool, a miss whose host block the request has not
 * reserved (status NO_HOST_ROW, checked last).
 * Errors: INVALID_ARG, LAYER (skip layer or out of range).
 */
int hisparse_swap_in(hisparse_t h, int32_t layer, const int32_t *topk_idx,
                     const int32_t *seq_lens, int32_t *out_slot_ids,
                     const hisparse_plan *out_plan, void *stream);

/*
 * hisparse_swap_in_resident: hisparse_swap_in with the resident-page tier in
 * front of the hot buffer ([Arch] Resident device pages: one fused resolver
 * checks resident pages first, then hot rows, then pinned host memory, and a
 * resident hit exits before the hot-LRU lookup or a host copy; [Arch]
 * Performance invariants).
 *   resident_blocks  device int32 [R][max_blocks]: for request r, entry b is
 *                    the id of the resident page holding its tokens
 *                    [b * block_size, (b + 1) * block_size) in the caller's
 *                    paged pool, or -1 if that block is not resident.
 *   block_size       tokens per resident page (>= 1); max_blocks >= 1.
 * A position t with id = resident_blocks[r][t / block_size] >= 0 (blocks at
 * or past max_blocks are not resident) resolves to
 *     HISPARSE_RESIDENT_FLAG | (id * block_size + t % block_size)
 * and touches no hot state: no stamp, no map change, no plan entry, not a
 * miss -- also on the fast path.  Every other position is resolved as by
 * hisparse_swap_in.  A looked-up id below -1, or one whose rows reach the
 * flag bit, sets status BAD_RESIDENT (after BAD_INDEX and DUPLICATE) and
 * leaves the request untouched.  Errors: as hisparse_swap_in.
 */
int hisparse_swap_in_resident(hisparse_t h, int32_t layer, const int32_t *topk_idx,
                              const int32_t *seq_lens, const int32_t *resident_blocks,
                              int32_t max_blocks, int32_t block_size, int32_t *out_slot_ids,
                              const hisparse_plan *out_plan, void *stream);

/*
 * hisparse_replay_plan: copy-only replay of a recorded plan onto another
 * layer's storage ([Guide] Shared-index prefetch: skip layers replay the
 * anchor's plan as copy-only kernels pre-issued on a side stream, with a
 * small fixed grid to keep their SM footprint low).  For every request r and
 * i < counts[r]: layer `layer`'s device slot rows[r][i][1] <- its host row
 * rows[r][i][0].  No map or LRU changes.  `num_ctas` sets the grid (0 = 16).
 * Pairs whose host slot or device slot is out of range are skipped.  The caller orders
 * it after the recording swap-in (an event on `stream`).
 */
int hisparse_replay_plan(hisparse_t h, const hisparse_plan *plan, int32_t layer,
                         int32_t num_ctas, void *stream);

/*
 * hisparse_replay_plan_layers: hisparse_replay_plan for several layers in
 * one launch: layers (host int32 [num_layers], 1 <= num_layers <= 16) are
 * copied in order by the same `num_ctas` CTAs.  Pre-issued ahead of the
 * compute it overlaps, the grid is placed once and keeps its SMs until every
 * layer is done; separate launches per layer each have to find free SMs
 * again while the compute occupies them.
 */
int hisparse_replay_plan_layers(hisparse_t h, const hisparse_plan *plan, const int32_t *layers,
                                int32_t num_layers, int32_t num_ctas, void *stream);

/*
 * hisparse_backup: eager backup of each request's newest KV row to host
 * ([Guide] Decode Workflow, eager backup).
 *   rows       device [R][B] bytes, 16-byte aligned.
 *   positions  device int32 [R]: the row's token position, normally the
 *              request's current seq_len; -1 skips the request; outside
 *              [0, host_capacity[r]) sets status BAD_POSITION; with a paged
 *              host pool, a position whose block the request has not
 *              reserved sets status NO_HOST_ROW and writes nothing.
 * Host row p <- rows[r].  If p < D (a short request, whose buffer holds
 * every token at slot = token) device slot p is written too and, on a layer
 * with state, the maps pair slot p with token p.  Stamps are unchanged.
 */
int hisparse_backup(hisparse_t h, int32_t layer, const void *rows,
                    const int32_t *positions, void *stream);

/*
 * hisparse_backup_layers: hisparse_backup for several layers in one launch.
 *   layers     host int32 [num_layers], distinct, 1 <= num_layers <= 16.
 *   rows       device [num_layers][R][B] bytes, 16-byte aligned: the new rows
 *              of layers[i] at rows + i * R * B.
 *   positions  device int32 [R], shared by the layers.
 * The result equals num_layers hisparse_backup calls.  A bad position or a
 * missing host row sets the same status bit from every layer.
 */
int hisparse_backup_layers(hisparse_t h, const int32_t *layers, int32_t num_layers,
                           const void *rows, const int32_t *positions, void *stream);

/*
 * hisparse_status: device pointer to the int32 [R] status array ([Arch]
 * Performance invariants: no device readback on the decode path, so a data
 * error stays on the device until the caller reads it).  Entry r is a word
 * of error bits: every call that meets an error for request r -- a swap-in
 * (any variant, any layer), a prefill or a backup -- sets bit
 * HISPARSE_STATUS_BIT(code) of it, and calls that succeed leave it alone, so
 * an error of layer 0 is still visible after a whole multi-layer step (for
 * example one CUDA graph) has run.  0 = no error since the handle was created
 * or the word was last cleared (hisparse_status_clear).  The entry is
 * written with an atomic OR.  Read it stream-ordered.
 */
int hisparse_status(hisparse_t h, int32_t **dev_status);

/*
 * hisparse_status_clear: reset every request's status word to 0, stream-
 * ordered on `stream` (one memset node; capturable).  Nothing else clears
 * it.  Errors: INVALID_ARG, CUDA.
 */
int hisparse_status_clear(hisparse_t h, void *stream);

/*
 * hisparse_read_state: synchronous copy of a state-owning layer's hot state
 * to host memory, for checking (not on the decode path).  Any pointer may be
 * NULL.  slot2tok int32 [R][D], last_used uint32 [R][D], tok2slot int32
 * [sum of host_capacity] (request-major), lru_order int32 [R][D] (slots from
 * least to most recently used), ticks uint32 [R].  `stream` is synchronised
 * first.
 */
int hisparse_read_state(hisparse_t h, int32_t layer, int32_t *slot2tok,
                        uint32_t *last_used, int32_t *tok2slot, int32_t *lru_order,
                        uint32_t *ticks, void *stream);

/*
 * hisparse_write_state: restore a state-owning layer's hot state from host
 * arrays, e.g. ones saved by hisparse_read_state (checkpoint and resume).
 *   slot2tok   host int32 [R][D]: -1 or a token in [0, host_capacity[r]),
 *              no token twice within a request.
 *   last_used  host uint32 [R][D]; ticks host uint32 [R]; every stamp of
 *              request r is at most ticks[r] (a stamp is the tick of the
 *              call that selected the slot).
 *   rebuild_rows  nonzero: also copy each filled slot's row from the pinned
 *              pool into this layer's hot buffer and those of the layers
 *              anchored on it (with a paged pool, every such token's block
 *              must be reserved).
 * The token->slot map and the LRU order are derived (slots sorted by
 * (last_used, slot)).  `stream` is synchronised first; the call is
 * synchronous and allocates scratch for the rebuild.  INVALID_ARG for a
 * malformed slot->token row or a stamp above its request's tick (nothing is
 * written), LAYER for a skip layer, NO_MEMORY when the rebuild's scratch
 * cannot be allocated (the state is written, the rows are not).  Not for
 * the decode path.
 */
int hisparse_write_state(hisparse_t h, int32_t layer, const int32_t *slot2tok,
                         const uint32_t *last_used, const uint32_t *ticks, int32_t rebuild_rows,
                         void *stream);

/* hisparse_set_copy_mode: how hisparse_swap_in (and _resident) copy the
 * misses; results are identical, only the launch shape differs.
 *   HISPARSE_COPY_FUSED (default)  each request's CTA copies its own rows:
 *                                  one launch per call.
 *   HISPARSE_COPY_SPLIT            the resolve grid records the plan and a
 *                                  full-GPU copy grid, launched behind it
 *                                  with a programmatic dependency, copies.
 *   HISPARSE_COPY_AUTO             with fewer than 8 requests: fused, except
 *                                  that a request whose misses exceed 256 KB
 *                                  is flagged on the device and left to the
 *                                  full-GPU copy grid that follows (two
 *                                  launches per call; no readback) -- one SM
 *                                  alone copies such a volume slowly; with
 *                                  8 or more requests: the same as FUSED. */
int hisparse_set_copy_mode(hisparse_t h, int32_t mode);

/*
 * hisparse_set_stage_rows: how the fused copy (HISPARSE_COPY_FUSED) moves a
 * request's miss rows.  With rows > 0, the first `rows` misses of a request
 * to be found are fetched by the bulk-copy engine (cp.async.bulk) into the
 * resolving CTA's shared memory as soon as their lookups return, before their
 * victim slots are known, and stored to their slots once the victims are
 * chosen; the others are loaded by the CTA's threads into registers right
 * after classification.  0 (the default) stages none; -1 stages as many as
 * the shared memory left over by the resolver holds (~259 rows of 656 B at
 * k 2048, D 6144); a larger count is clamped to that.  Results are
 * identical whatever the count; only the route of the bytes differs.
 * Measured on GB300 with an earlier kernel of this design, one CTA per
 * request (kernel-only step time): decode_40k 45.6 us with 0,
 * 46.5 us with 16, 48.9 us with 64 and 57.6 us with all; mixed_len 1.009 ms
 * with 0, 1.003 ms with all; spec_verify 3.576 ms with 0, 3.591 ms with
 * all.  Read at each swap-in launch.  INVALID_ARG for rows < -1.
 */
int hisparse_set_stage_rows(hisparse_t h, int32_t rows);

/*
 * hisparse_set_copy_ctas: how many CTAs serve each request of a fused-copy
 * swap-in (HISPARSE_COPY_FUSED with no staged rows; other modes ignore it).
 * A new handle starts with the largest count, up to 4, at which the GPU
 * holds the clusters of all its requests at once (see
 * hisparse_get_copy_ctas).  ctas = 1: the one CTA that resolves the request
 * also loads its miss rows from pinned host memory.  ctas = 2..4: each
 * request gets a thread-block cluster of that many CTAs on different SMs;
 * rank 0 resolves (hit lookup, victims, every state write) and issues no
 * host loads, and the ctas - 1 others copy.  With the resident-token bitmap
 * (the lookup the handle picks when it fits in shared memory) each copier
 * stages the same rows as rank 0, finds the same misses in the same order
 * and starts loading their rows from the host at once; otherwise rank 0
 * writes the list of miss rows into the copiers' shared memory at
 * classification.  Once the victims are chosen rank 0 writes the victim
 * slots there, and the copiers store the rows.  Each SM then keeps one kind
 * of traffic in flight: on one SM, host loads in flight hold up that SM's
 * stores to the hot state.  Results are identical whatever the count.
 * Measured on GB300 (decode_40k, 32 requests, kernel-only): 41.5-41.7 us per
 * call with 4, 42.5 us with 3, 43.3 us with 2.  INVALID_ARG unless
 * 1 <= ctas <= 4; UNSUPPORTED if the GPU cannot hold even one such cluster of
 * resolve CTAs.  Read at each swap-in launch.
 */
int hisparse_set_copy_ctas(hisparse_t h, int32_t ctas);

/*
 * hisparse_get_copy_ctas: the CTAs per request that fused-copy swap-ins use
 * now (see hisparse_set_copy_ctas).  A new handle starts with the largest
 * count, up to 4, at which the GPU holds the clusters of all its requests at
 * once (1 if not even 2 fit so).  INVALID_ARG for a null pointer.
 */
int hisparse_get_copy_ctas(hisparse_t h, int32_t *ctas);

/*
 * hisparse_set_programmatic_launch: on = 1 launches the swap-in's resolve grid
 * and the backups with a programmatic dependency on the previous kernel of
 * the stream (programmatic dependent launch): when that kernel signals its
 * dependents early (griddepcontrol.launch_dependents, or
 * cudaTriggerProgrammaticLaunchCompletion), this library's grid is placed on
 * free SMs before it ends and waits for it on the device (griddepcontrol.wait).
 * A grid waits before it reads anything, except a swap-in whose previous
 * kernel on the stream, as far as this handle knows, is one of its own
 * launches on that stream that wrote nothing of the swap-in's layer (its hot
 * state, device rows or host rows; a prefill, a host block table edit or a
 * state write counts as writing every layer): that swap-in reads its
 * inputs, the layer's state and its first host rows at once, and waits only
 * before its first write to global memory.  Either way a grid signals its
 * own dependents only after its wait, so a swap-in never starts while an
 * older call that is not the one just before it still runs.  The caller's
 * part: a kernel of its own that it places directly before a library call on
 * the stream, if launched so that it may signal early, must have written the
 * call's inputs (top-k rows, lengths, backup rows and positions, resident
 * tables) and be done with the library's device rows before it signals.
 * on = 0 (the default) launches plainly.  Results are identical either way.
 * Measured on GB300, kernel-only step times against on = 0 (two
 * interleaved runs each): mixed_len (4 resolves on 4 layers and a backup,
 * back to back) 1.0117 against 1.0190 ms; spec_verify (3 sub-steps on one
 * layer and a backup) 3.591 against 3.594 ms; decode_40k steps (each resolve
 * behind an L2-flush kernel that signals nothing) +0.45 us.  Read at each launch (a
 * captured graph keeps the launch as captured).  INVALID_ARG unless on is 0
 * or 1.
 */
int hisparse_set_programmatic_launch(hisparse_t h, int32_t on);

/*
 * hisparse_set_protected_calls: keep the hot rows of a request's last
 * `calls` swap-in calls out of the victims ([Arch] Resident device pages:
 * speculative verification steps share the request's hot state, and a later
 * step may not reuse a hot row before an earlier step has consumed it).  A
 * slot whose stamp is at least max(1, tick - calls) -- selected by one of
 * those calls; prefill stamps never count -- is not evicted.  A call whose
 * misses outnumber the remaining non-hit slots sets status CAPACITY (checked
 * last) and leaves the request untouched, with -1 outputs and a 0 plan count.
 * 0 (the default) turns protection off: sub-steps resolved and consumed in
 * stream order need none.  Read at each swap-in launch (a captured graph
 * keeps the value it was captured with).  INVALID_ARG for calls < 0.
 */
int hisparse_set_protected_calls(hisparse_t h, int32_t calls);

/*
 * hisparse_swap_in_noalloc: hisparse_swap_in in the split copy shape (a
 * resolve grid, then a full-GPU copy grid), for callers that must not cause
 * any device allocation -- for example a serving process whose device memory
 * is owned up front by one pool, or a call site that runs where allocation
 * is forbidden.  The miss plan handed from the resolve grid to the copy grid
 * lives in a fixed array of HISPARSE_NOALLOC_SCRATCH_BYTES inside the library
 * (one per GPU, held until the process exits) instead of memory from
 * cudaMalloc; this call allocates nothing, and no plan is returned to the
 * caller.  Arguments, results and status codes are those of hisparse_swap_in
 * with out_plan = NULL.
 *   - The array must hold (2 * top_k + 1) * num_requests int32 values; a
 *     larger handle gets HISPARSE_ERR_UNSUPPORTED and nothing is launched.
 *   - hisparse_create looks the array's device address up
 *     (cudaGetSymbolAddress, with the handle's device current), which also
 *     loads the part of the library that holds it, and keeps the address in
 *     the handle; this call itself loads, looks up and allocates nothing.
 *     After a device reset the handle is invalid anyway: create a new one.
 *   - Every call on a device shares the one array and leaves the last call's
 *     contents in it.  Each call writes everything it later reads, so nothing
 *     needs clearing, but calls whose work overlaps on the GPU (two streams,
 *     two handles) race on it: order them.
 * The pages this library follows have no counterpart to this call.
 */
#define HISPARSE_NOALLOC_SCRATCH_BYTES (8 << 20)
int hisparse_swap_in_noalloc(hisparse_t h, int32_t layer, const int32_t *topk_idx,
                             const int32_t *seq_lens, int32_t *out_slot_ids, void *stream);

/*
 * hisparse_check_guards: for testing.  A handle created while the
 * environment variable HISPARSE_DEBUG_GUARDS is "1" allocates every device
 * array it owns with a 4 KB band of a known byte on each side.  This call
 * synchronises the device and writes to *overwritten how many bands no
 * longer hold that byte (0 = no write left its array).  UNSUPPORTED for a
 * handle created without the bands.
 */
int hisparse_check_guards(hisparse_t h, int32_t *overwritten);

/* Text of a return code (static storage). */
const char *hisparse_error_string(int code);

/* ABI version: 100 * major + minor. */
int hisparse_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HISPARSE_H */
