/*
 * ice.h - C ABI of the GB300-native IceCache decode-time library (libice.so).
 *
 * IceCache ("IceCache", arXiv 2604.10539) keeps the KV cache of each attention
 * head in pages that are the leaves of a DCI-tree built over the keys in a
 * transformed key space (Figure 2 step 1; Figure 3 maps tree nodes to physical
 * pages). Generated tokens are inserted without a rebuild (the abstract
 * describes the structure as updatable in place). At each decode step a prioritised tree search
 * finds the query's top keys, the pages holding them are selected (Figure 2
 * steps 2-3), and attention runs over every token of those pages.
 *
 * This library runs all of it on one GPU with its own CUDA kernels. The four
 * calls of the method are ice_build, ice_insert, ice_select and
 * ice_sparse_attn; they work on a grid of independent UNITS, one unit being
 * one (sequence b, layer l, KV head h), unit index u = (b * n_layers + l) *
 * n_kv_heads + h. Query head g of unit u is q_head = h * G + g with
 * G = n_q_heads / n_kv_heads (grouped-query attention).
 *
 * Conventions for every call:
 *  - Pointers named as device pointers must point to device memory of the
 *    current CUDA device; the caller owns them. Host pointers are named so.
 *  - The calls that run a decode step (ice_insert, ice_select,
 *    ice_select_attn, ice_select_attn_reuse, ice_decode_step,
 *    ice_select_heads, ice_sparse_attn) also take page-locked host memory
 *    (cudaHostAlloc, cudaMallocHost, cudaHostRegister) for any of their
 *    device buffers: the kernels read and write it in place over the CPU-GPU
 *    link, with no staging copy. Each buffer pointer is checked before
 *    anything is launched, and memory the GPU cannot address (pageable host
 *    memory, another GPU's memory) gives ICE_ERR_INVALID_ARG. While `stream`
 *    is being captured into a CUDA graph the pointers are not checked (the
 *    eager calls before a capture check the same buffers). ice_build and
 *    ice_key_codes_noalloc take device memory only.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls enqueue work on it and return without waiting, except where stated.
 *  - Return value: ICE_OK (0) or a negative ICE_ERR_* code. Argument errors
 *    are found on the host before anything is launched. Errors that only the
 *    GPU can see (a page id out of range, an exhausted capacity) are recorded
 *    in a per-index device status word that ice_get_error() returns. Kernels
 *    never trap; the only waits between blocks are the barriers of one
 *    thread-block cluster, whose blocks run together.
 *  - One handle is used by one host thread at a time: the calls keep host-side
 *    state (the token count, the stream of the last insert). Separate handles
 *    are independent. Calls on one stream run in order; calls on different
 *    streams that touch one handle must be ordered by the caller (events).
 *  - Element type of keys, values, queries and outputs is the index's dtype
 *    (ICE_BF16 or ICE_F32); rows of d elements are contiguous.
 */
#ifndef ICE_H_
#define ICE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define ICE_OK 0
#define ICE_ERR_INVALID_ARG (-1) /* bad argument; nothing was launched          */
#define ICE_ERR_CAPACITY (-2)    /* token / page / leaf capacity exhausted        */
#define ICE_ERR_CUDA (-3)        /* a CUDA runtime call failed                    */
#define ICE_ERR_TIMEOUT (-4)     /* a bounded device wait ran out (device status) */
#define ICE_ERR_BOUNDS (-5)      /* a page id or count given to a kernel is bad   */
#define ICE_ERR_UNSUPPORTED (-6) /* valid request the library does not implement */

/* ---- element types ----------------------------------------------------- */
#define ICE_F32 0
#define ICE_BF16 1

typedef struct ice_index ice_index; /* opaque; owns the page pool and the index */

/* Shape and method parameters of an index. */
typedef struct ice_params {
    int32_t d;           /* head dimension; the kernels support 128                  */
    int32_t n_kv_heads;  /* KV heads per layer (>= 1)                                */
    int32_t n_q_heads;   /* query heads per layer, a multiple of n_kv_heads; G <= 8  */
    int32_t n_layers;    /* layers (>= 1)                                            */
    int32_t batch;       /* sequences (>= 1)                                         */
    int32_t page_size;   /* P: tokens per page = leaf capacity, 1..64                */
    int32_t n_proj;      /* m: projections per composite index; must be 8            */
    int32_t n_composite; /* L: composite indices, 1..2                               */
    int32_t n_cand;      /* candidates taken per composite; 0 = the token budget     */
    int32_t dtype;       /* ICE_BF16 or ICE_F32                                      */
    int64_t max_tokens;  /* token capacity per unit (>= n_tokens of ice_build)       */
    uint64_t seed;       /* seed of the random projection directions (splitmix64)    */
    int32_t kv_location; /* ICE_KV_DEVICE: the page pool in device memory (HBM);     */
                         /* ICE_KV_HOST: in pinned host memory mapped into the       */
                         /* GPU's address space, read by the kernels over the        */
                         /* CPU-GPU link (the paper's offloaded KV tier)             */
    int32_t dir_kind;    /* projection directions: ICE_DIR_RADEMACHER (+-1/16 per   */
                         /* component, one splitmix64 draw each) or ICE_DIR_GAUSSIAN */
                         /* (z/16, z from the Box-Muller transform of two draws)     */
} ice_params;

/* Distribution of the random projection directions (ice_params.dir_kind). */
enum { ICE_DIR_RADEMACHER = 0, ICE_DIR_GAUSSIAN = 1 };

/* Page pool placement (ice_params.kv_location). With ICE_KV_HOST the index
 * (leaf tables, slot lists, token locations) stays in device memory and only
 * the K/V rows live on the host; ice_select_attn then runs as ice_select
 * followed by ice_sparse_attn (both read the pool with plain or cp.async
 * loads). */
enum { ICE_KV_DEVICE = 0, ICE_KV_HOST = 1 };

/*
 * ice_build - index the prefill keys and values (Figure 2 step 1, Figure 3).
 *
 * keys, values: device, [batch][n_layers][n_kv_heads][n_tokens][d], dtype.
 * For each unit: squared key norms set the scale c = 2^e (smallest power of
 * two with c^2 >= max ||k||^2, frozen for later inserts); each key is mapped to
 * k~ = [k / c, sqrt(1 - ||k||^2 / c^2)] and projected on the L*m random +-1/16
 * directions; the 8-bit codes are Morton-interleaved into a 64-bit key, the
 * token index breaks ties, and the keys are sorted. A binary trie over these
 * 96-bit keys splits every node that holds more than P tokens; its non-empty
 * leaves are the leaves of each composite, and the leaves of composite 0 are
 * the physical pages (ids 0.. left to right), into which K and V are copied.
 * The library keeps its own copy of K and V; the inputs may be reused as soon
 * as the call returns.
 *
 * This call waits for its stream once (to size the page pool from the leaf
 * counts) and returns with the build complete. On success *out receives a new
 * handle that the caller releases with ice_destroy.
 */
int ice_build(const ice_params* params, const void* keys, const void* values, int64_t n_tokens,
              void* stream, ice_index** out);

/*
 * ice_insert - add one generated token to every unit without a rebuild (the
 * abstract's in-place update of the index).
 *
 * k, v: device, [batch][n_layers][n_kv_heads][d], dtype. The token gets index
 * n (the unit's current token count). Its key is transformed with the frozen
 * scale, then in each composite it is appended to the leaf whose prefix it
 * carries; a leaf that would exceed P splits in two (the left part keeps the
 * page id, the right part takes the next free id); a key that falls where no
 * leaf exists opens a new leaf with the next free id. The result equals a
 * fresh build of all tokens with the same scale.
 * Returns ICE_ERR_CAPACITY if the units already hold max_tokens tokens.
 */
int ice_insert(ice_index* ix, const void* k, const void* v, void* stream);

/*
 * ice_select - the prioritised query: pages holding the query's top keys
 * (Figure 2 steps 2-3).
 *
 * q: device, [batch][n_layers][n_q_heads][d], dtype.
 * token_budget: T, a multiple of page_size with T >= page_size; n_sel = T / P
 *   pages are selected per unit.
 * page_ids: device int32 [units][n_sel]; receives the selected page ids in
 *   selection order, -1 after the last one.
 * n_pages: device int32 [units]; receives the number of pages selected (< n_sel
 *   only when the candidates span fewer pages).
 * stats: device int32 [units][4] or NULL. When given: [0] leaf records scanned
 *   (all composites), [1] distinct candidate keys rescored, [2] tokens in the
 *   selected pages, [3] candidate tokens taken before de-duplication.
 *
 * Per unit: the group's query heads are summed in fp32 (q_sel), normalised and
 * projected to codes; in each composite the leaves are taken in increasing
 * (L-infinity code distance to the leaf's cell, position) order until n_cand
 * tokens are collected; the union of those tokens is rescored exactly with a
 * fixed-order fp32 dot q_sel . k, ranked by (score desc, token asc), and the
 * pages of the ranked tokens are taken in first-occurrence order.
 */
int ice_select(ice_index* ix, const void* q, int32_t token_budget, int32_t* page_ids,
               int32_t* n_pages, int32_t* stats, void* stream);

/*
 * ice_select_attn - ice_select followed by ice_sparse_attn over the selected
 * pages, in one kernel launch per call (each unit's pages are attended as soon
 * as they are known, without a round trip of the page list through memory).
 * Arguments and results are those of the two calls: page_ids, n_pages and
 * stats as in ice_select, out as in ice_sparse_attn with page_stride =
 * token_budget / page_size. The pages chosen and the attention computed are
 * the same as with the two separate calls.
 */
int ice_select_attn(ice_index* ix, const void* q, int32_t token_budget, int32_t* page_ids,
                    int32_t* n_pages, int32_t* stats, void* out, void* stream);

/*
 * ice_select_attn_reuse - ice_select_attn that keeps a unit's pages across
 * calls ("IceCache" paper, the IceCache(r) variant, whose mechanism the paper
 * leaves open). Reading: a unit reuses the pages of its last selection for up
 * to r further calls while its query codes (the 8-bit codes of the group
 * query on every projection direction, which the selection computes first)
 * are exactly those of the call that selected the pages. Any changed code, r
 * reuses in a row, a unit without a selection yet or a changed token_budget
 * selects again. Inserted tokens are seen: the attention reads each page's
 * current tokens.
 *
 * page_ids, n_pages: device, as in ice_select; they carry the selection from
 * call to call, so the same buffers must be passed every time (in: the pages
 * in use; out: the pages used by this call).
 * r: >= 0 (0 selects on every call, the same as ice_select_attn).
 * reselected: optional device int32 [units]; 1 where this call selected.
 * out: as in ice_select_attn.
 * The per-unit codes and reuse counts live in the index (allocated on the
 * first call, ICE_ERR_CAPACITY if that fails). stats are not written.
 */
int ice_select_attn_reuse(ice_index* ix, const void* q, int32_t token_budget, int32_t r,
                          int32_t* page_ids, int32_t* n_pages, int32_t* reselected, void* out,
                          void* stream);

/*
 * ice_select_heads - per-query-head selection with a union over the group (a
 * variant of Figure 2 step 2): every query head g of unit u selects pages with
 * its own query as q_sel (the same search and ranking as ice_select, G = 1),
 * and the unit's pages are the union of its heads' lists, head 0's pages first
 * in their order, then each later head's pages not yet listed.
 *
 * head_page_ids: device int32 [units][G][n_sel]; head_n_pages: [units][G].
 * page_ids: device int32 [units][G * n_sel] (the union, -1 padded); n_pages:
 * [units]. Attend with ice_sparse_attn(..., page_stride = G * n_sel, ...).
 * G * n_sel must be <= 512 (ICE_ERR_UNSUPPORTED otherwise).
 */
int ice_select_heads(ice_index* ix, const void* q, int32_t token_budget, int32_t* head_page_ids,
                     int32_t* head_n_pages, int32_t* page_ids, int32_t* n_pages, void* stream);

/*
 * ice_decode_step - one decode step of every unit: ice_insert of the new
 * token's k, v, then ice_select_attn for the query q (the new token is a
 * candidate like any other). For a launch of many units, one kernel launch on
 * `stream` (each block inserts its unit's token, then selects and attends);
 * when the selection runs on a cluster of blocks per unit (few units, see
 * ice_set_cluster_size), with a host-resident pool, or when the split's staging
 * does not fit, the insert and the selection are separate launches. No host
 * synchronisation and no allocation, so a sequence of steps can be captured
 * once in a CUDA graph and replayed: the insert takes the token index from a
 * per-unit count kept on the device, which every replay advances (a unit at
 * max_tokens reports ICE_ERR_CAPACITY through ice_get_error and is left
 * unchanged). Arguments as in ice_insert and ice_select_attn.
 */
int ice_decode_step(ice_index* ix, const void* k, const void* v, const void* q,
                    int32_t token_budget, int32_t* page_ids, int32_t* n_pages, void* out,
                    void* stream);

/* ice_reuse_reset - forget every unit's kept selection (the next
 * ice_select_attn_reuse selects everywhere). Asynchronous on `stream`. */
int ice_reuse_reset(ice_index* ix, void* stream);

/*
 * ice_sparse_attn - attention of each query head over every token of the
 * selected pages (Figure 2 step 3).
 *
 * q: device, [batch][n_layers][n_q_heads][d], dtype.
 * page_ids: device int32 [units][page_stride]; n_pages: device int32 [units],
 *   0 <= n_pages[u] <= page_stride (as written by ice_select).
 * out: device, [batch][n_layers][n_q_heads][d], dtype. For query head g of
 *   unit u: out = sum_t softmax_t(q . k_t / sqrt(d)) v_t over the tokens t of
 *   the pages (fp32 accumulation). A unit with no pages gets zeros.
 * Page ids outside the unit's allocated range are skipped and reported as
 * ICE_ERR_BOUNDS through ice_get_error().
 */
int ice_sparse_attn(ice_index* ix, const void* q, const int32_t* page_ids, const int32_t* n_pages,
                    int32_t page_stride, void* out, void* stream);

/*
 * ice_get_error - waits for `stream`, then returns and clears the index's
 * device status word (ICE_OK if no kernel reported an error).
 */
int ice_get_error(ice_index* ix, void* stream);

/* ice_destroy - waits for the device, then frees everything the handle owns. */
void ice_destroy(ice_index* ix);

/* ice_status_string - static text for a status code. */
const char* ice_status_string(int status);

/* Host-side facts about an index. */
typedef struct ice_info {
    int64_t n_units;       /* batch * n_layers * n_kv_heads                     */
    int64_t n_tokens;      /* tokens per unit (build + inserts)                 */
    int64_t max_tokens;    /* token capacity per unit                           */
    int64_t list_capacity; /* leaf / page capacity per unit and composite       */
    int64_t pool_bytes;    /* device bytes held by the handle                   */
    int32_t group;         /* G                                                 */
    int32_t n_composite;   /* L                                                 */
    int32_t page_size;     /* P                                                 */
    int32_t dtype;         /* ICE_BF16 / ICE_F32                                */
    int64_t host_bytes;    /* pinned host bytes held by the handle (host pool)  */
    int32_t kv_location;   /* ICE_KV_DEVICE / ICE_KV_HOST                       */
    int32_t reserved;
} ice_info;

int ice_get_info(const ice_index* ix, ice_info* info);

/*
 * ice_set_cluster_size - how many thread blocks share one unit in the selection
 * of ice_select and ice_select_attn (a tuning knob; results do not depend on it).
 * The selection of a unit is a chain of dependent phases (IceCache page, Figure 2
 * steps 2-3); with few units per launch (one layer of a decode step) one block
 * per unit leaves most SMs idle. A thread-block cluster of k blocks splits the
 * leaf scan, the rescoring and the attended pages of a unit, and merges the
 * priority histograms, the page keys and the softmax partials over distributed
 * shared memory.
 *   k = 0: automatic (8, 4 or 2 blocks per unit for launches of up to 19, 38 or
 *          76 units; one block per unit above that, and a cluster whenever one
 *          block cannot hold the unit's tables);
 *   k = 1: one block per unit;
 *   k = 2, 4, 8, 16: that many blocks per unit (k >= n_composite).
 * The cluster path takes budget/page_size <= 32 pages; ice_decode_step uses it
 * after a separate insert launch; ice_select_attn_reuse and ice_select_heads
 * always use one block per unit. A call
 * whose forced k cannot be launched (tables too large, or clusters of that
 * size not resident on this GPU) returns ICE_ERR_UNSUPPORTED or ICE_ERR_CUDA.
 * Returns ICE_ERR_INVALID_ARG for any other k.
 */
int ice_set_cluster_size(ice_index* ix, int32_t k);

/*
 * Debug views (tests only). ice_debug_dump copies the index of one unit to
 * host memory and waits for the copy. Layout of host_buf, little endian:
 *   int64 header[16]: L, P, list_capacity C, n_tokens n, e, n_leaf[0..3],
 *                     next_id[0..3], reserved
 *   per composite l (repeated L times):
 *     leaf key   [C] x {uint64 morton_prefix, uint32 token_prefix, uint32 t}
 *     leaf rec   [C] x {uint8 lo[8], uint32 list id << 8 | token count, uint32 t}
 *                (lo = lower corner of the leaf's code cell; the upper corner
 *                 is lo_j | (2^(8 - b_j) - 1), b_j the known bits of code j)
 *     list count [C] x int32 (tokens in list/page id)
 *     slot token [C][P] x int32 (token of each slot of list/page id)
 *     slot key   [C][P] x uint64 (Morton key of that token)
 *   token location [max_tokens] x int32 (page id * P + slot, composite 0)
 *   only when L = 2:
 *     slot location [C][P] x int32 (token location of the token in each
 *                   composite-1 slot; meaningful where the slot holds a token)
 *     token slot    [max_tokens] x int32 (composite-1 list id * P + slot of
 *                   each token, -1 for none)
 * Only the first n_leaf[l] leaf records and the first next_id[l] lists are
 * meaningful. Returns the byte size required when host_buf is NULL or cap is
 * too small (as a positive number), ICE_OK after a copy, or an error.
 */
int64_t ice_debug_dump(ice_index* ix, int32_t unit, void* host_buf, int64_t cap, void* stream);

/* Copies page `page_id` of unit `unit` (P rows of K and of V, dtype) to host
 * buffers of P*d elements each and waits for the copy. */
int ice_debug_page(ice_index* ix, int32_t unit, int32_t page_id, void* host_k, void* host_v,
                   void* stream);

/*
 * ice_debug_set_flags - test hooks (0 = normal operation).
 * ICE_DEBUG_STALL_ATTN: the fused call's page staging expects 16 bytes more
 * than its copies deliver, so its bounded wait (200 ms of wall time) runs out
 * twice; the call then skips the attention of that round, writes zeros and
 * reports ICE_ERR_TIMEOUT through ice_get_error(). Nothing is left in flight
 * and the context stays usable. Used to test the timeout path.
 */
enum { ICE_DEBUG_STALL_ATTN = 1 };
int ice_debug_set_flags(ice_index* ix, int32_t flags);


/*
 * ice_key_codes_noalloc - the key transform of ice_build (squared norms, the
 * frozen scale exponent per unit, the 8-bit codes of every key on the L x 8
 * random directions, their Morton interleave) without allocating any memory.
 * The paper has no counterpart of this call; it exists for callers that
 * cannot allocate device memory while they run (a process whose memory is all
 * handed to its own pool allocator, or a latency-critical loop where a
 * cudaMalloc, which can synchronise the device, is not acceptable).
 *
 * params: as for ice_build (d = 128, n_proj = 8, n_composite, dtype, seed, and
 *   batch x n_layers x n_kv_heads units; the other fields are ignored).
 * keys: device, [units][n_tokens][d], dtype; 16-byte aligned.
 * morton_out: device uint64 [n_composite][units][n_tokens]; receives the
 *   Morton key of each token (the same value ice_build indexes).
 * e_out: device int32 [units]; receives the scale exponent e (c = 2^e).
 *
 * Scratch lives in fixed device arrays inside the library: at most
 * units * n_tokens <= 1,048,576 tokens and units <= 4096 per call; larger
 * requests return ICE_ERR_CAPACITY before anything runs. The arrays (about
 * 4.1 MB) stay on every GPU that loads the library until the process exits.
 * All calls share them: calls that overlap on the GPU (two streams) race; calls
 * on one stream are ordered. The first call on each device looks up the arrays'
 * device addresses (cudaGetSymbolAddress); make that first call before any
 * stream capture. The call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine) and returns without waiting.
 */
int ice_key_codes_noalloc(const ice_params* params, const void* keys, int64_t n_tokens,
                          uint64_t* morton_out, int32_t* e_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ICE_H_ */
