/*
 * pkv — paged KV-cache decode attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libpkv.so.  Plain pointers and sizes only.
 *
 * Sources the operations follow (page title, section):
 *   [SERVE-FLOW]   "Incremental Serving", section "Request flow".
 *   [SERVE-PAGED]  "Incremental Serving", section "Paged KV-cache layout".
 *   [SERVE-CABI]   "Incremental Serving", section "Stable C and Python sessions".
 *   [SERVE-SCOPE]  "Incremental Serving", section "Current scope".
 *   [CACHED-MIX]   "38 · Cached generation", section "Prepare every block, then
 *                  commit every cache together" (function incremental_mixture,
 *                  and the prepared-ticket commit).
 *   [CACHED-BIND]  "38 · Cached generation", section "Bind one decoder to its
 *                  model-wide cache, then advance every block coherently".
 *   [CACHED-CELLS] "38 · Cached generation", section "Count attention-score
 *                  cells, not total runtime".
 *   [ROLLOUT-KV]   "Rollout Serving, Caching, and Batching", KV-cache memory formula
 *                  (and its note that grouped-query or multi-query attention has
 *                  fewer KV heads than query heads).
 *
 * Conventions (all entry points):
 *   - Every call returns a pkv_status.  PKV_OK is 0.  A call that returns an
 *     error has changed no state ([CACHED-BIND]: rejected operations leave the
 *     committed state unchanged).  pkv_last_error() then describes the failure
 *     (thread-local, valid until the next call on the same thread).
 *   - Handles are opaque.  A pool owns its device K/V storage; requests point at
 *     their pool, and a pool cannot be destroyed while requests are alive.
 *   - Not thread-safe: calls that touch the same pool must be serialised by the
 *     caller ([SERVE-CABI]: the raw C ABI requires external synchronisation).
 *   - Device work is asynchronous on the caller's stream (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream).  No entry point
 *     synchronises except pkv_check_device_status.  The caller's current CUDA
 *     device must be the device the pool was created on.
 *   - The q, k, v and out tensors of every attention call must each start on a
 *     multiple of min(16, bytes of one head row) (head_dim x element size);
 *     others are rejected with PKV_ERR_INVALID_ARGUMENT.  Workspaces start on a
 *     multiple of 16 bytes.
 *   - Device-side faults are never raised by trapping: a kernel that meets an
 *     out-of-range length or page id, or a wait that runs out, sets a bit in the
 *     pool's device error word, skips the bad access and returns;
 *     pkv_check_device_status reports it.
 *
 * Layout ([SERVE-PAGED]): per layer, key pages and value pages are each
 *   [physical_page][head][page_offset][head_width]  (row-major, storage dtype)
 * and one physical page id addresses the matching K and V page in every layer.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_pool pkv_pool;
typedef struct pkv_request pkv_request;

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARGUMENT = 1,   /* bad pointer, size, layer, shape */
    PKV_ERR_OUT_OF_PAGES = 2,       /* the pool has no free page left */
    PKV_ERR_CAPACITY_EXCEEDED = 3,  /* request at its maximum context ([SERVE-CABI]) */
    PKV_ERR_BAD_STATE = 4,          /* call out of order (token pending / not pending, ...) */
    PKV_ERR_OUT_OF_MEMORY = 5,      /* host or device allocation failed */
    PKV_ERR_CUDA = 6,               /* a CUDA runtime call failed */
    PKV_ERR_DEVICE_CHECK = 7,       /* a kernel flagged bad input (see pkv_check_device_status) */
    PKV_ERR_NO_STORAGE = 8,         /* bookkeeping-only pool has no device storage */
    PKV_ERR_UNSUPPORTED = 9         /* geometry the kernels do not implement */
} pkv_status;

typedef enum pkv_dtype {
    PKV_F32 = 0,    /* 4-byte IEEE float */
    PKV_BF16 = 1    /* 2-byte bfloat16 (upper half of an IEEE float) */
} pkv_dtype;

/* pkv_pool_create flags */
#define PKV_POOL_HOST_ONLY 1u   /* bookkeeping only: free list, tables, transactions; no device
                                   storage, so append/attend entry points return PKV_ERR_NO_STORAGE */

#define PKV_POOL_CUDA_CORES 2u  /* use the CUDA-core kernel even where the tensor-core kernel
                                   applies (bf16 or fp32 storage, head_dim 64 or 128, 2 or
                                   more query heads per KV head) */

/* bits of the device error word */
#define PKV_DEVERR_SEQ_LEN 1u   /* a seq_len < 1, > max_seq_len, or needing > max_pages pages */
#define PKV_DEVERR_PAGE_ID 2u   /* a page-table entry outside [0, pages) */
#define PKV_DEVERR_TIMEOUT 4u   /* a bounded wait for an async copy ran out */
#define PKV_DEVERR_SHARED 8u    /* a request's page table differs from request 0's within the
                                   declared shared prefix (pkv_paged_decode_attention_shared) */

/* Work counters of one request ([CACHED-BIND] work counters; [CACHED-CELLS]).
 * They advance only when a token commits; reset (release) zeroes them. */
typedef struct pkv_counters {
    int64_t committed_tokens;   /* tokens made visible by pkv_commit_token */
    int64_t cache_appends;      /* layers x committed tokens */
    int64_t score_cells;        /* sum over committed tokens of layers x query_heads x
                                   min(t, window) (t without a window) */
} pkv_counters;

/* ---------------------------------------------------------------- pool -- */

/*
 * Pool geometry for pkv_pool_create_ex.  pkv_pool_options_init fills the
 * defaults: 1 layer, pages 0, 1 KV head, query_heads 0, head_dim 128,
 * page_size 16, PKV_BF16, max_context 4096, seed 0, flags 0.
 *   kv_heads:    heads stored in every page (the K/V layout's head axis).
 *   query_heads: heads of the query and of the output; 0 means kv_heads.  A
 *                multiple of kv_heads: query head q reads KV head
 *                q / (query_heads / kv_heads) (grouped-query attention,
 *                [ROLLOUT-KV]; kv_heads == 1 is multi-query attention).
 *   window:      sliding window ([ROLLOUT-KV]'s fixed window of W positions):
 *                > 0 makes every query attend only to the last `window`
 *                positions (itself included); 0 (default) attends to the whole
 *                prefix.  Pages before the window stay leased.
 * The other fields are those of pkv_pool_create.
 */
typedef struct pkv_pool_options {
    int layers;
    int64_t pages;
    int kv_heads;
    int query_heads;
    int head_dim;
    int page_size;
    int dtype;
    int64_t max_context;
    uint64_t seed;
    unsigned flags;
    int64_t window;
} pkv_pool_options;

int pkv_pool_options_init(pkv_pool_options* options);

/*
 * Create a paged pool ([SERVE-PAGED]).
 *   layers, heads, head_dim: geometry of every request served from the pool.
 *   pages:       physical pages per layer; 0 = enough pages for one
 *                maximum-length context, ceil(max_context / page_size)
 *                ([SERVE-PAGED]: a block count of 0 sizes one full context).
 *   page_size:   tokens per page; the sources' default is 16.  Kernels require a
 *                multiple of 16 (a contiguous one-page-per-request layout uses
 *                page_size = max_context rounded up to 16).
 *   dtype:       storage dtype of K and V (PKV_F32 or PKV_BF16).
 *   max_context: largest retained length of one request (>= 1).
 *   seed:        free-list order: a FIFO queue initialised to a Fisher-Yates
 *                shuffle of 0..pages-1 driven by SplitMix64(seed), swap index
 *                next() mod (i + 1) for i = pages-1 down to 1.
 *   flags:       0, or PKV_POOL_HOST_ONLY and/or PKV_POOL_CUDA_CORES.
 * Supported by the kernels: head_dim a power of two, 2 <= head_dim <= 128 for
 * PKV_F32 and <= 256 for PKV_BF16 (else PKV_ERR_UNSUPPORTED, unless HOST_ONLY).
 * Equivalent to pkv_pool_create_ex with kv_heads = query_heads = heads.
 * Device storage is 2 * layers * pages * page_size * heads * head_dim * element
 * size bytes ([ROLLOUT-KV]), zero-filled; the pool also allocates a 4-byte
 * device error word.  A device pool also makes sure that the library's fixed
 * scratch array of pkv_paged_decode_attention_static (PKV_STATIC_SCRATCH_BYTES)
 * is loaded on the current device, once per context.  On success *out receives
 * the handle.
 */
int pkv_pool_create(int layers, int64_t pages, int heads, int head_dim, int page_size, int dtype,
                    int64_t max_context, uint64_t seed, unsigned flags, pkv_pool** out);

/* Create a pool from options (see pkv_pool_options).  Grouped-query and
 * multi-query pools (query_heads = G x kv_heads) are implemented for G in
 * {2, 4, 8, 16, 32, 64, 128} at head_dim 64 and 128 (else PKV_ERR_UNSUPPORTED,
 * unless HOST_ONLY).  Decode on the bf16 tensor-core kernel runs a group above 16
 * as G / 16 lanes of 16 query heads per KV head, the other kernels a group above 8
 * as G / 8 lanes of 8, each lane reading the KV head's pages (the repeats mostly
 * from L2). */
int pkv_pool_create_ex(const pkv_pool_options* options, pkv_pool** out);

/* KV heads stored per page and heads of the query (either pointer may be NULL). */
int pkv_pool_heads(const pkv_pool* pool, int* kv_heads, int* query_heads);

/* *tensor_cores = 1 if the pool's decode attention runs the tensor-core kernel
 * (head_dim 64 or 128, 2 or more query heads per KV head, not
 * PKV_POOL_CUDA_CORES; bf16 products with fp32 accumulation for bf16 pools, and
 * for fp32 pools tf32 products of each operand's two tf32 parts, which keep fp32
 * accuracy), 0 for the CUDA-core kernel. */
int pkv_pool_kernel(const pkv_pool* pool, int* tensor_cores);

/* Free the pool and its device storage.  PKV_ERR_BAD_STATE while any request
 * created from it is alive.  NULL is accepted. */
int pkv_pool_destroy(pkv_pool* pool);

/* Device base addresses of one layer's key and value pages (layout above).
 * Owned by the pool; valid until pkv_pool_destroy.  NO_STORAGE for host-only pools. */
int pkv_pool_kv_ptr(const pkv_pool* pool, int layer, void** k_pages, void** v_pages);

/* Bytes of device K/V storage (2 * layers * pages * page_size * heads * head_dim * es). */
int pkv_pool_bytes(const pkv_pool* pool, uint64_t* bytes);

/* Physical pages per layer, and how many are currently free. */
int pkv_pool_pages(const pkv_pool* pool, int64_t* pages, int64_t* free_pages);

/* Copy the free list, front first, into host_out[0 .. cap); *n receives its
 * length (the copy is truncated to cap). */
int pkv_pool_free_list(const pkv_pool* pool, int32_t* host_out, int64_t cap, int64_t* n);

/* ------------------------------------------------------------- requests -- */

/* New empty request (length 0, no pages) drawing pages from `pool`. */
int pkv_request_create(pkv_pool* pool, pkv_request** out);

/* Abort a pending token if any, drop the request's reference to every page it
 * holds (pages nobody else references go back to the pool), free the request
 * ([SERVE-PAGED]: pages go back when a request is destroyed).  NULL ok. */
int pkv_request_destroy(pkv_request* req);

/*
 * Prefix sharing ([SERVE-SCOPE]: page sharing between matching prompts and
 * copy-on-write prefix management, listed there as future work).  Create a
 * request that shares every page of `parent` at the parent's visible length:
 * nothing is copied, each shared page gains a reference.  Either request may
 * then decode on its own: a token that would be written into a page another
 * request still references first moves the writer to a private copy
 * (pkv_begin_token leases it, each layer's pkv_append_and_attend copies that
 * layer's page before its kernel).  Full shared pages are never written.
 * BAD_STATE if the parent has a token pending.
 */
int pkv_request_fork(const pkv_request* parent, pkv_request** child);

/* Number of requests referencing physical page `page` (0: free). */
int pkv_pool_page_refs(const pkv_pool* pool, int32_t page, int* refs);

/*
 * Lease n more pages now, appended to the request's logical page table in the
 * order they leave the free list's front.  Pages are otherwise leased lazily
 * by pkv_begin_token ([SERVE-PAGED]).  All or nothing: OUT_OF_PAGES if fewer
 * than n are free, CAPACITY_EXCEEDED if the table would pass
 * ceil(max_context / page_size), BAD_STATE while a token is pending.
 */
int pkv_lease_pages(pkv_request* req, int64_t n);

/* Reset: drop the request's reference to every page in logical order (a page
 * nobody else references goes to the back of the free list), set the visible
 * length to 0 and zero the counters ([SERVE-PAGED]; [CACHED-BIND] reset).
 * BAD_STATE while a token is pending. */
int pkv_release_pages(pkv_request* req);

/* Visible (committed) length. */
int pkv_request_length(const pkv_request* req, int64_t* visible_len);

/* Copy the logical page table (physical ids) into host_out[0 .. cap); *n_pages
 * receives its length. */
int pkv_request_page_table(const pkv_request* req, int32_t* host_out, int64_t cap,
                           int64_t* n_pages);

/* Counters of the request. */
int pkv_request_counters(const pkv_request* req, pkv_counters* out);

/* ---------------------------------------------------------- transaction -- */

/*
 * Reserve the next logical position ([SERVE-FLOW] step 1).  *position receives
 * it (= the visible length).  If that position starts a page the request does
 * not hold yet, one page is leased from the free list's front; if it falls in a
 * page another request also references (after pkv_request_fork), a private
 * page is leased from the front to replace it (copy-on-write); the request
 * keeps its reference to the shared page until pkv_commit_token drops it (to
 * the free list's back if it was the last one), so an abort can restore it.
 * BAD_STATE if a token is already pending; CAPACITY_EXCEEDED at max_context;
 * OUT_OF_PAGES if a page is needed and none is free.
 */
int pkv_begin_token(pkv_request* req, int64_t* position);

/*
 * One layer's step for the pending token ([SERVE-FLOW] step 2): store the
 * new key and value rows at the pending position of `layer`'s pools, then
 * attend the newest query over all t = position + 1 retained keys of that
 * layer, the new one included ([CACHED-MIX]: scores q.k / sqrt(head_dim),
 * stable softmax, weighted sum of values).
 *   q   [query_heads][head_dim] fp32, device
 *   k,v [kv_heads][head_dim] storage dtype, device
 *   out [query_heads][head_dim] fp32, device (the [1,H,1,d_h] attention context)
 *   stream: cudaStream_t
 * Call once per layer per pending token; BAD_STATE if none is pending or the
 * layer already ran for it.  The new row is written into the page at once but
 * is visible to later tokens only after pkv_commit_token.
 * Enqueues at most one 4-byte host-to-device copy of a newly leased page-table
 * entry and two kernels on `stream`; returns without waiting.
 */
int pkv_append_and_attend(pkv_request* req, int layer, const float* q, const void* k,
                          const void* v, float* out, void* stream);

/*
 * Open a chunk of n >= 1 positions at the visible length, the batched prefill
 * of one request taken through the same transaction ([SERVE-PAGED]: a batched
 * prefill writing the same paged cache; [SERVE-FLOW] steps 1-4 for n positions
 * at once).  *position receives the first.  Pages for all n positions are
 * leased now from the free list's front: first a private copy for every page
 * another request also references among those the chunk writes (ascending
 * logical index; copy-on-write), then the pages the request does not hold yet.
 * All or nothing: BAD_STATE if a token or chunk is pending; CAPACITY_EXCEEDED
 * if length + n passes max_context; OUT_OF_PAGES if too few pages are free.
 * Then pkv_prefill_chunk once per layer and pkv_commit_token or
 * pkv_abort_token.
 */
int pkv_begin_chunk(pkv_request* req, int64_t n, int64_t* position);

/*
 * One layer's step for the pending chunk: store its n key/value rows at
 * positions position .. position+n-1 of `layer`'s pools and attend each of its
 * queries causally, as pkv_paged_prefill does for one request (chunk token i
 * over positions 0 .. position+i, the window applied).
 *   q   [n][query_heads][head_dim] storage dtype, device
 *   k,v [n][kv_heads][head_dim] storage dtype, device
 *   out [n][query_heads][head_dim] fp32, device
 * Call once per layer per pending chunk; BAD_STATE if no chunk is pending (a
 * pending single token takes pkv_append_and_attend) or the layer already ran.
 * The rows are written at once but are visible to later tokens only after
 * pkv_commit_token.  Enqueues a page-table upload of the changed entries, one
 * device-to-device copy per copy-on-write page and the prefill kernels on
 * `stream`; returns without waiting.  Pools pkv_paged_prefill serves through
 * decode lanes keep a per-request scratch that grows to the largest chunk: a
 * chunk larger than any before frees and reallocates it, which waits for the
 * device (OUT_OF_MEMORY, nothing changed, if the allocation fails).
 */
int pkv_prefill_chunk(pkv_request* req, int layer, const void* q, const void* k, const void* v,
                      float* out, void* stream);

/* Make the pending position, or every position of the pending chunk, visible
 * ([SERVE-FLOW] step 3).  BAD_STATE unless a token or chunk is pending and
 * every layer ran pkv_append_and_attend (pkv_prefill_chunk) for it exactly
 * once ([CACHED-BIND]: all layers advance together).  Counters count each
 * position as one committed token: appends advance by layers, score cells by
 * layers x query_heads x min(t, window) for each new retained length t. */
int pkv_commit_token(pkv_request* req);

/* Drop the pending token or chunk ([SERVE-FLOW] step 4): the visible length
 * stays, the pages its begin leased (new or copy-on-write) go back to the
 * front of the free list, last leased first, and shared pages get their places
 * back, so table, page references and free list are exactly as before the
 * begin.  Rows already written stay in the pages, unreachable, and are
 * overwritten by the retry.  BAD_STATE if nothing is pending. */
int pkv_abort_token(pkv_request* req);

/* -------------------------------------------------------------- batched -- */

/*
 * Device scratch bytes that pkv_paged_decode_attention needs for `batch`
 * requests of at most max_seq_len tokens (split partial results and the
 * per-request tile prefix).  Depends on the pool's geometry and device.
 */
int pkv_workspace_size(const pkv_pool* pool, int batch, int64_t max_seq_len, size_t* bytes);

/*
 * Batched paged decode attention for one layer ([SERVE-PAGED] layout and
 * page table; [CACHED-MIX] arithmetic).  For every request b with retained
 * length t_b = seq_lens[b] (new token included, >= 1):
 *   1. store k_new[b], v_new[b] at logical position t_b - 1, i.e. physical page
 *      page_tables[b][(t_b - 1) / page_size], slot (t_b - 1) % page_size;
 *   2. for each query head q (KV head h = q / (query_heads / kv_heads)):
 *      out[b][q] = sum_j softmax_j(q[b][q] . K_j / sqrt(head_dim)) V_j, over the
 *      t_b keys K_j = K[page_tables[b][j / page_size]][h][j % page_size].
 *   q            [batch][query_heads][head_dim] fp32, device
 *   k_new, v_new [batch][kv_heads][head_dim] storage dtype, device
 *   page_tables  [batch][max_pages] int32, device (entries past ceil(t_b/page_size) unread)
 *   seq_lens     [batch] int32, device
 *   max_seq_len  host bound on every seq_lens entry (sizes the launch)
 *   out          [batch][query_heads][head_dim] fp32, device
 *   workspace    device scratch of >= pkv_workspace_size bytes (caller owned,
 *                16-byte aligned, contents need no initialisation)
 * Stateless over bookkeeping: the caller owns lengths and tables.  Bad
 * lengths or page ids found on the device set the pool's error word; the
 * affected request's rows of `out` are then unspecified.  Enqueues three kernels
 * on `stream` and returns without waiting.  Calls whose device work can overlap
 * must use different workspaces.
 */
int pkv_paged_decode_attention(pkv_pool* pool, int layer, int batch, const float* q,
                               const void* k_new, const void* v_new, const int32_t* page_tables,
                               int max_pages, const int32_t* seq_lens, int64_t max_seq_len,
                               float* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Device scratch bytes that pkv_paged_decode_attention_shared needs (see there);
 * equal to pkv_workspace_size when shared_len is 0.
 */
int pkv_workspace_size_shared(const pkv_pool* pool, int batch, int64_t max_seq_len,
                              int64_t shared_len, size_t* bytes);

/*
 * pkv_paged_decode_attention for a batch whose requests share a prefix: the
 * first shared_len positions of every request map to the same physical pages
 * (request 0's table entries 0 .. shared_len/page_size - 1), as after
 * pkv_request_fork of one prompt ([SERVE-SCOPE]: page sharing between
 * requests).  Same arguments, layout and results as pkv_paged_decode_attention;
 * the shared pages are read once per KV head instead of once per request.
 * The softmax over all t_b keys splits exactly into the shared keys and the
 * request's own keys and is merged back:
 *   out = (2^(m1-M) o1 + 2^(m2-M) o2) / (2^(m1-M) l1 + 2^(m2-M) l2),
 * (m, l, o) being each part's maximum, sum and unnormalised output.  The shared
 * part runs on the tensor cores with q and the weights split into bf16 hi + lo
 * (fp32-level products); the rest is the batched decode path.
 *   shared_len  multiple of page_size, 0 <= shared_len < max_seq_len; every
 *               request needs t_b > shared_len (its new row is its own); 0 is
 *               pkv_paged_decode_attention
 *   workspace   >= pkv_workspace_size_shared bytes
 * bf16 pools of head_dim 64 or 128: a table that differs from request 0's
 * within the prefix sets PKV_DEVERR_SHARED, a t_b <= shared_len sets
 * PKV_DEVERR_SEQ_LEN (rows of the affected requests unspecified); enqueues four
 * kernels on `stream` (plan, prefix, split over each request's own positions,
 * and a merge of the partials) and returns without waiting.  Other pools (fp32,
 * other head widths) run pkv_paged_decode_attention with the same arguments:
 * each request over its own pages, the same results, no shared reading and no
 * PKV_DEVERR_SHARED check.
 */
int pkv_paged_decode_attention_shared(pkv_pool* pool, int layer, int batch, const float* q,
                                      const void* k_new, const void* v_new,
                                      const int32_t* page_tables, int max_pages,
                                      const int32_t* seq_lens, int64_t max_seq_len,
                                      int64_t shared_len, float* out, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * Bytes of the fixed device array that pkv_paged_decode_attention_static uses
 * as scratch (8 MiB).  The CUDA runtime loads the array lazily, in each context
 * the first time its address is asked for; pkv_pool_create does so on the
 * pool's device, so the array is in place once a device pool exists, and it
 * stays until the context is destroyed (normally at process exit).
 */
#define PKV_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * pkv_paged_decode_attention without a workspace argument and without any
 * allocation.  The source pages have no counterpart to this call: it exists for
 * callers that cannot allocate device memory themselves, such as code embedded
 * in an application that has already reserved the GPU's memory for its own
 * arena and lends no allocator, or code that must not call cudaMalloc /
 * cudaFree on a latency-critical path because those calls can synchronise the
 * device.  Arguments, layout and results are those of
 * pkv_paged_decode_attention.
 *
 * Scratch is a file-scope device array of PKV_STATIC_SCRATCH_BYTES inside the
 * library.  The call makes no cudaMalloc, cudaFree or other allocating call: it
 * asks the runtime for the array's device address in the current context
 * (cudaGetSymbolAddress) on every call, a lookup once the array is loaded.  The
 * array is loaded when the pool is created (see PKV_STATIC_SCRATCH_BYTES); in a
 * context where no pool was created, for instance after a device reset, the
 * first call loads it and so allocates it, and should come before the
 * application reserves the rest of the device's memory and before any stream
 * capture.  A batch whose scratch need (pkv_workspace_size) exceeds
 * PKV_STATIC_SCRATCH_BYTES is rejected with PKV_ERR_INVALID_ARGUMENT and
 * changes nothing.  All calls on a device share the array and it keeps the last
 * call's contents: the per-lane arrival counters, the only part that must start
 * at zero, are cleared by each call's own plan kernel.  Calls whose device work
 * can overlap race on the array and must be serialised by the caller, for
 * instance by issuing them on one stream.
 */
int pkv_paged_decode_attention_static(pkv_pool* pool, int layer, int batch, const float* q,
                                      const void* k_new, const void* v_new,
                                      const int32_t* page_tables, int max_pages,
                                      const int32_t* seq_lens, int64_t max_seq_len, float* out,
                                      void* stream);

/* ------------------------------------------------------------- prefill -- */

/*
 * Device scratch bytes that pkv_paged_prefill needs for `batch` requests and
 * total_new new tokens (0 when either is 0).  The tensor-core implementation
 * needs a few bytes per request and query tile; the decode-lane one needs the
 * decode scratch of total_new requests, or of total_new / (8 / G) + batch blocks
 * of tokens (per chunk row about (head_dim + 2) * 4 bytes for each query head,
 * plus the split workers' partials) and, for bf16 storage, an fp32 copy of q.
 */
int pkv_prefill_workspace_size(const pkv_pool* pool, int batch, int64_t total_new, size_t* bytes);

/*
 * Batched prefill for one layer, writing the paged cache that decode reads
 * ([SERVE-PAGED]: a batched prefill may use a tiled, FlashAttention-style
 * computation while it writes the same paged cache; [SERVE-SCOPE] lists it as
 * not yet present there).  Request b appends n_b = cu_new[b+1] - cu_new[b] tokens
 * after its L0_b = seq_lens[b] - n_b cached ones.  For chunk token i of request
 * b (batch row x = cu_new[b] + i, position L0_b + i):
 *   1. store k_new[x], v_new[x] at that position, i.e. physical page
 *      page_tables[b][(L0_b + i) / page_size], slot (L0_b + i) % page_size;
 *   2. for each query head q (KV head h = q / (query_heads / kv_heads)):
 *      out[x][q] = sum_j softmax_j(q[x][q] . K_j / sqrt(head_dim)) V_j over the
 *      positions j = 0 .. L0_b + i (the pool's window, if any, keeps the last
 *      `window` of them) -- the outputs n_b successive decode steps would give.
 *   q            [total_new][query_heads][head_dim] storage dtype, device
 *   k_new, v_new [total_new][kv_heads][head_dim] storage dtype, device
 *   cu_new       [batch + 1] int32, device: row offsets, cu_new[0] = 0,
 *                non-decreasing, cu_new[batch] <= total_new
 *   page_tables  [batch][max_pages] int32, device (entries past
 *                ceil(seq_lens[b] / page_size) unread)
 *   seq_lens     [batch] int32, device: lengths after the chunk (>= n_b)
 *   out          [total_new][query_heads][head_dim] fp32, device
 *   workspace    device scratch of >= pkv_prefill_workspace_size bytes
 *                (caller owned, 16-byte aligned, no initialisation needed)
 * Two implementations, chosen by the pool.  bf16 pools of head_dim 64 or 128:
 * the tcgen05 tensor cores, bf16 products with fp32 accumulation, the weights
 * split into bf16 hi + lo before they multiply V (each weight carried
 * to about 2^-16); batch <= 1024.  Every other pool (fp32
 * storage, other head widths): decode lanes -- every chunk row is stored first,
 * then chunk token i of request b runs as one decode request of retained length
 * L0_b + i + 1 over request b's pages, all in one decode launch, with the decode
 * kernels' precision (fp32 weights; a bf16 q widened exactly to fp32).  fp32 pools
 * of head_dim 64 or 128 with 1, 2 or 4 query heads per KV head and no window run
 * 8 / G consecutive chunk tokens as one decode request (each token's rows masked
 * at its own position: the same results, each K/V tile read once per block).
 * Stateless over bookkeeping: the caller owns lengths and tables.  Bad lengths
 * or page ids found on the device set the pool's error word (a bad page reads as
 * zeros); the affected rows of `out` are then unspecified.  Once a wait has run out (PKV_DEVERR_TIMEOUT), later prefill
 * calls skip their attention work until pkv_check_device_status clears the
 * word.  Enqueues three kernels on `stream` (plan, append, attention; or rows,
 * decode plan, decode split) and returns without waiting; calls whose device
 * work can overlap must use different workspaces.
 */
int pkv_paged_prefill(pkv_pool* pool, int layer, int batch, int64_t total_new, const void* q,
                      const void* k_new, const void* v_new, const int32_t* cu_new,
                      const int32_t* page_tables, int max_pages, const int32_t* seq_lens,
                      float* out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------- tracing -- */

/*
 * Kernel timing hook.  When `before` and `after` are non-NULL cudaEvent_t
 * handles, every later pkv_append_and_attend / pkv_paged_decode_attention /
 * pkv_paged_prefill on this pool records `before` on its stream immediately
 * before the attention kernel and `after` immediately after it, so
 * cudaEventElapsedTime(before, after) is that kernel's device time.  NULL,
 * NULL turns the hook off.  The events stay owned by the caller.
 */
int pkv_pool_set_timing_events(pkv_pool* pool, void* before, void* after);

/* ----------------------------------------------------- failure injection -- */

/*
 * Test hooks that make one later call fail the way a real failure would, so that
 * the recovery the sources prescribe can be checked: after a failure,
 * pkv_abort_token leaves the visible length unchanged ([SERVE-FLOW] step 4), and a
 * rejected operation changes nothing ([CACHED-BIND]).  Nothing is armed unless this is
 * called; every hook fires once and is then disarmed.  One hook of each kind at a
 * time (arming a kind again replaces its hook).
 *   PKV_INJECT_NONE         disarm every hook.
 *   PKV_INJECT_LEASE        arg = n >= 1: the call that would take the n-th page
 *                           lease from now (pkv_lease_pages, pkv_begin_token,
 *                           pkv_begin_chunk; copy-on-write pages included) fails
 *                           with PKV_ERR_OUT_OF_PAGES and changes nothing.
 *   PKV_INJECT_LAYER        arg = layer: the next pkv_append_and_attend or
 *                           pkv_prefill_chunk on that layer that passes its
 *                           argument and state checks fails with PKV_ERR_CUDA
 *                           before it enqueues anything; the layer stays not run.
 *   PKV_INJECT_DEVICE_WAIT  arg = split-kernel worker (0 .. workers - 1), device
 *                           pools: in the split kernel of the next
 *                           pkv_append_and_attend or batched decode call
 *                           (pkv_paged_decode_attention and its _shared and
 *                           _static forms) on this pool, that worker arms the
 *                           barrier of its first staged tile
 *                           without issuing the tile's copy, and every bounded
 *                           wait of that launch gives up after wait_limit_ns
 *                           (1 ms .. 4 s).  The worker's wait runs out: it sets
 *                           PKV_DEVERR_TIMEOUT, lets the copies it did issue land
 *                           and returns; the rows its tiles feed are unspecified.
 *                           Nothing faults or hangs, and the context stays usable.
 * wait_limit_ns is read for PKV_INJECT_DEVICE_WAIT only.
 */
#define PKV_INJECT_NONE 0
#define PKV_INJECT_LEASE 1
#define PKV_INJECT_LAYER 2
#define PKV_INJECT_DEVICE_WAIT 3
int pkv_pool_inject_fault(pkv_pool* pool, int kind, int64_t arg, uint64_t wait_limit_ns);

/* -------------------------------------------------------------- status -- */

/* Synchronise the device, then read and clear the pool's device error word.
 * *bits (may be NULL) receives the PKV_DEVERR_* bits.  Returns
 * PKV_ERR_DEVICE_CHECK if any bit was set, PKV_ERR_CUDA if the device reports a
 * CUDA error. */
int pkv_check_device_status(pkv_pool* pool, uint32_t* bits);

/* Message of the last failed call on this thread ("" if none). */
const char* pkv_last_error(void);

/* Name of a status code. */
const char* pkv_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
