// Internal interface between the host library (pool.cpp) and the kernels
// (decode.cu).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

struct pkv_pool;

namespace pkv {

// Tuning constants of the split kernel (compile-time; overridable with -D for sweeps).
#ifndef PKV_SPLIT_WARPS
#define PKV_SPLIT_WARPS 8          // warps per CTA (one CTA per SM); each warp is one worker
#endif

constexpr int kTile = 16;          // key rows staged and processed as one unit
constexpr int kSplitWarps = PKV_SPLIT_WARPS;

// One launch of the decode path for one layer.
struct DecodeArgs {
    int dtype;               // PKV_F32 / PKV_BF16
    int B, H, D, P;          // requests, lane heads (KV heads << kv_shift), head width, page size
    int G;                   // query heads per lane (1: multi-head attention; at most 8)
    int kv_shift;            // lane head h reads KV head h >> kv_shift; H counts lanes, so
                             // more than 8 query heads per KV head run as 2^kv_shift lanes
    int64_t window;          // attend to the last `window` positions (0: the whole prefix)
    const float* q;          // [B][H*G][D]
    const void* k_new;       // [B][H][D] storage dtype
    const void* v_new;
    void* k_pages;           // this layer's pools, [pages][H][P][D]
    void* v_pages;
    int64_t n_pages;
    const int32_t* tables;   // [B][max_pages], or rows chosen by table_rows
    int max_pages;
    const int32_t* table_rows;  // nullptr, or [B] device: the table row request b reads
    const int32_t* seq_lens; // [B] device; nullptr => single request of length single_t
    int64_t single_t;
    int64_t max_seq_len;
    float* out;              // [B][H*G][D]
    void* workspace;
    size_t workspace_bytes;
    int workers;             // workers of this launch (split-kernel warps)
    unsigned* dev_error;
    cudaEvent_t ev_before;   // optional: recorded around the split kernel
    cudaEvent_t ev_after;
    uint32_t epoch;          // single request only: nonzero call epoch of the lane counters
                             // (no plan kernel; the workspace's counters started at zero)
    const void* tmap_k;      // CUtensorMap of this layer's K / V pools (host memory), or
    const void* tmap_v;      // nullptr: selects the tensor-core kernel when non-null
    // shared prefix (batched calls): the split kernel reads positions >= key_start and
    // merges pre_splits partials per query row from the prefix kernel, which
    // before_split(before_split_ctx, stream) enqueues between the plan and split kernels
    int64_t key_start;
    const void* pre_ml;      // float2 [pre_splits][pre_stride]: (max in log2 units, sum)
    const float* pre_o;      // float [pre_splits][pre_stride][D]: unnormalised outputs
    int pre_splits;
    int64_t pre_stride;      // query rows per split (B * query heads)
    cudaError_t (*before_split)(const void* ctx, cudaStream_t stream);
    const void* before_split_ctx;
    bool allow_empty;        // a seq_len of 0 is a request with no work (not an error)
    const int32_t* blk_tok0; // block lanes (see PrefillLanesArgs::block_tokens): [B] first
    const int32_t* blk_ntok; //   chunk row and token count of decode request x; nullptr: off
    int blk_gp, blk_hq;      //   the pool's query heads per KV head, and query heads
    uint64_t wait_limit_ns;  // bounded waits give up after this long (0: the default, 4 s)
    int inject_worker;       // failure injection: 0 off; else split worker inject_worker - 1
                             // arms its first stage's barrier without issuing the copy
};

// Bytes of a CUtensorMap (the driver's TMA descriptor).
constexpr int kTensorMapBytes = 128;

// True if the tensor-core kernel implements (dtype, D, G).
bool mma_supported(int dtype, int D, int G);

// Byte offsets of the scratch areas inside a workspace.
struct WorkspaceLayout {
    size_t req_prefix;   // int64 [B + 1]: tiles-per-lane prefix over requests
    size_t worker_req;   // int32 [workers]: request holding each worker's first tile
    size_t lane_cnt;     // uint64 [B*H]: partials deposited per lane (plan-zeroed or epoch-tagged)
    size_t part_ml;      // float2 [B*H + workers][G]: (running max in log2 units, sum)
    size_t part_o;       // float [B*H + workers][G][D]: unnormalised partial outputs
    size_t total;
};

WorkspaceLayout workspace_layout(int B, int H, int D, int workers, int G);

// Workers one launch uses: the pool's resident worker count, capped by the
// number of tiles the launch can hold (B * H * ceil(max_seq_len / kTile)).
int launch_workers(int pool_workers, int B, int H, int64_t max_seq_len, int kv_shift);

// Longest stretch of positions one query reads: max_seq_len, or with a
// sliding window the window plus one partial tile.
inline int64_t attended_len(int64_t max_seq_len, int64_t window) {
    return (window > 0 && window + kTile < max_seq_len) ? window + kTile : max_seq_len;
}

// Resident split-kernel warps per SM x SMs for this geometry on the current
// device; 0 if the geometry is not implemented.
int resident_workers(int dtype, int D, int G, int num_sms, bool tensor_cores);

// True if the kernels implement (dtype, D, G).
bool decode_supported(int dtype, int D, int G);

// Enqueue the plan and split kernels on `stream`.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// Device address, in the current context, of the fixed scratch array of
// pkv_paged_decode_attention_static; the first call in a context loads it.
cudaError_t static_scratch_address(void** ptr);

// Record a failed call in the thread's last-error message; returns `status`.
int record_error(int status, const char* fmt, ...);

// Validate the arguments of a batched call and fill `a` (all but the
// workspace); `*workspace_bytes` receives the scratch the launch needs.
// Returns PKV_OK (with a.B == 0 for an empty batch) or a recorded error.
int prepare_batched(pkv_pool* pool, int layer, int batch, const float* q, const void* k_new,
                    const void* v_new, const int32_t* page_tables, int max_pages,
                    const int32_t* seq_lens, int64_t max_seq_len, float* out, DecodeArgs* a,
                    size_t* workspace_bytes);

// ---------------------------------------------------------------- prefill --

// One launch of the batched prefill for one layer (bf16 pools, D 64 or 128).
struct PrefillArgs {
    int B, H, G, D, P;
    int64_t window;
    const void* q;           // [N][H*G][D] bf16
    const void* k_new;       // [N][H][D] bf16
    const void* v_new;
    void* k_pages;           // this layer's pools, [pages][H][P][D]
    void* v_pages;
    int64_t n_pages;
    const int32_t* cu_new;   // [B + 1] device; nullptr: one request, values below
    const int32_t* seq_lens; // [B] device, lengths after the chunk; nullptr: single_t
    int64_t single_n;        // one request without device arrays: its chunk length
    int64_t single_t;        //   and its length after the chunk
    const int32_t* tables;   // [B][max_pages] device
    int max_pages;
    int64_t total_new;       // N, rows of q / k_new / v_new / out
    float* out;              // [N][H*G][D] fp32
    void* workspace;
    unsigned* dev_error;
    cudaEvent_t ev_before;   // optional: recorded around the attention kernel
    cudaEvent_t ev_after;
    const void* tmap_k;      // CUtensorMap of this layer's K / V pools (host memory)
    const void* tmap_v;
};

// Upper bound on the query tiles of a call (sum over requests of ceil(n_b / (128 / G))).
int64_t prefill_max_tiles(int B, int G, int64_t total_new);

// Scratch bytes of one call.
size_t prefill_workspace_bytes(int B, int G, int64_t total_new);

// True if the prefill kernels implement (dtype, D, G).
bool prefill_supported(int dtype, int D, int G);

// Largest batch one call takes.
int prefill_max_batch();

// Enqueue the plan, append and attention kernels on `stream`.
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Batched prefill through decode lanes, for pools the tensor-core prefill does not
// serve (fp32 storage, other head widths): every chunk row is first stored in its
// page, then chunk token x of request b runs as decode request x of retained
// length L0_b + i + 1 over request b's table row -- the n_b successive decode
// steps the prefill stands for, at the decode kernels' precision.
struct PrefillLanesArgs {
    int dtype, D, P, kv_heads, query_heads;
    int lane_heads, lane_group, kv_shift;   // the pool's decode lanes
    int64_t window;
    int batch;
    int64_t total_new;
    const void* q;                // [N][query_heads][D] storage dtype
    const void* k_new;            // [N][kv_heads][D] storage dtype
    const void* v_new;
    void* k_pages;
    void* v_pages;
    int64_t n_pages;
    const int32_t* cu_new;        // [batch + 1] device; nullptr: one request (single_n, single_t)
    const int32_t* seq_lens;      // [batch] device
    int single_n;
    int64_t single_t;
    const int32_t* tables;        // [batch][max_pages]
    int max_pages;
    float* out;                   // [N][query_heads][D]
    void* workspace;
    size_t workspace_bytes;
    int workers;                  // decode workers of the launch
    unsigned* dev_error;
    const void* tmap_k;           // tensor-core decode kernel when non-null
    const void* tmap_v;
    cudaEvent_t ev_before;
    cudaEvent_t ev_after;
    // > 0: block lanes -- decode request x is a block of up to block_tokens consecutive
    // chunk tokens of one request (its last block may hold fewer), each token's query
    // heads rows of one lane of the tensor-core kernel with its own causal end;
    // 0: one decode request per chunk token
    int block_tokens;
};

// Chunk tokens per decode request of the decode-lane prefill: block lanes for fp32
// pools of head width 64 or 128 with 1, 2 or 4 query heads per KV head and no
// sliding window (8 lane rows on the tensor-core kernel), else 0.
int prefill_block_tokens(int dtype, int D, int G, int kv_shift, int64_t window, bool tmaps);

struct PrefillLanesLayout {
    int64_t requests;             // decode requests of the launch
    size_t decode;                // their decode workspace, at offset 0
    size_t rows, lens;            // int32 [requests]: table rows, lengths
    size_t tok0, ntok, first;     // block lanes: int32 [requests] first chunk row and token
                                  // count of each block, int32 [batch + 1] first block of
                                  // each request
    size_t q32;                   // fp32 widened q (bf16 pools)
    size_t total;
};
PrefillLanesLayout prefill_lanes_layout(int64_t N, int batch, int block_tokens, int lane_heads,
                                        int D, int workers, int lane_group, int query_heads,
                                        bool widen_q);
cudaError_t launch_prefill_lanes(const PrefillLanesArgs& a, cudaStream_t stream);

// ---------------------------------------------------------- shared prefix --

// How the prefix kernel cuts its work: 128-row tiles of (request, query head)
// rows per KV head, and key splits of split_len positions (whole 128-key tiles).
struct SharedPrefixPlan {
    int row_tiles;
    int64_t split_len;
    int splits;
};

SharedPrefixPlan shared_prefix_plan(int B, int H, int G, int64_t shared_len, int num_sms);

// True if the prefix kernel implements (dtype, D, G).
bool shared_prefix_supported(int dtype, int D, int G);

// One launch of the prefix kernel (the shared part of a batch's decode attention).
struct SharedPrefixArgs {
    int B, H, G, D, P, max_pages;
    int64_t window;
    int64_t n_pages;
    const float* q;          // [B][H*G][D] fp32
    const int32_t* tables;   // [B][max_pages]; request 0's first shared_len / P entries
    const int32_t* seq_lens; // [B]
    int64_t shared_len;
    SharedPrefixPlan plan;
    float2* pre_ml;          // [splits][B*H*G]
    float* pre_o;            // [splits][B*H*G][D]
    unsigned* dev_error;
    const void* tmap_k;      // CUtensorMap of this layer's K / V pools (host memory)
    const void* tmap_v;
};

cudaError_t launch_shared_prefix(const SharedPrefixArgs& a, cudaStream_t stream);

// DecodeArgs::before_split for a shared prefix: ctx is a SharedPrefixArgs.
cudaError_t launch_shared_prefix_hook(const void* ctx, cudaStream_t stream);

}  // namespace pkv
