// Host side of libpkv: the paged pool, its free list, per-request page tables,
// the begin / append / commit / abort transaction and the C ABI.
//
// Sources: "Incremental Serving", sections "Request flow" (the per-token
// transaction), "Paged KV-cache layout" (pools, page table, lazy leasing,
// default page size 16, block count 0 = one full context) and "Stable C and
// Python sessions" (opaque handles, capacity exhaustion reported, external
// synchronisation); "38 · Cached generation", sections "Bind one decoder to its
// model-wide cache" and "Assemble model-wide ... evidence" (all layers advance
// together, counters advance on commit, reset zeroes them, rejected operations
// change nothing).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <new>
#include <string>
#include <vector>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int ok() {
    g_last_error.clear();
    return PKV_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}


// SplitMix64 (Steele, Lea & Flood 2014).
struct SplitMix64 {
    uint64_t state;
    uint64_t next() {
        uint64_t z = (state += 0x9e3779b97f4a7c15ull);
        z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
        z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
        return z ^ (z >> 31);
    }
};

}  // namespace

struct pkv_pool {
    int layers = 0, heads = 0, head_dim = 0, page_size = 0, dtype = 0;
    int query_heads = 0, group = 1;    // query heads = group x KV heads (grouped-query attention)
    // decode runs on lanes of at most 8 query heads (16 on the tensor-core kernel): a
    // larger group (multi-query layouts, up to 128) is 2^kv_shift lanes of dec_group
    // per KV head, dec_heads = heads << kv_shift
    int dec_heads = 0, dec_group = 1, kv_shift = 0;
    int64_t window = 0;                // sliding window in positions (0: whole prefix)
    int64_t pages = 0, max_context = 0, max_pages_per_request = 0;
    bool host_only = false;
    std::deque<int32_t> free_list;     // front = next page to lease
    std::vector<int32_t> refs;         // requests referencing each physical page (0: free)
    void* k_base = nullptr;            // [layers][pages][H][P][D]
    void* v_base = nullptr;
    size_t layer_bytes = 0;
    unsigned* dev_error = nullptr;
    int device = -1;
    int sms = 0;                       // streaming multiprocessors of the device
    int workers = 0;                   // resident split-kernel warps on the device
    int64_t live_requests = 0;
    cudaEvent_t ev_before = nullptr;   // optional split-kernel timing events
    cudaEvent_t ev_after = nullptr;
    bool tensor_cores = false;         // decode: K/V tiles by TMA tensor loads, products by MMA
    bool tmaps = false;                // tensor maps built (head_dim 64 or 128)
    std::vector<CUtensorMap> tmap_k;   // per layer, when tmaps
    std::vector<CUtensorMap> tmap_v;
    // failure injection (pkv_pool_inject_fault), each hook one-shot
    int64_t inject_lease = 0;          // > 0: page leases until the one that fails
    int inject_layer = -1;             // >= 0: the next layer call on this layer fails
    int inject_worker = -1;            // >= 0: the next decode launch's worker skips a copy
    uint64_t inject_wait_ns = 0;       //        with this wait limit
};

struct pkv_request {
    pkv_pool* pool = nullptr;
    std::vector<int32_t> table;        // logical page -> physical page
    int64_t length = 0;                // visible (committed) length
    bool pending = false;
    int64_t position = 0;              // pending position (the first of a pending chunk)
    int64_t pending_n = 0;             // positions pending: 1 (begin_token) or n (begin_chunk)
    bool chunk = false;                // pending positions are a chunk (pkv_prefill_chunk)
    int64_t leased_count = 0;          // pages the begin appended to the table (leased last)
    std::vector<uint8_t> appended;     // per layer, for the pending token or chunk
    int appended_count = 0;
    pkv_counters counters{};
    int32_t* dev_table = nullptr;      // device copy, max_pages_per_request entries
    int64_t dev_dirty_from = 0;        // entries [dev_dirty_from, table.size()) not on the device
    void* dev_workspace = nullptr;
    size_t workspace_bytes = 0;
    int workspace_workers = 0;
    uint32_t epoch = 0;                // calls made on dev_workspace (lane-counter epochs)
    // copy-on-write of the pending positions: logical page idx moved from the
    // shared page old_page to the private page new_page (leased in ascending
    // idx, before any appended page); each layer's bytes are copied by that
    // layer's append or prefill
    struct CowPage {
        int64_t idx;
        int32_t old_page, new_page;
    };
    std::vector<CowPage> cow;
    std::vector<uint8_t> cow_copied;
    void* dev_prefill_ws = nullptr;    // prefill scratch for one request's chunks
    size_t prefill_ws_bytes = 0;
};

namespace {

// The kernels move head rows of q, k, v and out in vectors of up to 16 bytes:
// each tensor must start on a multiple of min(16, bytes of one head row).
int check_rows_aligned(const pkv_pool* p, const void* q, int q_es, const void* k, const void* v,
                       const void* out) {
    auto ok_at = [&](const void* x, int es) {
        const int64_t row = (int64_t)p->head_dim * es;
        const int64_t a = row < 16 ? row : 16;
        return reinterpret_cast<uintptr_t>(x) % (uintptr_t)a == 0;
    };
    const int kv_es = p->dtype == PKV_BF16 ? 2 : 4;
    if (!ok_at(q, q_es) || !ok_at(k, kv_es) || !ok_at(v, kv_es) || !ok_at(out, 4))
        return fail(PKV_ERR_INVALID_ARGUMENT,
                    "q, k, v and out must each start on a multiple of min(16, one head row's bytes)");
    return PKV_OK;
}

int elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : 2; }

// Which batched prefill serves a pool: the tensor-core kernel (bf16, head_dim 64
// or 128), or decode lanes (every other pool): chunk token by chunk token as
// decode requests in one launch.
bool tensor_prefill(const pkv_pool* p) {
    return p->tmaps && pkv::prefill_supported(p->dtype, p->head_dim, p->group);
}

// Chunk tokens per decode request of the decode-lane prefill (0: one per token).
int block_tokens(const pkv_pool* p) {
    return pkv::prefill_block_tokens(p->dtype, p->head_dim, p->dec_group, p->kv_shift, p->window,
                                     p->tmaps);
}

// Decode workers of a decode-lane prefill of n chunk tokens over `batch` requests:
// block lanes run on the tensor-core kernel with 8 rows a lane.
int lanes_workers(const pkv_pool* p, int batch, int64_t n) {
    const int bt = block_tokens(p);
    if (bt > 0) {
        const int resident = pkv::resident_workers(p->dtype, p->head_dim, 8, p->sms, true);
        return pkv::launch_workers(resident, (int)(n / bt + batch), p->heads,
                                   pkv::attended_len(p->max_context, p->window), 0);
    }
    return pkv::launch_workers(p->workers, (int)n, p->dec_heads,
                               pkv::attended_len(p->max_context, p->window), p->kv_shift);
}

size_t lanes_bytes(const pkv_pool* p, int batch, int64_t n) {
    return pkv::prefill_lanes_layout(n, batch, block_tokens(p), p->dec_heads, p->head_dim,
                                     lanes_workers(p, batch, n), p->dec_group, p->query_heads,
                                     p->dtype == PKV_BF16)
        .total;
}

pkv::PrefillLanesArgs lanes_args(pkv_pool* p, int layer, int batch, int64_t n) {
    pkv::PrefillLanesArgs a{};
    a.dtype = p->dtype;
    a.D = p->head_dim;
    a.P = p->page_size;
    a.kv_heads = p->heads;
    a.query_heads = p->query_heads;
    a.lane_heads = p->dec_heads;
    a.lane_group = p->dec_group;
    a.kv_shift = p->kv_shift;
    a.window = p->window;
    a.total_new = n;
    a.k_pages = static_cast<unsigned char*>(p->k_base) + (size_t)layer * p->layer_bytes;
    a.v_pages = static_cast<unsigned char*>(p->v_base) + (size_t)layer * p->layer_bytes;
    a.n_pages = p->pages;
    a.batch = batch;
    a.workers = lanes_workers(p, batch, n);
    a.dev_error = p->dev_error;
    a.ev_before = p->ev_before;
    a.ev_after = p->ev_after;
    // decode lanes read table rows: on the tensor-core kernel for fp32 pools that use
    // it or that run block lanes (the bf16 pools it serves prefill on the tcgen05
    // kernel, not through lanes)
    a.block_tokens = block_tokens(p);
    const bool tc = (p->tensor_cores && p->dtype == PKV_F32) || a.block_tokens > 0;
    a.tmap_k = tc ? &p->tmap_k[(size_t)layer] : nullptr;
    a.tmap_v = tc ? &p->tmap_v[(size_t)layer] : nullptr;
    return a;
}

// The driver's tensor-map encoder, fetched through the runtime (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    }
    return fn;
}

// One layer's K or V pool as a 2-D tensor [pages*H*P rows][D columns] of the
// storage type, read in boxes of 16 rows x 128 bytes (64 bf16 or 32 fp32 columns)
// with the 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, void* base, int64_t rows, int D, int dtype) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const int es = dtype == PKV_F32 ? 4 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * es};
    cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)pkv::kTile};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype == PKV_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void mark_dirty(pkv_request* r, int64_t from) {
    if (from < r->dev_dirty_from) r->dev_dirty_from = from;
}

// Take the free list's front page with one reference.
int32_t lease_front(pkv_pool* p) {
    const int32_t page = p->free_list.front();
    p->free_list.pop_front();
    p->refs[(size_t)page] = 1;
    return page;
}

// Drop one reference; a page nobody references goes back to the free list.
void drop_page(pkv_pool* p, int32_t page, bool front) {
    if (--p->refs[(size_t)page] == 0) {
        if (front) p->free_list.push_front(page);
        else p->free_list.push_back(page);
    }
}

// Failure injection: true (and the hook disarmed) when a call about to lease n
// pages reaches the lease armed to fail; else the leases are counted.
bool lease_fault(pkv_pool* p, int64_t n) {
    if (p->inject_lease <= 0 || n <= 0) return false;
    if (n >= p->inject_lease) {
        p->inject_lease = 0;
        return true;
    }
    p->inject_lease -= n;
    return false;
}

// Failure injection: true (and the hook disarmed) for the armed layer.
bool layer_fault(pkv_pool* p, int layer) {
    if (p->inject_layer < 0 || p->inject_layer != layer) return false;
    p->inject_layer = -1;
    return true;
}

// Failure injection: hand the armed split-worker copy skip to one launch.
void take_wait_fault(pkv_pool* p, pkv::DecodeArgs* a) {
    if (p->inject_worker < 0) return;
    a->inject_worker = p->inject_worker + 1;
    a->wait_limit_ns = p->inject_wait_ns;
    p->inject_worker = -1;
}

int check_device(const pkv_pool* p) {
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (cur != p->device)
        return fail(PKV_ERR_INVALID_ARGUMENT, "current device %d is not the pool's device %d", cur,
                    p->device);
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_version(void) { return 10000; }

const char* pkv_last_error(void) { return g_last_error.c_str(); }

const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARGUMENT: return "PKV_ERR_INVALID_ARGUMENT";
        case PKV_ERR_OUT_OF_PAGES: return "PKV_ERR_OUT_OF_PAGES";
        case PKV_ERR_CAPACITY_EXCEEDED: return "PKV_ERR_CAPACITY_EXCEEDED";
        case PKV_ERR_BAD_STATE: return "PKV_ERR_BAD_STATE";
        case PKV_ERR_OUT_OF_MEMORY: return "PKV_ERR_OUT_OF_MEMORY";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_DEVICE_CHECK: return "PKV_ERR_DEVICE_CHECK";
        case PKV_ERR_NO_STORAGE: return "PKV_ERR_NO_STORAGE";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        default: return "PKV_ERR_UNKNOWN";
    }
}

int pkv_pool_options_init(pkv_pool_options* o) {
    if (!o) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL options");
    *o = pkv_pool_options{};
    o->layers = 1;
    o->pages = 0;
    o->kv_heads = 1;
    o->query_heads = 0;
    o->head_dim = 128;
    o->page_size = 16;
    o->dtype = PKV_BF16;
    o->max_context = 4096;
    o->seed = 0;
    o->flags = 0;
    o->window = 0;
    return ok();
}

int pkv_pool_create(int layers, int64_t pages, int heads, int head_dim, int page_size, int dtype,
                    int64_t max_context, uint64_t seed, unsigned flags, pkv_pool** out) {
    pkv_pool_options o{};
    o.layers = layers;
    o.pages = pages;
    o.kv_heads = heads;
    o.query_heads = heads;
    o.head_dim = head_dim;
    o.page_size = page_size;
    o.dtype = dtype;
    o.max_context = max_context;
    o.seed = seed;
    o.flags = flags;
    o.window = 0;
    return pkv_pool_create_ex(&o, out);
}

int pkv_pool_create_ex(const pkv_pool_options* opts, pkv_pool** out) {
    if (!out || !opts) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    *out = nullptr;
    const int layers = opts->layers, heads = opts->kv_heads, head_dim = opts->head_dim;
    const int page_size = opts->page_size, dtype = opts->dtype;
    int64_t pages = opts->pages;
    const int64_t max_context = opts->max_context;
    const uint64_t seed = opts->seed;
    const unsigned flags = opts->flags;
    const int query_heads = opts->query_heads == 0 ? heads : opts->query_heads;
    if (opts->window < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "negative window");
    if (heads >= 1 && (query_heads < heads || query_heads % heads != 0))
        return fail(PKV_ERR_INVALID_ARGUMENT, "query_heads %d is not a multiple of kv_heads %d",
                    query_heads, heads);
    if (layers < 1 || heads < 1 || head_dim < 1 || page_size < 1 || max_context < 1 || pages < 0)
        return fail(PKV_ERR_INVALID_ARGUMENT,
                    "bad geometry: layers=%d heads=%d head_dim=%d page_size=%d max_context=%lld "
                    "pages=%lld",
                    layers, heads, head_dim, page_size, (long long)max_context, (long long)pages);
    if (dtype != PKV_F32 && dtype != PKV_BF16)
        return fail(PKV_ERR_INVALID_ARGUMENT, "dtype %d is neither PKV_F32 nor PKV_BF16", dtype);
    if (flags & ~(PKV_POOL_HOST_ONLY | PKV_POOL_CUDA_CORES))
        return fail(PKV_ERR_INVALID_ARGUMENT, "unknown flags");
    const bool host_only = (flags & PKV_POOL_HOST_ONLY) != 0;
    const int64_t per_request = (max_context + page_size - 1) / page_size;
    if (pages == 0) pages = per_request;
    if (pages > INT32_MAX || per_request > INT32_MAX)
        return fail(PKV_ERR_INVALID_ARGUMENT, "page ids must fit in int32");
    if (!host_only) {
        if (page_size % pkv::kTile != 0)
            return fail(PKV_ERR_UNSUPPORTED, "page_size %d is not a multiple of %d", page_size,
                        pkv::kTile);
        const int g = query_heads / heads;
        const bool group_ok = g <= 8 || (g <= 128 && (g & (g - 1)) == 0);
        if (!group_ok || !pkv::decode_supported(dtype, head_dim, g <= 8 ? g : 8))
            return fail(PKV_ERR_UNSUPPORTED,
                        "head_dim %d with %d query heads per KV head not implemented (powers of "
                        "two, 2..128 fp32, 2..256 bf16; groups of 2, 4, ..., 128 at head_dim 64, "
                        "128)",
                        head_dim, g);
    }

    pkv_pool* p = new (std::nothrow) pkv_pool;
    if (!p) return fail(PKV_ERR_OUT_OF_MEMORY, "host allocation failed");
    p->layers = layers;
    p->heads = heads;
    p->query_heads = query_heads;
    p->group = query_heads / heads;
    p->dec_group = p->group <= 8 ? p->group : 8;
    while ((p->dec_group << p->kv_shift) < p->group) ++p->kv_shift;
    p->dec_heads = heads << p->kv_shift;
    p->window = opts->window;
    p->head_dim = head_dim;
    p->page_size = page_size;
    p->dtype = dtype;
    p->pages = pages;
    p->max_context = max_context;
    p->max_pages_per_request = per_request;
    p->host_only = host_only;

    // free list: Fisher-Yates shuffle of 0..pages-1 with SplitMix64(seed)
    std::vector<int32_t> order((size_t)pages);
    for (int64_t i = 0; i < pages; ++i) order[(size_t)i] = (int32_t)i;
    SplitMix64 rng{seed};
    for (int64_t i = pages - 1; i > 0; --i) {
        const int64_t j = (int64_t)(rng.next() % (uint64_t)(i + 1));
        std::swap(order[(size_t)i], order[(size_t)j]);
    }
    p->free_list.assign(order.begin(), order.end());
    p->refs.assign((size_t)pages, 0);

    if (!host_only) {
        cudaError_t e = cudaGetDevice(&p->device);
        int sms = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
        if (e != cudaSuccess) {
            delete p;
            return cuda_fail(e, "device query");
        }
        p->sms = sms;
        const int64_t rows = pages * page_size * heads;   // pool rows of one layer
        p->tmaps = (head_dim == 64 || head_dim == 128) && rows < INT32_MAX &&
                   tensor_map_encoder() != nullptr;
        p->tensor_cores = p->tmaps && !(flags & PKV_POOL_CUDA_CORES) &&
                          pkv::mma_supported(dtype, head_dim, p->dec_group);
        if (p->tensor_cores && p->group >= 16 && pkv::mma_supported(dtype, head_dim, 16)) {
            // lanes of 16 query heads
            p->dec_group = 16;
            p->kv_shift = 0;
            while ((p->dec_group << p->kv_shift) < p->group) ++p->kv_shift;
            p->dec_heads = heads << p->kv_shift;
        }
        p->workers = pkv::resident_workers(dtype, head_dim, p->dec_group, sms, p->tensor_cores);
        if (p->workers <= 0) {
            delete p;
            return fail(PKV_ERR_CUDA, "split kernel cannot be resident on this device");
        }
        p->layer_bytes = (size_t)pages * page_size * heads * head_dim * elem_bytes(dtype);
        const size_t total = p->layer_bytes * (size_t)layers;
        if ((e = cudaMalloc(&p->k_base, total)) != cudaSuccess ||
            (e = cudaMalloc(&p->v_base, total)) != cudaSuccess ||
            (e = cudaMalloc(&p->dev_error, sizeof(unsigned))) != cudaSuccess) {
            cudaFree(p->k_base);
            cudaFree(p->v_base);
            cudaFree(p->dev_error);
            delete p;
            cudaGetLastError();
            return fail(PKV_ERR_OUT_OF_MEMORY, "cudaMalloc of 2 x %zu bytes: %s", total,
                        cudaGetErrorString(e));
        }
        if (p->tmaps) {
            p->tmap_k.resize((size_t)layers);
            p->tmap_v.resize((size_t)layers);
            for (int l = 0; l < layers; ++l) {
                char* kb = static_cast<char*>(p->k_base) + p->layer_bytes * (size_t)l;
                char* vb = static_cast<char*>(p->v_base) + p->layer_bytes * (size_t)l;
                if (!encode_pool_map(&p->tmap_k[(size_t)l], kb, rows, head_dim, dtype) ||
                    !encode_pool_map(&p->tmap_v[(size_t)l], vb, rows, head_dim, dtype)) {
                    cudaFree(p->k_base);
                    cudaFree(p->v_base);
                    cudaFree(p->dev_error);
                    delete p;
                    return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for layer %d", l);
                }
            }
        }
        // load the fixed scratch array of pkv_paged_decode_attention_static on this
        // device now, while memory is available, rather than in that call
        void* static_scratch = nullptr;
        if ((e = pkv::static_scratch_address(&static_scratch)) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(p->k_base);
            cudaFree(p->v_base);
            cudaFree(p->dev_error);
            delete p;
            return cuda_fail(e, "loading the static scratch array");
        }
        if ((e = cudaMemset(p->k_base, 0, total)) != cudaSuccess ||
            (e = cudaMemset(p->v_base, 0, total)) != cudaSuccess ||
            (e = cudaMemset(p->dev_error, 0, sizeof(unsigned))) != cudaSuccess ||
            (e = cudaDeviceSynchronize()) != cudaSuccess) {
            cudaFree(p->k_base);
            cudaFree(p->v_base);
            cudaFree(p->dev_error);
            delete p;
            return cuda_fail(e, "zero-fill pool");
        }
    }
    *out = p;
    return ok();
}

int pkv_pool_destroy(pkv_pool* p) {
    if (!p) return ok();
    if (p->live_requests != 0)
        return fail(PKV_ERR_BAD_STATE, "%lld requests still use the pool",
                    (long long)p->live_requests);
    if (!p->host_only) {
        cudaFree(p->k_base);
        cudaFree(p->v_base);
        cudaFree(p->dev_error);
    }
    delete p;
    return ok();
}

int pkv_pool_kv_ptr(const pkv_pool* p, int layer, void** k_pages, void** v_pages) {
    if (!p || !k_pages || !v_pages) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    if (layer < 0 || layer >= p->layers)
        return fail(PKV_ERR_INVALID_ARGUMENT, "layer %d outside [0, %d)", layer, p->layers);
    if (p->host_only) return fail(PKV_ERR_NO_STORAGE, "host-only pool has no device storage");
    *k_pages = static_cast<char*>(p->k_base) + p->layer_bytes * (size_t)layer;
    *v_pages = static_cast<char*>(p->v_base) + p->layer_bytes * (size_t)layer;
    return ok();
}

int pkv_pool_heads(const pkv_pool* p, int* kv_heads, int* query_heads) {
    if (!p) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pool");
    if (kv_heads) *kv_heads = p->heads;
    if (query_heads) *query_heads = p->query_heads;
    return ok();
}

int pkv_pool_kernel(const pkv_pool* p, int* tensor_cores) {
    if (!p || !tensor_cores) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    *tensor_cores = p->tensor_cores ? 1 : 0;
    return ok();
}

int pkv_pool_bytes(const pkv_pool* p, uint64_t* bytes) {
    if (!p || !bytes) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    *bytes = 2ull * (uint64_t)p->layers * (uint64_t)p->pages * (uint64_t)p->page_size *
             (uint64_t)p->heads * (uint64_t)p->head_dim * (uint64_t)elem_bytes(p->dtype);
    return ok();
}

int pkv_pool_pages(const pkv_pool* p, int64_t* pages, int64_t* free_pages) {
    if (!p) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pool");
    if (pages) *pages = p->pages;
    if (free_pages) *free_pages = (int64_t)p->free_list.size();
    return ok();
}

int pkv_pool_free_list(const pkv_pool* p, int32_t* host_out, int64_t cap, int64_t* n) {
    if (!p || !n || cap < 0 || (cap > 0 && !host_out))
        return fail(PKV_ERR_INVALID_ARGUMENT, "bad argument");
    *n = (int64_t)p->free_list.size();
    int64_t i = 0;
    for (auto it = p->free_list.begin(); it != p->free_list.end() && i < cap; ++it) host_out[i++] = *it;
    return ok();
}

int pkv_request_create(pkv_pool* p, pkv_request** out) {
    if (!p || !out) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    *out = nullptr;
    pkv_request* r = new (std::nothrow) pkv_request;
    if (!r) return fail(PKV_ERR_OUT_OF_MEMORY, "host allocation failed");
    r->pool = p;
    r->appended.assign((size_t)p->layers, 0);
    r->cow_copied.assign((size_t)p->layers, 0);
    r->table.reserve((size_t)p->max_pages_per_request);
    if (!p->host_only) {
        int rc = check_device(p);
        if (rc != PKV_OK) {
            delete r;
            return rc;
        }
        r->workspace_workers =
            pkv::launch_workers(p->workers, 1, p->dec_heads, pkv::attended_len(p->max_context, p->window), p->kv_shift);
        r->workspace_bytes =
            pkv::workspace_layout(1, p->dec_heads, p->head_dim, r->workspace_workers, p->dec_group).total;
        if (p->tmaps && pkv::prefill_supported(p->dtype, p->head_dim, p->group))
            r->prefill_ws_bytes = pkv::prefill_workspace_bytes(1, p->group, p->max_context);
        cudaError_t e = cudaMalloc(&r->dev_table, sizeof(int32_t) * (size_t)p->max_pages_per_request);
        if (e == cudaSuccess) e = cudaMalloc(&r->dev_workspace, r->workspace_bytes);
        if (e == cudaSuccess) e = cudaMemset(r->dev_workspace, 0, r->workspace_bytes);
        if (e == cudaSuccess && r->prefill_ws_bytes)
            e = cudaMalloc(&r->dev_prefill_ws, r->prefill_ws_bytes);
        if (e != cudaSuccess) {
            cudaFree(r->dev_table);
            cudaFree(r->dev_workspace);
            cudaFree(r->dev_prefill_ws);
            delete r;
            cudaGetLastError();
            return fail(PKV_ERR_OUT_OF_MEMORY, "cudaMalloc for request: %s", cudaGetErrorString(e));
        }
    }
    ++p->live_requests;
    *out = r;
    return ok();
}

int pkv_request_destroy(pkv_request* r) {
    if (!r) return ok();
    pkv_pool* p = r->pool;
    if (r->pending) pkv_abort_token(r);
    for (int32_t pg : r->table) drop_page(p, pg, false);
    if (!p->host_only) {
        cudaFree(r->dev_table);
        cudaFree(r->dev_workspace);
        cudaFree(r->dev_prefill_ws);
    }
    --p->live_requests;
    delete r;
    return ok();
}

int pkv_lease_pages(pkv_request* r, int64_t n) {
    if (!r) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL request");
    pkv_pool* p = r->pool;
    if (r->pending) return fail(PKV_ERR_BAD_STATE, "a token is pending");
    if (n < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "negative page count %lld", (long long)n);
    if ((int64_t)r->table.size() + n > p->max_pages_per_request)
        return fail(PKV_ERR_CAPACITY_EXCEEDED,
                    "%lld + %lld pages exceed one maximum-length context (%lld pages)",
                    (long long)r->table.size(), (long long)n, (long long)p->max_pages_per_request);
    if (n > (int64_t)p->free_list.size())
        return fail(PKV_ERR_OUT_OF_PAGES, "%lld pages requested, %lld free", (long long)n,
                    (long long)p->free_list.size());
    if (lease_fault(p, n)) return fail(PKV_ERR_OUT_OF_PAGES, "injected lease failure");
    mark_dirty(r, (int64_t)r->table.size());
    for (int64_t i = 0; i < n; ++i) r->table.push_back(lease_front(p));
    return ok();
}

int pkv_release_pages(pkv_request* r) {
    if (!r) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL request");
    if (r->pending) return fail(PKV_ERR_BAD_STATE, "a token is pending");
    for (int32_t pg : r->table) drop_page(r->pool, pg, false);
    r->table.clear();
    r->length = 0;
    r->counters = pkv_counters{};
    r->dev_dirty_from = 0;
    return ok();
}

int pkv_request_length(const pkv_request* r, int64_t* visible_len) {
    if (!r || !visible_len) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    *visible_len = r->length;
    return ok();
}

int pkv_request_page_table(const pkv_request* r, int32_t* host_out, int64_t cap, int64_t* n_pages) {
    if (!r || !n_pages || cap < 0 || (cap > 0 && !host_out))
        return fail(PKV_ERR_INVALID_ARGUMENT, "bad argument");
    *n_pages = (int64_t)r->table.size();
    const int64_t n = *n_pages < cap ? *n_pages : cap;
    if (n > 0) std::memcpy(host_out, r->table.data(), sizeof(int32_t) * (size_t)n);
    return ok();
}

int pkv_request_counters(const pkv_request* r, pkv_counters* out) {
    if (!r || !out) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    *out = r->counters;
    return ok();
}

}  // extern "C"

namespace {

// Open n pending positions at the visible length: copy-on-write replacements
// for the shared pages among those the positions write (ascending logical
// index), then pages for logical indices the request does not hold yet, all
// from the free list's front.  All or nothing.
int begin_pending(pkv_request* r, int64_t n, bool chunk, int64_t* position) {
    pkv_pool* p = r->pool;
    if (r->pending) return fail(PKV_ERR_BAD_STATE, "a token is already pending");
    if (r->length + n > p->max_context)
        return fail(PKV_ERR_CAPACITY_EXCEEDED, "%lld + %lld positions pass the maximum context %lld",
                    (long long)r->length, (long long)n, (long long)p->max_context);
    const int64_t first = r->length / p->page_size;
    const int64_t last = (r->length + n - 1) / p->page_size;
    const int64_t held = (int64_t)r->table.size();
    int64_t shared = 0;
    for (int64_t idx = first; idx <= last && idx < held; ++idx)
        if (p->refs[(size_t)r->table[(size_t)idx]] > 1) ++shared;
    const int64_t fresh = last + 1 > held ? last + 1 - held : 0;
    if (shared + fresh > (int64_t)p->free_list.size())
        return fail(PKV_ERR_OUT_OF_PAGES, "%lld pages needed, %lld free", (long long)(shared + fresh),
                    (long long)p->free_list.size());
    if (lease_fault(p, shared + fresh)) return fail(PKV_ERR_OUT_OF_PAGES, "injected lease failure");
    r->cow.clear();
    for (int64_t idx = first; idx <= last && idx < held; ++idx) {
        const int32_t old = r->table[(size_t)idx];
        if (p->refs[(size_t)old] <= 1) continue;
        // the page is shared with another request: write into a private copy;
        // the reference to the shared page is kept until commit
        const int32_t page = lease_front(p);
        r->table[(size_t)idx] = page;
        r->cow.push_back({idx, old, page});
        mark_dirty(r, idx);
    }
    if (fresh) mark_dirty(r, held);
    for (int64_t i = 0; i < fresh; ++i) r->table.push_back(lease_front(p));
    r->leased_count = fresh;
    std::fill(r->cow_copied.begin(), r->cow_copied.end(), 0);
    r->pending = true;
    r->position = r->length;
    r->pending_n = n;
    r->chunk = chunk;
    std::fill(r->appended.begin(), r->appended.end(), 0);
    r->appended_count = 0;
    if (position) *position = r->position;
    return ok();
}

// Before a layer's first write for the pending positions: upload the changed
// page-table entries and copy this layer's bytes of every shared page into its
// private replacement.
int prepare_layer_write(pkv_request* r, int layer, cudaStream_t s) {
    pkv_pool* p = r->pool;
    const int64_t n = (int64_t)r->table.size();
    if (r->dev_dirty_from < n) {
        cudaError_t e = cudaMemcpyAsync(r->dev_table + r->dev_dirty_from,
                                        r->table.data() + r->dev_dirty_from,
                                        sizeof(int32_t) * (size_t)(n - r->dev_dirty_from),
                                        cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "page-table upload");
        r->dev_dirty_from = n;
    }
    if (!r->cow.empty() && !r->cow_copied[(size_t)layer]) {
        const size_t page_bytes = (size_t)p->page_size * p->heads * p->head_dim * elem_bytes(p->dtype);
        char* kb = static_cast<char*>(p->k_base) + p->layer_bytes * (size_t)layer;
        char* vb = static_cast<char*>(p->v_base) + p->layer_bytes * (size_t)layer;
        for (const auto& c : r->cow) {
            cudaError_t e = cudaMemcpyAsync(kb + page_bytes * (size_t)c.new_page,
                                            kb + page_bytes * (size_t)c.old_page, page_bytes,
                                            cudaMemcpyDeviceToDevice, s);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(vb + page_bytes * (size_t)c.new_page,
                                    vb + page_bytes * (size_t)c.old_page, page_bytes,
                                    cudaMemcpyDeviceToDevice, s);
            if (e != cudaSuccess) return cuda_fail(e, "copy-on-write page copy");
        }
        r->cow_copied[(size_t)layer] = 1;
    }
    return PKV_OK;
}

// Sum over t = t0+1 .. t0+n of min(t, window) (window 0: of t).
int64_t attended_sum(int64_t t0, int64_t n, int64_t window) {
    const int64_t a = t0 + 1, b = t0 + n;
    if (window <= 0 || b <= window) return (a + b) * n / 2;
    if (a > window) return window * n;
    return (a + window) * (window - a + 1) / 2 + window * (b - window);
}

}  // namespace

extern "C" {

int pkv_begin_token(pkv_request* r, int64_t* position) {
    if (!r) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL request");
    return begin_pending(r, 1, false, position);
}

int pkv_begin_chunk(pkv_request* r, int64_t n, int64_t* position) {
    if (!r) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL request");
    if (n < 1) return fail(PKV_ERR_INVALID_ARGUMENT, "a chunk holds at least one token");
    return begin_pending(r, n, true, position);
}

int pkv_append_and_attend(pkv_request* r, int layer, const float* q, const void* k, const void* v,
                          float* out, void* stream) {
    if (!r) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL request");
    pkv_pool* p = r->pool;
    if (!q || !k || !v || !out) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL tensor pointer");
    if (layer < 0 || layer >= p->layers)
        return fail(PKV_ERR_INVALID_ARGUMENT, "layer %d outside [0, %d)", layer, p->layers);
    if (int rc = check_rows_aligned(p, q, 4, k, v, out); rc != PKV_OK) return rc;
    if (p->host_only) return fail(PKV_ERR_NO_STORAGE, "host-only pool has no device storage");
    if (!r->pending) return fail(PKV_ERR_BAD_STATE, "no token pending");
    if (r->chunk) return fail(PKV_ERR_BAD_STATE, "a chunk is pending (pkv_prefill_chunk)");
    if (r->appended[(size_t)layer]) return fail(PKV_ERR_BAD_STATE, "layer %d already ran", layer);
    int rc = check_device(p);
    if (rc != PKV_OK) return rc;
    if (layer_fault(p, layer)) return fail(PKV_ERR_CUDA, "injected failure on layer %d", layer);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = prepare_layer_write(r, layer, s);
    if (rc != PKV_OK) return rc;
    pkv::DecodeArgs a{};
    a.dtype = p->dtype;
    a.B = 1;
    a.H = p->dec_heads;
    a.G = p->dec_group;
    a.kv_shift = p->kv_shift;
    a.window = p->window;
    a.tmap_k = p->tensor_cores ? &p->tmap_k[(size_t)layer] : nullptr;
    a.tmap_v = p->tensor_cores ? &p->tmap_v[(size_t)layer] : nullptr;
    a.D = p->head_dim;
    a.P = p->page_size;
    a.q = q;
    a.k_new = k;
    a.v_new = v;
    void *kp, *vp;
    pkv_pool_kv_ptr(p, layer, &kp, &vp);
    a.k_pages = kp;
    a.v_pages = vp;
    a.n_pages = p->pages;
    a.tables = r->dev_table;
    a.max_pages = (int)p->max_pages_per_request;
    a.seq_lens = nullptr;
    a.single_t = r->position + 1;
    a.max_seq_len = r->position + 1;
    a.out = out;
    a.workspace = r->dev_workspace;
    a.workspace_bytes = r->workspace_bytes;
    a.workers = pkv::launch_workers(r->workspace_workers, 1, p->dec_heads, pkv::attended_len(r->position + 1, p->window), p->kv_shift);
    a.dev_error = p->dev_error;
    a.ev_before = p->ev_before;
    a.ev_after = p->ev_after;
    take_wait_fault(p, &a);
    if (r->epoch == UINT32_MAX) {
        // epochs must increase: after 2^32 - 1 calls start over from zeroed counters
        cudaError_t z = cudaMemsetAsync(r->dev_workspace, 0, r->workspace_bytes, s);
        if (z != cudaSuccess) return cuda_fail(z, "workspace reset");
        r->epoch = 0;
    }
    a.epoch = r->epoch + 1;
    cudaError_t e = pkv::launch_decode(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    r->epoch = a.epoch;
    r->appended[(size_t)layer] = 1;
    ++r->appended_count;
    return ok();
}

int pkv_prefill_chunk(pkv_request* r, int layer, const void* q, const void* k, const void* v,
                      float* out, void* stream) {
    if (!r) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL request");
    pkv_pool* p = r->pool;
    if (!q || !k || !v || !out) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL tensor pointer");
    if (layer < 0 || layer >= p->layers)
        return fail(PKV_ERR_INVALID_ARGUMENT, "layer %d outside [0, %d)", layer, p->layers);
    if (int rc = check_rows_aligned(p, q, elem_bytes(p->dtype), k, v, out); rc != PKV_OK) return rc;
    if (p->host_only) return fail(PKV_ERR_NO_STORAGE, "host-only pool has no device storage");
    if (!r->pending || !r->chunk) return fail(PKV_ERR_BAD_STATE, "no chunk pending");
    if (r->appended[(size_t)layer]) return fail(PKV_ERR_BAD_STATE, "layer %d already ran", layer);
    int rc = check_device(p);
    if (rc != PKV_OK) return rc;
    if (layer_fault(p, layer)) return fail(PKV_ERR_CUDA, "injected failure on layer %d", layer);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!tensor_prefill(p)) {
        // decode lanes: the request's scratch grows to the chunk (freeing the old
        // one waits for the device)
        const size_t need = lanes_bytes(p, 1, r->pending_n);
        if (r->prefill_ws_bytes < need) {
            void* ws = nullptr;
            cudaError_t e = cudaMalloc(&ws, need);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return fail(PKV_ERR_OUT_OF_MEMORY, "prefill scratch of %zu bytes", need);
            }
            if (r->dev_prefill_ws) cudaFree(r->dev_prefill_ws);
            r->dev_prefill_ws = ws;
            r->prefill_ws_bytes = need;
        }
        rc = prepare_layer_write(r, layer, s);
        if (rc != PKV_OK) return rc;
        pkv::PrefillLanesArgs a = lanes_args(p, layer, 1, r->pending_n);
        a.q = q;
        a.k_new = k;
        a.v_new = v;
        a.cu_new = nullptr;
        a.seq_lens = nullptr;
        a.single_n = (int)r->pending_n;
        a.single_t = r->position + r->pending_n;
        a.tables = r->dev_table;
        a.max_pages = (int)p->max_pages_per_request;
        a.out = out;
        a.workspace = r->dev_prefill_ws;
        a.workspace_bytes = r->prefill_ws_bytes;
        cudaError_t e = pkv::launch_prefill_lanes(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
        r->appended[(size_t)layer] = 1;
        ++r->appended_count;
        return ok();
    }
    rc = prepare_layer_write(r, layer, s);
    if (rc != PKV_OK) return rc;
    pkv::PrefillArgs a{};
    a.B = 1;
    a.H = p->heads;
    a.G = p->group;
    a.D = p->head_dim;
    a.P = p->page_size;
    a.window = p->window;
    a.q = q;
    a.k_new = k;
    a.v_new = v;
    void *kp, *vp;
    pkv_pool_kv_ptr(p, layer, &kp, &vp);
    a.k_pages = kp;
    a.v_pages = vp;
    a.n_pages = p->pages;
    a.cu_new = nullptr;
    a.seq_lens = nullptr;
    a.single_n = r->pending_n;
    a.single_t = r->position + r->pending_n;
    a.tables = r->dev_table;
    a.max_pages = (int)p->max_pages_per_request;
    a.total_new = r->pending_n;
    a.out = out;
    a.workspace = r->dev_prefill_ws;
    a.dev_error = p->dev_error;
    a.ev_before = p->ev_before;
    a.ev_after = p->ev_after;
    a.tmap_k = &p->tmap_k[(size_t)layer];
    a.tmap_v = &p->tmap_v[(size_t)layer];
    cudaError_t e = pkv::launch_prefill(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    r->appended[(size_t)layer] = 1;
    ++r->appended_count;
    return ok();
}

int pkv_commit_token(pkv_request* r) {
    if (!r) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL request");
    pkv_pool* p = r->pool;
    if (!r->pending) return fail(PKV_ERR_BAD_STATE, "no token pending");
    if (r->appended_count != p->layers)
        return fail(PKV_ERR_BAD_STATE, "%d of %d layers appended", r->appended_count, p->layers);
    const int64_t n = r->pending_n;
    for (const auto& c : r->cow) drop_page(p, c.old_page, false);
    r->counters.committed_tokens += n;
    r->counters.cache_appends += (int64_t)p->layers * n;
    r->counters.score_cells +=
        (int64_t)p->layers * p->query_heads * attended_sum(r->position, n, p->window);
    r->length = r->position + n;
    r->pending = false;
    r->chunk = false;
    r->leased_count = 0;
    r->cow.clear();
    return ok();
}

int pkv_abort_token(pkv_request* r) {
    if (!r) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL request");
    if (!r->pending) return fail(PKV_ERR_BAD_STATE, "no token pending");
    pkv_pool* p = r->pool;
    // back to the free list's front, last leased first, so the pool is exactly
    // as before the begin
    for (int64_t i = 0; i < r->leased_count; ++i) {
        const int32_t pg = r->table.back();
        r->table.pop_back();
        drop_page(p, pg, true);
    }
    if (r->leased_count) mark_dirty(r, (int64_t)r->table.size());
    for (auto it = r->cow.rbegin(); it != r->cow.rend(); ++it) {
        r->table[(size_t)it->idx] = it->old_page;
        drop_page(p, it->new_page, true);
        mark_dirty(r, it->idx);
    }
    r->pending = false;
    r->chunk = false;
    r->leased_count = 0;
    r->cow.clear();
    return ok();
}

int pkv_request_fork(const pkv_request* parent, pkv_request** out) {
    if (!parent || !out) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    *out = nullptr;
    if (parent->pending) return fail(PKV_ERR_BAD_STATE, "the parent has a token pending");
    pkv_request* child = nullptr;
    int rc = pkv_request_create(parent->pool, &child);
    if (rc != PKV_OK) return rc;
    child->table = parent->table;
    child->length = parent->length;
    child->dev_dirty_from = 0;
    for (int32_t pg : child->table) ++parent->pool->refs[(size_t)pg];
    *out = child;
    return ok();
}

int pkv_pool_page_refs(const pkv_pool* p, int32_t page, int* refs) {
    if (!p || !refs) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    if (page < 0 || page >= p->pages) return fail(PKV_ERR_INVALID_ARGUMENT, "page outside the pool");
    *refs = p->refs[(size_t)page];
    return ok();
}

int pkv_workspace_size(const pkv_pool* p, int batch, int64_t max_seq_len, size_t* bytes) {
    if (!p || !bytes) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    if (batch < 0 || max_seq_len < 1) return fail(PKV_ERR_INVALID_ARGUMENT, "bad batch or length");
    if (p->host_only) return fail(PKV_ERR_NO_STORAGE, "host-only pool has no device storage");
    const int w = pkv::launch_workers(p->workers, batch, p->dec_heads, pkv::attended_len(max_seq_len, p->window), p->kv_shift);
    *bytes = pkv::workspace_layout(batch, p->dec_heads, p->head_dim, w, p->dec_group).total;
    return ok();
}

int pkv_paged_decode_attention(pkv_pool* p, int layer, int batch, const float* q,
                               const void* k_new, const void* v_new, const int32_t* page_tables,
                               int max_pages, const int32_t* seq_lens, int64_t max_seq_len,
                               float* out, void* workspace, size_t workspace_bytes, void* stream) {
    if (!p) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pool");
    if (layer < 0 || layer >= p->layers)
        return fail(PKV_ERR_INVALID_ARGUMENT, "layer %d outside [0, %d)", layer, p->layers);
    if (batch < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "negative batch");
    if (batch > 0) {
        if (!q || !k_new || !v_new || !page_tables || !seq_lens || !out || !workspace)
            return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pointer");
        if (max_pages < 1 || max_seq_len < 1)
            return fail(PKV_ERR_INVALID_ARGUMENT, "max_pages and max_seq_len must be >= 1");
        if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
            return fail(PKV_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
        if (int rc = check_rows_aligned(p, q, 4, k_new, v_new, out); rc != PKV_OK) return rc;
    }
    if (p->host_only) return fail(PKV_ERR_NO_STORAGE, "host-only pool has no device storage");
    if (batch == 0) return ok();
    const int w = pkv::launch_workers(p->workers, batch, p->dec_heads, pkv::attended_len(max_seq_len, p->window), p->kv_shift);
    const size_t need = pkv::workspace_layout(batch, p->dec_heads, p->head_dim, w, p->dec_group).total;
    if (workspace_bytes < need)
        return fail(PKV_ERR_INVALID_ARGUMENT, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    need);
    int rc = check_device(p);
    if (rc != PKV_OK) return rc;
    pkv::DecodeArgs a{};
    a.dtype = p->dtype;
    a.B = batch;
    a.H = p->dec_heads;
    a.G = p->dec_group;
    a.kv_shift = p->kv_shift;
    a.window = p->window;
    a.tmap_k = p->tensor_cores ? &p->tmap_k[(size_t)layer] : nullptr;
    a.tmap_v = p->tensor_cores ? &p->tmap_v[(size_t)layer] : nullptr;
    a.D = p->head_dim;
    a.P = p->page_size;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    void *kp, *vp;
    pkv_pool_kv_ptr(p, layer, &kp, &vp);
    a.k_pages = kp;
    a.v_pages = vp;
    a.n_pages = p->pages;
    a.tables = page_tables;
    a.max_pages = max_pages;
    a.seq_lens = seq_lens;
    a.single_t = 0;
    a.max_seq_len = max_seq_len;
    a.out = out;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.workers = w;
    a.dev_error = p->dev_error;
    a.ev_before = p->ev_before;
    a.ev_after = p->ev_after;
    take_wait_fault(p, &a);
    cudaError_t e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return ok();
}

int pkv_prefill_workspace_size(const pkv_pool* p, int batch, int64_t total_new, size_t* bytes) {
    if (!p || !bytes) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    if (batch < 0 || total_new < 0)
        return fail(PKV_ERR_INVALID_ARGUMENT, "negative batch or token count");
    *bytes = (batch == 0 || total_new == 0) ? 0
             : tensor_prefill(p)            ? pkv::prefill_workspace_bytes(batch, p->group, total_new)
                                            : lanes_bytes(p, batch, total_new);
    return ok();
}

int pkv_paged_prefill(pkv_pool* p, int layer, int batch, int64_t total_new, const void* q,
                      const void* k_new, const void* v_new, const int32_t* cu_new,
                      const int32_t* page_tables, int max_pages, const int32_t* seq_lens,
                      float* out, void* workspace, size_t workspace_bytes, void* stream) {
    if (!p) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pool");
    if (p->host_only) return fail(PKV_ERR_NO_STORAGE, "host-only pool has no device storage");
    if (layer < 0 || layer >= p->layers)
        return fail(PKV_ERR_INVALID_ARGUMENT, "layer %d outside [0, %d)", layer, p->layers);
    if (batch < 0 || total_new < 0)
        return fail(PKV_ERR_INVALID_ARGUMENT, "negative batch or token count");
    const bool tc = tensor_prefill(p);
    if (tc && batch > pkv::prefill_max_batch())
        return fail(PKV_ERR_INVALID_ARGUMENT, "batch %d above %d", batch, pkv::prefill_max_batch());
    if (total_new > INT32_MAX) return fail(PKV_ERR_INVALID_ARGUMENT, "more than 2^31 - 1 tokens");
    if (batch == 0 || total_new == 0) return ok();
    if (!q || !k_new || !v_new || !cu_new || !page_tables || !seq_lens || !out || !workspace)
        return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pointer");
    if (max_pages < 1) return fail(PKV_ERR_INVALID_ARGUMENT, "max_pages must be >= 1");
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return fail(PKV_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
    if (int rc = check_rows_aligned(p, q, elem_bytes(p->dtype), k_new, v_new, out); rc != PKV_OK)
        return rc;
    if (tc && pkv::prefill_max_tiles(batch, p->group, total_new) * p->heads > INT32_MAX)
        return fail(PKV_ERR_INVALID_ARGUMENT, "%lld tokens need more CTAs than one launch holds",
                    (long long)total_new);
    const size_t need =
        tc ? pkv::prefill_workspace_bytes(batch, p->group, total_new) : lanes_bytes(p, batch, total_new);
    if (workspace_bytes < need)
        return fail(PKV_ERR_INVALID_ARGUMENT, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    need);
    int rc = check_device(p);
    if (rc != PKV_OK) return rc;
    if (!tc) {
        pkv::PrefillLanesArgs a = lanes_args(p, layer, batch, total_new);
        a.q = q;
        a.k_new = k_new;
        a.v_new = v_new;
        a.cu_new = cu_new;
        a.seq_lens = seq_lens;
        a.tables = page_tables;
        a.max_pages = max_pages;
        a.out = out;
        a.workspace = workspace;
        a.workspace_bytes = workspace_bytes;
        cudaError_t e = pkv::launch_prefill_lanes(a, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
        return ok();
    }
    pkv::PrefillArgs a{};
    a.B = batch;
    a.H = p->heads;
    a.G = p->group;
    a.D = p->head_dim;
    a.P = p->page_size;
    a.window = p->window;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    void *kp, *vp;
    pkv_pool_kv_ptr(p, layer, &kp, &vp);
    a.k_pages = kp;
    a.v_pages = vp;
    a.n_pages = p->pages;
    a.cu_new = cu_new;
    a.seq_lens = seq_lens;
    a.tables = page_tables;
    a.max_pages = max_pages;
    a.total_new = total_new;
    a.out = out;
    a.workspace = workspace;
    a.dev_error = p->dev_error;
    a.ev_before = p->ev_before;
    a.ev_after = p->ev_after;
    a.tmap_k = &p->tmap_k[(size_t)layer];
    a.tmap_v = &p->tmap_v[(size_t)layer];
    cudaError_t e = pkv::launch_prefill(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return ok();
}

}  // extern "C"

namespace {

// Scratch of a shared-prefix call: the decode workspace, then the prefix partials.
struct SharedLayout {
    size_t decode, pre_ml, pre_o, total;
    pkv::SharedPrefixPlan plan;
};

SharedLayout shared_layout(const pkv_pool* p, int batch, int64_t max_seq_len, int64_t shared_len) {
    SharedLayout L{};
    const int w = pkv::launch_workers(p->workers, batch, p->dec_heads,
                                      pkv::attended_len(max_seq_len, p->window), p->kv_shift);
    L.decode = (pkv::workspace_layout(batch, p->dec_heads, p->head_dim, w, p->dec_group).total + 255) /
               256 * 256;
    L.plan = pkv::shared_prefix_plan(batch, p->heads, p->group, shared_len, p->sms);
    const size_t rows = (size_t)L.plan.splits * batch * p->query_heads;
    L.pre_ml = L.decode;
    L.pre_o = L.pre_ml + (rows * sizeof(float2) + 255) / 256 * 256;
    L.total = L.pre_o + rows * p->head_dim * sizeof(float);
    return L;
}

int check_shared(const pkv_pool* p, int64_t max_seq_len, int64_t shared_len) {
    if (p->host_only) return fail(PKV_ERR_NO_STORAGE, "host-only pool has no device storage");
    if (shared_len < 0 || shared_len % p->page_size != 0)
        return fail(PKV_ERR_INVALID_ARGUMENT, "shared_len %lld is not a multiple of page_size %d",
                    (long long)shared_len, p->page_size);
    if (shared_len > 0 && shared_len >= max_seq_len)
        return fail(PKV_ERR_INVALID_ARGUMENT, "shared_len %lld leaves no position of a request's own",
                    (long long)shared_len);
    return PKV_OK;
}

// The pool has the shared-prefix kernel (bf16, head_dim 64 or 128); other pools take
// the plain batched call, each request over its own pages.
bool shared_kernel(const pkv_pool* p) {
    return p->tmaps && pkv::shared_prefix_supported(p->dtype, p->head_dim, p->group);
}

}  // namespace

extern "C" {

int pkv_workspace_size_shared(const pkv_pool* p, int batch, int64_t max_seq_len, int64_t shared_len,
                              size_t* bytes) {
    if (!p || !bytes) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL argument");
    if (batch < 0 || max_seq_len < 1) return fail(PKV_ERR_INVALID_ARGUMENT, "bad batch or length");
    int rc = check_shared(p, max_seq_len, shared_len);
    if (rc != PKV_OK) return rc;
    if (shared_len == 0 || !shared_kernel(p)) return pkv_workspace_size(p, batch, max_seq_len, bytes);
    *bytes = batch == 0 ? 0 : shared_layout(p, batch, max_seq_len, shared_len).total;
    return ok();
}

int pkv_paged_decode_attention_shared(pkv_pool* p, int layer, int batch, const float* q,
                                      const void* k_new, const void* v_new,
                                      const int32_t* page_tables, int max_pages,
                                      const int32_t* seq_lens, int64_t max_seq_len,
                                      int64_t shared_len, float* out, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    if (!p) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pool");
    if (max_seq_len < 1) return fail(PKV_ERR_INVALID_ARGUMENT, "max_seq_len must be >= 1");
    int rc = check_shared(p, max_seq_len, shared_len);
    if (rc != PKV_OK) return rc;
    if (shared_len == 0 || !shared_kernel(p))
        return pkv_paged_decode_attention(p, layer, batch, q, k_new, v_new, page_tables, max_pages,
                                          seq_lens, max_seq_len, out, workspace, workspace_bytes,
                                          stream);
    if (shared_len / p->page_size > max_pages)
        return fail(PKV_ERR_INVALID_ARGUMENT, "shared_len %lld needs more than max_pages pages",
                    (long long)shared_len);
    pkv::DecodeArgs a{};
    size_t need = 0;
    rc = pkv::prepare_batched(p, layer, batch, q, k_new, v_new, page_tables, max_pages, seq_lens,
                              max_seq_len, out, &a, &need);
    if (rc != PKV_OK || a.B == 0) return rc;
    if (!workspace) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL workspace");
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return fail(PKV_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
    const SharedLayout L = shared_layout(p, batch, max_seq_len, shared_len);
    if (workspace_bytes < L.total)
        return fail(PKV_ERR_INVALID_ARGUMENT, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    L.total);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    pkv::SharedPrefixArgs sp{};
    sp.B = batch;
    sp.H = p->heads;
    sp.G = p->group;
    sp.D = p->head_dim;
    sp.P = p->page_size;
    sp.max_pages = max_pages;
    sp.window = p->window;
    sp.n_pages = p->pages;
    sp.q = q;
    sp.tables = page_tables;
    sp.seq_lens = seq_lens;
    sp.shared_len = shared_len;
    sp.plan = L.plan;
    sp.pre_ml = reinterpret_cast<float2*>(ws + L.pre_ml);
    sp.pre_o = reinterpret_cast<float*>(ws + L.pre_o);
    sp.dev_error = p->dev_error;
    sp.tmap_k = &p->tmap_k[(size_t)layer];
    sp.tmap_v = &p->tmap_v[(size_t)layer];
    a.workspace = workspace;
    a.workspace_bytes = L.decode;
    a.key_start = shared_len;
    a.pre_ml = sp.pre_ml;
    a.pre_o = sp.pre_o;
    a.pre_splits = L.plan.splits;
    a.pre_stride = (int64_t)batch * p->query_heads;
    a.before_split = pkv::launch_shared_prefix_hook;
    a.before_split_ctx = &sp;
    cudaError_t e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "shared-prefix decode launch");
    return ok();
}

int pkv_pool_set_timing_events(pkv_pool* p, void* before, void* after) {
    if (!p) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pool");
    if ((before == nullptr) != (after == nullptr))
        return fail(PKV_ERR_INVALID_ARGUMENT, "give both events or neither");
    p->ev_before = static_cast<cudaEvent_t>(before);
    p->ev_after = static_cast<cudaEvent_t>(after);
    return ok();
}

int pkv_pool_inject_fault(pkv_pool* p, int kind, int64_t arg, uint64_t wait_limit_ns) {
    if (!p) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pool");
    switch (kind) {
        case PKV_INJECT_NONE:
            p->inject_lease = 0;
            p->inject_layer = -1;
            p->inject_worker = -1;
            return ok();
        case PKV_INJECT_LEASE:
            if (arg < 1) return fail(PKV_ERR_INVALID_ARGUMENT, "lease count must be >= 1");
            p->inject_lease = arg;
            return ok();
        case PKV_INJECT_LAYER:
            if (arg < 0 || arg >= p->layers)
                return fail(PKV_ERR_INVALID_ARGUMENT, "layer %lld outside [0, %d)", (long long)arg,
                            p->layers);
            p->inject_layer = (int)arg;
            return ok();
        case PKV_INJECT_DEVICE_WAIT:
            if (p->host_only) return fail(PKV_ERR_NO_STORAGE, "host-only pool has no device storage");
            if (arg < 0 || arg >= p->workers)
                return fail(PKV_ERR_INVALID_ARGUMENT, "worker %lld outside [0, %d)", (long long)arg,
                            p->workers);
            if (wait_limit_ns < 1000000ull || wait_limit_ns > 4000000000ull)
                return fail(PKV_ERR_INVALID_ARGUMENT, "wait limit must be within [1 ms, 4 s]");
            p->inject_worker = (int)arg;
            p->inject_wait_ns = wait_limit_ns;
            return ok();
        default:
            return fail(PKV_ERR_INVALID_ARGUMENT, "unknown fault kind %d", kind);
    }
}

int pkv_check_device_status(pkv_pool* p, uint32_t* bits) {
    if (!p) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pool");
    if (bits) *bits = 0;
    if (p->host_only) return ok();
    int rc = check_device(p);
    if (rc != PKV_OK) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned word = 0;
    if ((e = cudaMemcpy(&word, p->dev_error, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "read device error word");
    if (word != 0 && (e = cudaMemset(p->dev_error, 0, sizeof word)) != cudaSuccess)
        return cuda_fail(e, "clear device error word");
    if (bits) *bits = word;
    if (word != 0) return fail(PKV_ERR_DEVICE_CHECK, "device error bits 0x%x", word);
    return ok();
}

}  // extern "C"

namespace pkv {

int record_error(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int prepare_batched(pkv_pool* p, int layer, int batch, const float* q, const void* k_new,
                    const void* v_new, const int32_t* page_tables, int max_pages,
                    const int32_t* seq_lens, int64_t max_seq_len, float* out, DecodeArgs* a,
                    size_t* workspace_bytes) {
    if (!p) return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pool");
    if (layer < 0 || layer >= p->layers)
        return fail(PKV_ERR_INVALID_ARGUMENT, "layer %d outside [0, %d)", layer, p->layers);
    if (batch < 0) return fail(PKV_ERR_INVALID_ARGUMENT, "negative batch");
    *a = DecodeArgs{};
    *workspace_bytes = 0;
    if (batch > 0) {
        if (!q || !k_new || !v_new || !page_tables || !seq_lens || !out)
            return fail(PKV_ERR_INVALID_ARGUMENT, "NULL pointer");
        if (max_pages < 1 || max_seq_len < 1)
            return fail(PKV_ERR_INVALID_ARGUMENT, "max_pages and max_seq_len must be >= 1");
        const int rc = check_rows_aligned(p, q, 4, k_new, v_new, out);
        if (rc != PKV_OK) return rc;
    }
    if (p->host_only) return fail(PKV_ERR_NO_STORAGE, "host-only pool has no device storage");
    if (batch == 0) return ok();
    int rc = check_device(p);
    if (rc != PKV_OK) return rc;
    const int w = launch_workers(p->workers, batch, p->dec_heads, attended_len(max_seq_len, p->window), p->kv_shift);
    *workspace_bytes = workspace_layout(batch, p->dec_heads, p->head_dim, w, p->dec_group).total;
    a->dtype = p->dtype;
    a->B = batch;
    a->H = p->dec_heads;
    a->G = p->dec_group;
    a->kv_shift = p->kv_shift;
    a->window = p->window;
    a->tmap_k = p->tensor_cores ? &p->tmap_k[(size_t)layer] : nullptr;
    a->tmap_v = p->tensor_cores ? &p->tmap_v[(size_t)layer] : nullptr;
    a->D = p->head_dim;
    a->P = p->page_size;
    a->q = q;
    a->k_new = k_new;
    a->v_new = v_new;
    a->k_pages = static_cast<char*>(p->k_base) + p->layer_bytes * (size_t)layer;
    a->v_pages = static_cast<char*>(p->v_base) + p->layer_bytes * (size_t)layer;
    a->n_pages = p->pages;
    a->tables = page_tables;
    a->max_pages = max_pages;
    a->seq_lens = seq_lens;
    a->max_seq_len = max_seq_len;
    a->out = out;
    a->workers = w;
    a->dev_error = p->dev_error;
    a->ev_before = p->ev_before;
    a->ev_after = p->ev_after;
    take_wait_fault(p, a);
    return ok();
}

}  // namespace pkv
