// Paged decode attention kernels for sm_103a.
//
// What is computed ("Incremental Serving", sections "Request flow" and "Paged
// KV-cache layout"; "38 · Cached generation", function incremental_mixture):
// for each request b and head h, the new key/value row is stored at logical
// position t_b - 1 of the paged pools, then the single query row attends over
// the t_b keys found through the request's page table:
//     out = sum_j softmax_j(q . K_j / sqrt(d_h)) V_j.
//
// Work decomposition.  Every (request, head) lane is cut into tiles of 16 key
// rows (a tile never straddles a page because page sizes are multiples of 16).
// All tiles of all lanes are laid end to end, lane after lane, and the
// resulting index range is cut into W equal contiguous pieces, one per worker.
// A worker is one warp of a persistent grid that fills the GPU once, so the
// load is balanced to within one tile whatever the mix of lengths.  A worker
// streams its tiles through its own ring of shared-memory stages: one lane
// issues 1-D bulk asynchronous copies (cp.async.bulk, the TMA engine without a
// tensor map) of the tile's K rows and V rows — each a contiguous
// 16 * d_h * element-size block of one (page, head) — and an mbarrier per
// stage tracks the bytes.  The warp runs an online softmax in fp32 in log2
// units (exp2 of q'.k with q' = q * log2(e) / sqrt(d_h)), with warp-shuffle
// reductions for the dot products and the row maximum.
//
// A lane that a single worker covers completely is finished by that worker.
// Otherwise each worker covering part of it writes a partial (m, l, o[d_h])
// into slot lane + worker of the workspace and bumps the lane's counter; the
// last of the lane's workers to arrive merges the partials:
//     out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s.
// Tile x belongs to worker floor(((x + 1) W - 1) / T), the inverse of
// begin(w) = floor(w T / W); slots never collide across lanes because the
// first worker of lane i + 1 is at least the last worker of lane i.  A small
// plan kernel runs first (lengths, tile prefix, worker table, counters); the
// split kernel is launched as its programmatic dependent.
//
// The append is fused into the worker that owns the lane's last tile: once that
// tile's copy has landed it overwrites row t_b - 1 of the staged tile with
// k_new / v_new (the pool may still hold stale bytes there) and stores the row
// into the page.  No other worker reads that tile, so nothing races.
//
// Faults are not raised by trapping: bad lengths and page ids, and waits that
// run out, set bits of a device error word and the offending work is skipped.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <cstring>

#include "pkv.h"
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

// ------------------------------------------------------- element access --

template <int BYTES>
struct VecBits;
template <>
struct VecBits<16> { using type = uint4; };
template <>
struct VecBits<8> { using type = uint2; };
template <>
struct VecBits<4> { using type = uint32_t; };

template <typename T>
struct Storage;

template <>
struct Storage<float> {
    // N elements -> N/2 float pairs
    template <int N>
    __device__ __forceinline__ static void to_float2(const void* bits, float2* out) {
        const float2* f = reinterpret_cast<const float2*>(bits);
#pragma unroll
        for (int i = 0; i < N / 2; ++i) out[i] = f[i];
    }
};

template <>
struct Storage<__nv_bfloat16> {
    // bf16 is the upper half of an fp32: element 2i is the low half of word i.
    template <int N>
    __device__ __forceinline__ static void to_float2(const void* bits, float2* out) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(bits);
#pragma unroll
        for (int i = 0; i < N / 2; ++i)
            out[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    }
};

#ifndef PKV_SM_SMEM_BUDGET
#define PKV_SM_SMEM_BUDGET 131072  // stage-ring bytes of one split CTA (one CTA per SM)
#endif
#ifndef PKV_SM_SMEM_BUDGET_GROUPED
// fp32 with several query heads per KV head: each tile carries G times the
// arithmetic, and a larger ring buys more warps to hide it (bf16 tiles are half
// the size and already get eight warps)
#define PKV_SM_SMEM_BUDGET_GROUPED 196608
#endif

// Warp geometry of one 16-row tile for storage type T and head width D, and
// the CTA shape.  TPR lanes share one row (VEC elements each, one 16-byte
// vector at most); RPI rows are read per warp step.  After the dot products, a
// transposed shuffle reduction leaves lane l holding the full score of row
// ((l % TPR) >> 1) * RPI + l / TPR (lanes l and l ^ 1 hold the same row when
// TPR >= 2), so each lane takes one exp2 per tile.  One CTA per SM: WARPS
// workers, each with STAGES tiles in flight, within the shared-memory budget.
template <typename T, int D, int G = 1>
struct Geo {
    static constexpr int BUDGET =
        (G > 1 && sizeof(T) == 4) ? PKV_SM_SMEM_BUDGET_GROUPED : PKV_SM_SMEM_BUDGET;
    static constexpr int ES = sizeof(T);
    static constexpr int VEC = (16 / ES) < D ? (16 / ES) : D;  // elements per lane vector
    static constexpr int VBYTES = VEC * ES;                    // 16, 8 or 4
    static constexpr int TPR = D / VEC;                        // lanes sharing one row
    static constexpr int RPI = 32 / TPR;                       // rows per warp step
    static constexpr int ITERS = TPR >= 2 ? TPR / 2 : 1;       // warp steps per tile
    static constexpr int DUP = TPR >= 2 ? 2 : 1;               // lanes holding each score
    static constexpr int HALVING_ROUNDS = ITERS == 16 ? 4 : ITERS == 8 ? 3 : ITERS == 4 ? 2
                                        : ITERS == 2 ? 1 : 0;  // log2(ITERS)
    static constexpr int TILE_BYTES = kTile * D * ES;          // K (or V) rows of one tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int STAGES_AT_WARPS = BUDGET / (kSplitWarps * STAGE_BYTES);
    static constexpr int WARPS = STAGES_AT_WARPS >= 2
        ? kSplitWarps : (BUDGET / (2 * STAGE_BYTES) > 0 ? BUDGET / (2 * STAGE_BYTES) : 1);
    static constexpr int STAGES_RAW = BUDGET / (WARPS * STAGE_BYTES);
    static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
    static constexpr int WARP_SMEM = STAGES * STAGE_BYTES;
    // per warp: stage buffers, then per stage an mbarrier (8 B) and the staged page id (4 B)
    static constexpr int CTA_SMEM = WARPS * (WARP_SMEM + STAGES * 12);
    static constexpr int DPL = D >= 32 ? D / 32 : 1;           // features per lane when merging
    // cluster lanes (a single request): after the rings, 8 lane mbarriers and a
    // partial slot (max, sum, o[D]) for each worker of up to 8 CTAs
    static constexpr int CLU_OFF = (CTA_SMEM + 15) / 16 * 16;
    static constexpr int LANE_SLOTS = 8 * WARPS;
    static constexpr int CLU_BYTES = 64 + LANE_SLOTS * (D + 2) * 4;
    static constexpr bool CLUSTER_LANES =
        (WARPS == 4 || WARPS == 8) && CLU_OFF + CLU_BYTES <= 227 * 1024;
    static_assert(D % VEC == 0 && VEC % 2 == 0, "unsupported head width");
    static_assert(TPR <= 32 && (TPR & (TPR - 1)) == 0, "unsupported head width");
    static_assert(RPI * ITERS >= kTile, "a warp step pattern must cover the tile");
    static_assert(TILE_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");
    static_assert(WARPS >= 1 && WARPS <= 32 && CTA_SMEM <= 227 * 1024, "CTA does not fit an SM");
};

constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s per bounded wait
constexpr int kEarlyTiles = 4;    // tiles a single-request worker fetches into L2 before its wait

// ----------------------------------------------------------- parameters --

struct KParams {
    const float* q;
    const void* k_new;
    const void* v_new;
    void* k_pages;
    void* v_pages;
    int64_t n_pages;
    const int32_t* tables;
    int max_pages;
    const int32_t* table_rows;  // nullptr: request b reads table row b; else row table_rows[b]
                                // (CUDA-core kernel only)
    bool allow_empty;           // seq_len 0: a request with no work, not an error
    const int32_t* seq_lens;    // nullptr: one request of length single_t
    int64_t single_t;
    int64_t max_seq_len;
    int B, H, P, tiles_per_page;
    // lane head h reads KV head h >> kv_shift of the pool's H >> kv_shift: a pool with
    // more query heads per KV head than a lane takes (8; 16 on the tensor-core kernel)
    // runs as 2^kv_shift lanes per KV head
    int kv_shift;
    int64_t window;             // attend to the last `window` positions (0: all)
    float qscale;               // log2(e) / sqrt(D)
    float* out;
    int64_t* req_prefix;        // [B + 1] tiles-per-lane prefix (plan kernel)
    int32_t* worker_req;        // [W] request of each worker's first tile (plan kernel)
    unsigned long long* lane_cnt;  // [B * H] partials deposited per split lane
    uint32_t epoch;             // 0: counters zeroed by the plan kernel; else the call's epoch
    float2* part_ml;
    float* part_o;
    int W;
    unsigned* err;
    // shared prefix: positions below key_start were attended by the prefix kernel,
    // whose pre_splits partials per query row (stride pre_stride rows) join the merge
    int64_t key_start;
    const float2* pre_ml;
    const float* pre_o;
    int pre_splits;
    int64_t pre_stride;
    uint64_t wait_ns;           // each bounded wait gives up after this long
    int inject_worker;          // failure injection: 0 off; else worker inject_worker - 1 arms
                                // its first stage without issuing the copy
    // cluster lanes (a single request on the CUDA-core kernel, multi-head pools):
    // > 0: each lane's tiles are split over lane_workers consecutive workers (of this
    // CTA when fewer than a CTA's warps, else of the lane_workers / WARPS CTAs of one
    // cluster), which merge through the lead CTA's shared memory instead of global
    // partials and counters; 0: off
    int lane_workers;
    // block lanes (prefill of fp32 pools on the tensor-core kernel's table-row form):
    // decode request x is a block of blk_ntok[x] consecutive chunk tokens starting at
    // chunk row blk_tok0[x]; lane row g is token g / blk_gp of the block and query
    // head h * blk_gp + g % blk_gp of the pool, attending positions up to its own
    // t - (ntok - 1 - g / blk_gp); nullptr: one query row per (request, query head)
    const int32_t* blk_tok0;
    const int32_t* blk_ntok;
    int blk_gp;                 // the pool's query heads per KV head
    int blk_hq;                 // the pool's query heads
};

__device__ __forceinline__ int64_t seq_len_at(const KParams& p, int b) {
    return p.seq_lens == nullptr ? p.single_t : (int64_t)__ldg(p.seq_lens + b);
}

// Block lanes: the q / out row of lane row g of decode request x, KV head h, or -1
// for a row past the block's tokens.
__device__ __forceinline__ int64_t block_row(const KParams& p, int x, int h, int g) {
    const int r = g / p.blk_gp;
    if (r >= __ldg(p.blk_ntok + x)) return -1;
    return ((int64_t)__ldg(p.blk_tok0 + x) + r) * p.blk_hq + (int64_t)h * p.blk_gp + g % p.blk_gp;
}


// Row block [page][KV head hk] of the K / V pools, and row of k_new / v_new for KV
// head hk of request b.  Lane head h of a request reads KV head h >> kv_shift.
__device__ __forceinline__ int64_t kv_block(const KParams& p, int64_t page, int hk) {
    return page * (p.H >> p.kv_shift) + hk;
}

__device__ __forceinline__ int64_t kv_new_row(const KParams& p, int b, int hk) {
    return (int64_t)b * (p.H >> p.kv_shift) + hk;
}

// First position this kernel reads for a query at retained length t: the
// window's first position, or the first position after a shared prefix that
// the prefix kernel attends.
__device__ __forceinline__ int64_t window_start(const KParams& p, int64_t t) {
    const int64_t w = (p.window > 0 && t > p.window) ? t - p.window : 0;
    return w > p.key_start ? w : p.key_start;
}

// Tiles a lane of retained length t reads: from the tile holding the window's
// first position to the tile holding position t - 1.
__device__ __forceinline__ int64_t lane_tiles(const KParams& p, int64_t t) {
    return (t + kTile - 1) / kTile - window_start(p, t) / kTile;
}

// Tiles-per-lane prefix over requests: closed form for a single request (no
// dependence on the plan kernel), else the plan kernel's table.
__device__ __forceinline__ int64_t req_prefix_at(const KParams& p, int b) {
    if (p.seq_lens == nullptr) return b == 0 ? 0 : lane_tiles(p, p.single_t);
    return __ldg(p.req_prefix + b);
}

// ----------------------------------------------------------- plan kernel --

constexpr int kPlanThreads = 1024;
constexpr int kPlanSmemRequests = 2048;   // prefix kept in shared memory up to this batch

// Validates lengths, writes the per-request tile prefix and the first request
// of every worker, and zeroes the per-lane partial counters.  One CTA.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const KParams p) {
    pdl_launch_dependents();   // the split grid may launch now; it waits for our writes
    __shared__ int64_t warp_sums[kPlanThreads / 32];
    __shared__ int64_t carry_s;
    __shared__ int64_t pre_s[kPlanSmemRequests + 1];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const bool in_smem = p.B <= kPlanSmemRequests;
    if (tid == 0) carry_s = 0;
    for (int64_t i = tid; i < (int64_t)p.B * p.H; i += kPlanThreads) p.lane_cnt[i] = 0ull;
    __syncthreads();
    for (int base = 0; base < p.B; base += kPlanThreads) {
        const int i = base + tid;
        int64_t n = 0;
        if (i < p.B) {
            const int64_t t = seq_len_at(p, i);
            const int64_t pages = (t + p.P - 1) / p.P;
            if (t == 0 && p.allow_empty) {
                // no work for this request
            } else if (t < 1 || t > p.max_seq_len || pages > p.max_pages || t <= p.key_start) {
                atomicOr(p.err, PKV_DEVERR_SEQ_LEN);
            } else {
                n = lane_tiles(p, t);
            }
        }
        int64_t incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_sums[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int64_t s = warp_sums[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += y;
            }
            warp_sums[lane] = s;   // inclusive over warps
        }
        __syncthreads();
        const int64_t carry = carry_s;
        const int64_t before = (wid > 0 ? warp_sums[wid - 1] : 0) + incl - n;
        if (i < p.B) {
            p.req_prefix[i] = carry + before;
            if (in_smem) pre_s[i] = carry + before;
        }
        __syncthreads();
        if (tid == 0) carry_s = carry + warp_sums[kPlanThreads / 32 - 1];
        __syncthreads();
    }
    const int64_t total = carry_s;
    if (tid == 0) {
        p.req_prefix[p.B] = total;
        if (in_smem) pre_s[p.B] = total;
    }
    __syncthreads();
    // ranges partition the KV lanes' tiles; worker w takes range w >> kv_shift
    const int Hk = p.H >> p.kv_shift, R = p.W >> p.kv_shift;
    const int64_t T = (int64_t)Hk * total;
    const int64_t* pre = in_smem ? pre_s : p.req_prefix;
    for (int w = tid; w < p.W; w += kPlanThreads) {
        const int64_t x = ((int64_t)(w >> p.kv_shift) * T) / R;
        int lo = 0, hi = p.B - 1;   // largest b with Hk * prefix[b] <= x
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)Hk * pre[mid] <= x) lo = mid; else hi = mid - 1;
        }
        p.worker_req[w] = lo;
    }
    // Launched as a dependent of the shared-prefix kernel (which needs no plan), the
    // plan runs beside it but completes only after it: whatever waits for the plan
    // then also sees the prefix kernel's partials.  After a plain launch this returns
    // at once.
    pdl_wait_primary();
}

// The plan kernel, then (shared-prefix calls) the prefix kernel.  With a prefix
// kernel the order is reversed: the prefix kernel first, and the plan as its
// dependent, which runs beside it.
static cudaError_t launch_plan(const DecodeArgs& a, const KParams& p, cudaStream_t stream) {
    if (a.before_split == nullptr) {
        plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
        return cudaGetLastError();
    }
    cudaError_t e = a.before_split(a.before_split_ctx, stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, plan_kernel, p);
}

// ---------------------------------------------------------- split kernel --

// Position of a worker inside the flattened (request, KV head, tile) sequence,
// with the tile's page-table index and first slot tracked incrementally.
struct Cursor {
    int b, h;          // request, KV head
    int tile;          // tile within the lane (0 .. n-1)
    int n;             // tiles of this lane
    int tile0;         // position / 16 of the lane's tile 0 (the window's first tile)
    int page_idx;      // logical page of the tile
    int slot0;         // first slot of the tile within its page
    int64_t first;     // flattened index of tile 0 of KV head 0 of request b
};

// Page index and slot of the lane's tile `tile`.
__device__ __forceinline__ void cursor_place(Cursor& c, const KParams& p) {
    const int abs = c.tile0 + c.tile;
    c.page_idx = abs / p.tiles_per_page;
    c.slot0 = (abs - c.page_idx * p.tiles_per_page) * kTile;
}

__device__ __forceinline__ void cursor_advance(Cursor& c, const KParams& p) {
    ++c.tile;
    c.slot0 += kTile;
    if (c.slot0 == p.P) {
        c.slot0 = 0;
        ++c.page_idx;
    }
    if (c.tile < c.n) return;
    c.tile = 0;
    if (++c.h < (p.H >> p.kv_shift)) {
        cursor_place(c, p);
        return;
    }
    c.h = 0;
    // next request with at least one tile
    int64_t pre = req_prefix_at(p, c.b + 1);
    while (c.b + 1 < p.B) {
        ++c.b;
        const int64_t nxt = req_prefix_at(p, c.b + 1);
        if (nxt > pre) {
            c.n = (int)(nxt - pre);
            c.first = (int64_t)(p.H >> p.kv_shift) * pre;
            c.tile0 = (int)(window_start(p, seq_len_at(p, c.b)) / kTile);
            cursor_place(c, p);
            return;
        }
        pre = nxt;
    }
    c.b = p.B;   // past the end; never dereferenced
}

// Release / acquire fence at GPU scope: with a relaxed atomic on the lane counter
// it orders a worker's partial before its count (writer) and every counted
// partial before the merge's reads (the last arriver).
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Worker that owns flattened tile x: the inverse of begin(w) = floor(w T / W).
__device__ __forceinline__ int64_t worker_of(int64_t x, int64_t T, int W) {
    return ((x + 1) * W - 1) / T;
}

// Combine the partials of query g of lane `lane_id` into out.  The lane's KV lane
// K (request b, KV head hk: K = b * (H >> kv_shift) + hk) has its tiles in ranges
// r_lo..r_hi (those owning at least one tile); sub-lane `sub` of range r wrote its
// partial to slot ((K + r) << kv_shift) | sub.  In a shared-prefix call (the
// combine kernel) the prefix kernel's pre_splits partials of the query row follow
// as partials cnt .. cnt + pre_splits - 1.
// One warp: lane j takes partials j, j + 32, ... for the maximum and the weights
// 2^(m_w - M), each (max, sum) loaded once; lane l sums features l * DPL .. of
// every partial's o vector, each weight broadcast by shuffle.  The o vectors are
// read CJ partials at a time with every load issued before any is used, and the
// first CJ together with the (max, sum) pairs, so a merge of up to CJ partials
// (32 at head width 64) costs one L2 round trip.  Partials are read from L2
// (other SMs wrote them during this kernel).
template <int D, int DPL, int G>
__device__ __forceinline__ void merge_query(const KParams& p, int64_t lane_id, int g, int64_t K,
                                            int sub, int64_t r_lo, int64_t r_hi, int64_t T_all,
                                            int lane) {
    constexpr int CJ = 64 / DPL < 32 ? 64 / DPL : 32;    // o vectors in flight (<= 64 floats)
    const int R = p.W >> p.kv_shift;
    auto owns_tiles = [&](int64_t r) { return (r * T_all) / R != ((r + 1) * T_all) / R; };
    auto slot_of = [&](int64_t r) { return ((K + r) << p.kv_shift) | sub; };
    const int cw = (int)(r_hi - r_lo + 1);
    const int cnt = cw + p.pre_splits;
    const int64_t row = lane_id * G + g;                  // query row (request, query head)
    const bool has_features = lane * DPL < D;
    // (max, sum) of partial j; a worker that owns no tile, or a prefix split with
    // no key of the row, contributes nothing
    auto load_ml = [&](int j) -> float2 {
        if (j < cw) {
            if (!owns_tiles(r_lo + j)) return make_float2(-INFINITY, 0.f);
            return __ldcg(&p.part_ml[slot_of(r_lo + j) * G + g]);
        }
        if (j >= cnt) return make_float2(-INFINITY, 0.f);
        const float2 ml = __ldcg(&p.pre_ml[(int64_t)(j - cw) * p.pre_stride + row]);
        return ml.y > 0.f ? ml : make_float2(-INFINITY, 0.f);
    };
    auto load_o = [&](int j, float (&v)[DPL]) {
        if (j < cnt && has_features) {
            const float* op = (j < cw ? p.part_o + (slot_of(r_lo + j) * G + g) * D
                                      : p.pre_o + ((int64_t)(j - cw) * p.pre_stride + row) * D) +
                              lane * DPL;
#pragma unroll
            for (int i = 0; i < DPL; ++i) v[i] = __ldcg(op + i);
        } else {
#pragma unroll
            for (int i = 0; i < DPL; ++i) v[i] = 0.f;
        }
    };
    const float2 ml0 = load_ml(lane);
    float v[CJ][DPL];
#pragma unroll
    for (int jj = 0; jj < CJ; ++jj) load_o(jj, v[jj]);
    float M = ml0.x;
    for (int j = 32 + lane; j < cnt; j += 32) M = fmaxf(M, load_ml(j).x);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    for (int base = 0; base < cnt; base += 32) {
        const float2 ml = base == 0 ? ml0 : load_ml(base + lane);
        const float wgt = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
        L = fmaf(ml.y, wgt, L);
        for (int c0 = 0; c0 < 32 && base + c0 < cnt; c0 += CJ) {
            if (base + c0 > 0) {
#pragma unroll
                for (int jj = 0; jj < CJ; ++jj) load_o(base + c0 + jj, v[jj]);
            }
#pragma unroll
            for (int jj = 0; jj < CJ; ++jj) {
                // partials with weight 0 (no tile, or past the lane's last) may hold
                // stale data: value dropped
                const float wj = __shfl_sync(0xffffffffu, wgt, c0 + jj);
#pragma unroll
                for (int i = 0; i < DPL; ++i)
                    acc[i] = wj != 0.f ? fmaf(wj, v[jj][i], acc[i]) : acc[i];
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (!has_features) return;
    const float inv = 1.f / L;
    float* out = p.out + row * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) out[i] = acc[i] * inv;
}

// Combine the partials of the G query rows of lane `lane_id` (G >= 2) into out,
// GB = min(G, 8) rows at a time; slots as for merge_query.
// For the maxima, sums and weights lane j takes worker slot j / GB of a chunk of
// 32 / GB slots and query row j % GB, so every row's max and sum reduce over the
// lanes of one residue class mod GB; for the o vectors lane j takes features
// j * D/32 .. of every row, each weight broadcast by shuffle.  The loads of a
// row block go out together: a few L2 round trips per lane instead of a few per
// query row, which matters because the merging warp's ring waits meanwhile.
template <int D, int G>
__device__ __forceinline__ void merge_lane(const KParams& p, int64_t lane_id, int64_t K, int sub,
                                           int64_t r_lo, int64_t r_hi, int64_t T_all, int lane) {
    constexpr int GB = G < 8 ? G : 8;    // rows merged together
    static_assert(GB >= 2 && 32 % GB == 0 && G % GB == 0 && D % 64 == 0,
                  "grouped merge: G a power of two, D 64 or 128");
    constexpr int SPC = 32 / GB;         // worker slots per chunk
    constexpr int DPL = D / 32;          // features per lane (2 or 4)
    const int R = p.W >> p.kv_shift;
    auto owns_tiles = [&](int64_t x) { return (x * T_all) / R != ((x + 1) * T_all) / R; };
    auto slot_of = [&](int64_t x) { return ((K + x) << p.kv_shift) | sub; };
    const int cnt = (int)(r_hi - r_lo + 1);
    const int r = lane % GB;             // the query row (within the block) this lane weighs
#pragma unroll 1
    for (int g0 = 0; g0 < G; g0 += GB) {
        float M = -INFINITY;
        for (int j = lane / GB; j < cnt; j += SPC)
            if (owns_tiles(r_lo + j)) M = fmaxf(M, __ldcg(&p.part_ml[slot_of(r_lo + j) * G + g0 + r]).x);
#pragma unroll
        for (int off = 16; off >= GB; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float L = 0.f;
        float acc[GB][DPL];
#pragma unroll
        for (int g = 0; g < GB; ++g)
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[g][i] = 0.f;
        for (int base = 0; base < cnt; base += SPC) {
            const int j = base + lane / GB;
            float wgt = 0.f;
            if (j < cnt && owns_tiles(r_lo + j)) {
                const float2 ml = __ldcg(&p.part_ml[slot_of(r_lo + j) * G + g0 + r]);
                wgt = exp2f(ml.x - M);
                L = fmaf(ml.y, wgt, L);
            }
            const int nj = cnt - base < SPC ? cnt - base : SPC;
#pragma unroll 1
            for (int jj = 0; jj < nj; ++jj) {
                const float* op = p.part_o + (slot_of(r_lo + base + jj) * G + g0) * D + lane * DPL;
                float v[GB][DPL];
#pragma unroll
                for (int g = 0; g < GB; ++g) {
                    if constexpr (DPL == 4) {
                        const float4 x = __ldcg(reinterpret_cast<const float4*>(op + g * D));
                        v[g][0] = x.x, v[g][1] = x.y, v[g][2] = x.z, v[g][3] = x.w;
                    } else {
                        const float2 x = __ldcg(reinterpret_cast<const float2*>(op + g * D));
                        v[g][0] = x.x, v[g][1] = x.y;
                    }
                }
#pragma unroll
                for (int g = 0; g < GB; ++g) {
                    // slots of workers that own no tile hold stale data: weight 0, value dropped
                    const float wj = __shfl_sync(0xffffffffu, wgt, jj * GB + g);
#pragma unroll
                    for (int i = 0; i < DPL; ++i)
                        acc[g][i] = wj != 0.f ? fmaf(wj, v[g][i], acc[g][i]) : acc[g][i];
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= GB; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
#pragma unroll
        for (int g = 0; g < GB; ++g) {
            const float inv = 1.f / __shfl_sync(0xffffffffu, L, g);
            int64_t orow = lane_id * G + g0 + g;
            if (p.blk_tok0 != nullptr) {   // block lanes: the row's chunk token, if any
                orow = block_row(p, (int)(lane_id / p.H), (int)(lane_id % p.H), g0 + g);
                if (orow < 0) continue;
            }
            float* out = p.out + orow * D + lane * DPL;
            if constexpr (DPL == 4) {
                *reinterpret_cast<float4*>(out) =
                    make_float4(acc[g][0] * inv, acc[g][1] * inv, acc[g][2] * inv, acc[g][3] * inv);
            } else {
                *reinterpret_cast<float2*>(out) = make_float2(acc[g][0] * inv, acc[g][1] * inv);
            }
        }
    }
}

// Shared-prefix calls: one warp per query row merges the row's worker partials
// and the prefix kernel's partials (after the split kernel, in stream order).
template <int D, int G>
__global__ void __launch_bounds__(256) combine_kernel(const KParams p) {
    constexpr int DPL = D >= 32 ? D / 32 : 1;
    const int64_t qrow = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (qrow >= (int64_t)p.B * p.H * G) return;
    const int64_t lane_id = qrow / G;
    const int g = (int)(qrow - lane_id * G);
    const int b = (int)(lane_id / p.H), h = (int)(lane_id - (int64_t)b * p.H);
    const int hk = h >> p.kv_shift, sub = h & ((1 << p.kv_shift) - 1);
    const int Hk = p.H >> p.kv_shift, R = p.W >> p.kv_shift;
    const int64_t pre_b = req_prefix_at(p, b);
    const int64_t n = req_prefix_at(p, b + 1) - pre_b;    // 0 for a request the plan rejected
    if (n <= 0) return;
    const int64_t T_all = (int64_t)Hk * req_prefix_at(p, p.B);
    const int64_t A = (int64_t)Hk * pre_b + (int64_t)hk * n;
    merge_query<D, DPL, G>(p, lane_id, g, (int64_t)b * Hk + hk, sub, worker_of(A, T_all, R),
                           worker_of(A + n - 1, T_all, R), T_all, lane);
}

// One worker (warp) of the split kernel.  A lane here is a (request, KV head)
// pair; its G query heads (grouped-query attention, G = 1 for multi-head) share
// every staged K/V tile: query head h*G + g of request b reads KV head h.  ROWS:
// request b reads page-table row p.table_rows[b] (the prefill through decode lanes);
// a separate instantiation, so the plain decode carries no extra live state.
template <typename T, int D, int G, bool ROWS = false>
__global__ void __launch_bounds__(Geo<T, D, G>::WARPS * 32, 1)
split_decode_kernel(const KParams p) {
    using Gm = Geo<T, D, G>;
    using VT = typename VecBits<Gm::VBYTES>::type;
    constexpr int NV = Gm::VEC / 2;   // float pairs per lane vector
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * Gm::WARPS + warp;
    // cluster lanes: every CTA's lane barriers are initialised before any worker of
    // the cluster can arrive on them (every thread takes part, so before any return)
    uint64_t* lane_bar = reinterpret_cast<uint64_t*>(smem + Gm::CLU_OFF);        // [8]
    float* lane_part = reinterpret_cast<float*>(smem + Gm::CLU_OFF + 64);        // [slots][D+2]
    if constexpr (Gm::CLUSTER_LANES) {
        if (p.lane_workers > 0) {
            // inside a CTA: one barrier per lane, every lane of its kw workers arrives.
            // Across a cluster: barrier 0 gathers this CTA's WARPS workers, barrier 1 (of
            // the lead CTA) the cluster's kw / WARPS CTA partials
            const uint32_t kw = (uint32_t)p.lane_workers;
            const uint32_t cnt = kw <= (uint32_t)Gm::WARPS ? 32u * kw
                                 : threadIdx.x == 1 ? 32u * (kw / Gm::WARPS) : 32u * Gm::WARPS;
            if (threadIdx.x < 8) mbar_init(&lane_bar[threadIdx.x], cnt);
            if (p.lane_workers > Gm::WARPS) {     // lanes span the CTAs of a cluster
                if (threadIdx.x == 0) fence_mbar_init();
                cluster_sync_all();
            } else {                               // lanes inside this CTA
                __syncthreads();
            }
        }
    }
    if (w >= p.W) return;

    unsigned char* ring = smem + warp * Gm::WARP_SMEM;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::WARPS * Gm::WARP_SMEM) + warp * Gm::STAGES;
    int32_t* stage_page =
        reinterpret_cast<int32_t*>(smem + Gm::WARPS * (Gm::WARP_SMEM + Gm::STAGES * 8)) +
        warp * Gm::STAGES;
    if (lane == 0) {
        for (int s = 0; s < Gm::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t policy = l2_stream_policy();

    // The plan kernel's prefix and worker table are needed now for a batch.  A
    // single request's partition is closed-form and its lane counters carry an
    // epoch, so it runs without a plan kernel; it is launched as a dependent of
    // whatever came before (the previous layer's call) and lets the next call's
    // kernel launch at once.  Either way nothing an earlier kernel may have written
    // is read before the previous grid is complete, so every such write is visible.
    const bool batched = p.seq_lens != nullptr;
    // A single request's page table is written only by copies in stream order, never
    // by a kernel, so its first entries are read (and this worker's tiles fetched into
    // L2, which changes no memory: a later write by the previous grid lands in L2
    // too) before the wait; the copies into shared memory and q come after it.
    const bool early = !batched && !ROWS;
    if (!batched) pdl_launch_dependents();
    if (!early) pdl_wait_primary();

    // this worker's tiles: range w >> kv_shift, [begin, end) of the flattened (request,
    // KV head, tile) sequence, for sub-lane w & (2^kv_shift - 1) of every KV head in it
    const int sub = (int)(w & ((1 << p.kv_shift) - 1));
    const int Hk = p.H >> p.kv_shift, R = p.W >> p.kv_shift;
    const int64_t T_all = (int64_t)Hk * req_prefix_at(p, p.B);
    const int64_t begin = ((w >> p.kv_shift) * T_all) / R;
    const int64_t end = (((w >> p.kv_shift) + 1) * T_all) / R;
    const int n_work = (int)(end - begin);
    if (n_work <= 0) {
        if (early) pdl_wait_primary();
        return;
    }

    Cursor cur;
    {
        const int b0 = batched ? __ldg(p.worker_req + w) : 0;
        const int64_t pre = req_prefix_at(p, b0);
        cur.b = b0;
        cur.n = (int)(req_prefix_at(p, b0 + 1) - pre);
        cur.first = (int64_t)Hk * pre;
        const int64_t local = begin - cur.first;
        cur.h = (int)(local / cur.n);
        cur.tile = (int)(local % cur.n);
        cur.tile0 = (int)(window_start(p, seq_len_at(p, b0)) / kTile);
        cursor_place(cur, p);
    }
    Cursor prod = cur;

    // Producer step (lane 0): stage tile `prod` into stage s.
    // page-table entries by warp: lane i holds entry tab_base + i of request tab_b, so
    // a tile's page id is a shuffle and the table is read once per 32 pages
    int tab_b = -1;
    int64_t tab_base = 0;
    int32_t tab_val = -1;
    // armed_only: failure injection -- the barrier expects the stage's bytes but no
    // copy is issued, so the wait on this stage runs out
    auto issue = [&](int s, bool armed_only) {
        if (prod.b != tab_b || prod.page_idx < tab_base || prod.page_idx >= tab_base + 32) {
            tab_b = prod.b;
            tab_base = prod.page_idx;
            const int64_t e = tab_base + lane;
            const int64_t row = ROWS ? (int64_t)__ldg(p.table_rows + tab_b) : (int64_t)tab_b;
            tab_val = e < p.max_pages ? __ldg(p.tables + row * p.max_pages + e) : -1;
        }
        const int32_t page = __shfl_sync(0xffffffffu, tab_val, (int)(prod.page_idx - tab_base));
        if (lane != 0) return;
        stage_page[s] = page;
        if (page < 0 || page >= p.n_pages) {
            atomicOr(p.err, PKV_DEVERR_PAGE_ID);
            mbar_arrive(&bars[s]);
            return;
        }
        const int64_t off = (kv_block(p, page, prod.h) * p.P + prod.slot0) * D;
        unsigned char* dst = ring + s * Gm::STAGE_BYTES;
        mbar_arrive_expect_tx(&bars[s], Gm::STAGE_BYTES);
        if (armed_only) return;
        bulk_copy_g2s(dst, static_cast<const T*>(p.k_pages) + off, Gm::TILE_BYTES, &bars[s], policy);
        bulk_copy_g2s(dst + Gm::TILE_BYTES, static_cast<const T*>(p.v_pages) + off, Gm::TILE_BYTES,
                      &bars[s], policy);
    };

    const int prologue = n_work < Gm::STAGES ? n_work : Gm::STAGES;
    if (early) {
        tab_b = prod.b;
        tab_base = prod.page_idx;
        tab_val = tab_base + lane < p.max_pages ? __ldg(p.tables + (int64_t)tab_b * p.max_pages +
                                                        tab_base + lane) : -1;
        // this worker's first tiles (inside the table window) go to L2 now: a few, so
        // that a long call's workers do not evict one another's
        Cursor pf = prod;
        for (int k = 0; k < n_work && k < kEarlyTiles; ++k) {
            if (pf.b != tab_b || pf.page_idx < tab_base || pf.page_idx >= tab_base + 32) break;
            const int32_t page = __shfl_sync(0xffffffffu, tab_val, (int)(pf.page_idx - tab_base));
            if (lane == 0 && page >= 0 && page < p.n_pages) {
                const int64_t off = (kv_block(p, page, pf.h) * p.P + pf.slot0) * D;
                bulk_prefetch_l2(static_cast<const T*>(p.k_pages) + off, Gm::TILE_BYTES);
                bulk_prefetch_l2(static_cast<const T*>(p.v_pages) + off, Gm::TILE_BYTES);
            }
            cursor_advance(pf, p);
        }
        // the entries are in registers before the wait, not loaded after it
        asm volatile("" ::"r"(tab_val));
        pdl_wait_primary();
    }
    for (int s = 0; s < prologue; ++s) {
        issue(s, s == 0 && p.inject_worker == w + 1);
        cursor_advance(prod, p);
    }

    const int rg = lane / Gm::TPR;             // row group of this lane
    const int col = (lane % Gm::TPR) * Gm::VEC; // first feature of this lane
    const int it_own = (lane % Gm::TPR) >> 1;  // warp step of the row this lane scores
    const int row_own = it_own * Gm::RPI + rg;

    float2 qv[G][NV];
    float2 o[G][NV];
    float m[G], l[G];
    int piece_first = 0, t_b = 0, w_start = 0;
    int s = 0;
    uint32_t parity = 0;

    for (int k = 0; k < n_work; ++k) {
        const int64_t lane_id = (int64_t)cur.b * p.H + ((cur.h << p.kv_shift) | sub);

        if (k == 0 || cur.tile == 0) {   // a new lane piece starts
            piece_first = cur.tile;
            t_b = (int)seq_len_at(p, cur.b);
            w_start = (int)window_start(p, t_b);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float2* qp = reinterpret_cast<const float2*>(p.q + (lane_id * G + g) * D + col);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const float2 qq = qp[v];
                    qv[g][v] = make_float2(qq.x * p.qscale, qq.y * p.qscale);
                    o[g][v] = make_float2(0.f, 0.f);
                }
                m[g] = -INFINITY;
                l[g] = 0.f;
            }
        }

        if (!mbar_wait_bounded(&bars[s], parity, p.wait_ns)) {
            if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            // let the copies already issued land before the shared memory goes away
            const int last = (k + Gm::STAGES - 1 < n_work - 1) ? k + Gm::STAGES - 1 : n_work - 1;
            int s2 = s;
            uint32_t par2 = parity;
            for (int j = k + 1; j <= last; ++j) {
                if (++s2 == Gm::STAGES) {
                    s2 = 0;
                    par2 ^= 1u;
                }
                mbar_wait_bounded(&bars[s2], par2, p.wait_ns);
            }
            return;
        }

        T* Ks = reinterpret_cast<T*>(ring + s * Gm::STAGE_BYTES);
        T* Vs = Ks + kTile * D;
        const int32_t page = stage_page[s];
        const bool page_ok = page >= 0 && page < p.n_pages;
        const bool last_tile = cur.tile == cur.n - 1;
        const int base = (cur.tile0 + cur.tile) * kTile;          // position of the tile's row 0
        const int rem = t_b - base;
        const int rows = !page_ok ? 0 : (rem < kTile ? rem : kTile);
        const int lo = w_start > base ? w_start - base : 0;       // rows before the window


        if (last_tile && page_ok) {
            // fused append: row t_b - 1 comes from k_new / v_new, into the tile and the page
            const int r = rows - 1;
            if (lane < Gm::TPR) {
                const int64_t src = kv_new_row(p, cur.b, cur.h) * D + col;
                const VT kb = *reinterpret_cast<const VT*>(static_cast<const T*>(p.k_new) + src);
                const VT vb = *reinterpret_cast<const VT*>(static_cast<const T*>(p.v_new) + src);
                *reinterpret_cast<VT*>(Ks + r * D + col) = kb;
                *reinterpret_cast<VT*>(Vs + r * D + col) = vb;
                const int64_t dst = (kv_block(p, page, cur.h) * p.P + cur.slot0 + r) * D + col;
                *reinterpret_cast<VT*>(static_cast<T*>(p.k_pages) + dst) = kb;
                *reinterpret_cast<VT*>(static_cast<T*>(p.v_pages) + dst) = vb;
            }
            __syncwarp();
        }

        if (rows > 0) {
            // partial dot products of this lane's features for its ITERS rows, per query
            float sc[G][Gm::ITERS];
#pragma unroll
            for (int it = 0; it < Gm::ITERS; ++it) {
                const int row = it * Gm::RPI + rg;
                float2 kf[NV];
                if (row < kTile) {
                    const VT kb = *reinterpret_cast<const VT*>(Ks + row * D + col);
                    Storage<T>::template to_float2<Gm::VEC>(&kb, kf);
                } else {
#pragma unroll
                    for (int v = 0; v < NV; ++v) kf[v] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int v = 0; v < NV; ++v) acc = __ffma2_rn(qv[g][v], kf[v], acc);
                    sc[g][it] = acc.x + acc.y;
                }
            }
            // transposed reduction over the TPR lanes of a row: each round halves
            // the values a lane keeps, the last round adds lane pairs
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int r = 0; r < Gm::HALVING_ROUNDS; ++r) {
                    const int half = Gm::ITERS >> (r + 1);   // lane offset of this round = 2 * half
                    const bool upper = (lane & (2 * half)) != 0;
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        const float send = upper ? sc[g][i] : sc[g][i + half];
                        const float keep = upper ? sc[g][i + half] : sc[g][i];
                        sc[g][i] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * half);
                    }
                }
                if (Gm::TPR >= 2) sc[g][0] += __shfl_xor_sync(0xffffffffu, sc[g][0], 1);
            }
            float p_own[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float s_own = (row_own >= lo && row_own < rows) ? sc[g][0] : -INFINITY;
                float tmax = s_own;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1)
                    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
                const float m_new = fmaxf(m[g], tmax);
                const float alpha = exp2f(m[g] - m_new);
                p_own[g] = exp2f(s_own - m_new);
                l[g] = fmaf(l[g], alpha, p_own[g]);
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int v = 0; v < NV; ++v) o[g][v] = __fmul2_rn(o[g][v], a2);
                m[g] = m_new;
            }
#pragma unroll
            for (int it = 0; it < Gm::ITERS; ++it) {
                const int row = it * Gm::RPI + rg;
                float pw[G];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    pw[g] = Gm::TPR >= 2
                        ? __shfl_sync(0xffffffffu, p_own[g], (lane & ~(Gm::TPR - 1)) | (it << 1))
                        : p_own[g];
                if (row >= lo && row < rows) {
                    float2 vf[NV];
                    const VT vb = *reinterpret_cast<const VT*>(Vs + row * D + col);
                    Storage<T>::template to_float2<Gm::VEC>(&vb, vf);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float2 p2 = make_float2(pw[g], pw[g]);
#pragma unroll
                        for (int v = 0; v < NV; ++v) o[g][v] = __ffma2_rn(p2, vf[v], o[g][v]);
                    }
                }
            }
        }

        // the stage is free again: hand it to the copy engine for tile k + STAGES
        fence_proxy_async_smem();
        __syncwarp();
        if (k + Gm::STAGES < n_work) {
            issue(s, false);
            cursor_advance(prod, p);
        }
        if (++s == Gm::STAGES) {
            s = 0;
            parity ^= 1u;
        }

        if (last_tile || k == n_work - 1) {
            // close the lane piece: sum the lanes' shares of l, and o over row groups
            float lt[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                lt[g] = l[g];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) lt[g] += __shfl_xor_sync(0xffffffffu, lt[g], off);
                lt[g] *= 1.f / Gm::DUP;
#pragma unroll
                for (int off = Gm::TPR; off < 32; off <<= 1) {
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        o[g][v].x += __shfl_xor_sync(0xffffffffu, o[g][v].x, off);
                        o[g][v].y += __shfl_xor_sync(0xffffffffu, o[g][v].y, off);
                    }
                }
            }
            if (piece_first == 0 && last_tile && p.pre_ml == nullptr) {
                if (lane < Gm::TPR) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float inv = 1.f / lt[g];
                        float2* op = reinterpret_cast<float2*>(p.out + (lane_id * G + g) * D + col);
#pragma unroll
                        for (int v = 0; v < NV; ++v)
                            op[v] = make_float2(o[g][v].x * inv, o[g][v].y * inv);
                    }
                }
            } else if (Gm::CLUSTER_LANES && G == 1 && p.lane_workers > 0) {
                // cluster lanes: the lane's kw workers merge their partials (max, sum, o)
                // in shared memory.  Inside one CTA (kw <= WARPS) worker j writes slot warp
                // and arrives on the lane's barrier; worker 0 waits and merges.  Across a
                // cluster of kw / WARPS CTAs, in two levels: every CTA's warps write their
                // slots and arrive on the CTA's barrier 0; its warp 0 merges those WARPS
                // partials and writes the result into slot WARPS + rank of the lead CTA
                // (cluster rank 0), arriving on the lead's barrier 1 (release, cluster
                // scope); the lead's warp 0 waits (acquire) and merges the CTA partials.
                constexpr int DPL = Gm::DPL;
                const int kw = p.lane_workers;
                const bool clu = kw > Gm::WARPS;
                const int j = (int)(w % kw);
                const int bidx = clu ? 0 : warp / kw;
                {
                    float* part = lane_part + warp * (D + 2);
                    if (lane < Gm::TPR) {
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            part[2 + col + 2 * v] = o[0][v].x;
                            part[3 + col + 2 * v] = o[0][v].y;
                        }
                    }
                    if (lane == 0) {
                        part[0] = m[0];
                        part[1] = lt[0];
                    }
                    mbar_arrive(&lane_bar[bidx]);   // release at CTA scope
                }
                const bool feat = lane * DPL < D;
                float M = -INFINITY, L = 0.f, acc[DPL];
                // n partials from `base` -> their common maximum M, sum L and this
                // lane's features of the weighted output
                auto merge = [&](const float* base, int n) {
                    M = -INFINITY;
                    for (int s2 = lane; s2 < n; s2 += 32) M = fmaxf(M, base[s2 * (D + 2)]);
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1)
                        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                    L = 0.f;
#pragma unroll
                    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
                    for (int s2 = 0; s2 < n; ++s2) {
                        const float* ps = base + s2 * (D + 2);
                        const float ls = ps[1];
                        const float ws = ls > 0.f ? exp2f(ps[0] - M) : 0.f;
                        L = fmaf(ls, ws, L);
                        if (feat) {
#pragma unroll
                            for (int i = 0; i < DPL; ++i) acc[i] = fmaf(ws, ps[2 + lane * DPL + i], acc[i]);
                        }
                    }
                };
                auto write_out = [&]() {
                    if (feat) {
                        const float inv = 1.f / L;
                        float* op = p.out + lane_id * D + lane * DPL;
#pragma unroll
                        for (int i = 0; i < DPL; ++i) op[i] = acc[i] * inv;
                    }
                };
                if (!clu) {
                    if (j == 0) {
                        if (!mbar_wait_bounded(&lane_bar[bidx], 0, p.wait_ns)) {
                            if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                        } else {
                            merge(lane_part + warp * (D + 2), kw);
                            write_out();
                        }
                    }
                } else if (warp == 0) {
                    if (!mbar_wait_bounded(&lane_bar[0], 0, p.wait_ns)) {
                        if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                    } else {
                        merge(lane_part, Gm::WARPS);
                        const int ctas = kw / Gm::WARPS;
                        const uint32_t rank = (uint32_t)(blockIdx.x % (unsigned)ctas);
                        const uint32_t dst =
                            cluster_map(smem_u32(lane_part + (Gm::WARPS + rank) * (D + 2)), 0);
                        if (feat) {
#pragma unroll
                            for (int i = 0; i < DPL; ++i)
                                st_cluster_f32(dst + 4u * (uint32_t)(2 + lane * DPL + i), acc[i]);
                        }
                        if (lane == 0) {
                            st_cluster_f32(dst, M);
                            st_cluster_f32(dst + 4u, L);
                        }
                        // each lane releases its own stores (cluster scope)
                        mbar_arrive_cluster(cluster_map(smem_u32(&lane_bar[1]), 0));
                        if (rank == 0) {
                            if (!mbar_wait_cluster_bounded(&lane_bar[1], 0, p.wait_ns)) {
                                if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                            } else {
                                merge(lane_part + Gm::WARPS * (D + 2), ctas);
                                write_out();
                            }
                        }
                    }
                }
                __syncwarp();
            } else {
                // deposit the partial; the last of the lane's workers to arrive merges
                const int64_t slot =      // partial of KV lane K from range r, this sub-lane
                    ((((int64_t)cur.b * Hk + cur.h) + (w >> p.kv_shift)) << p.kv_shift) | sub;
                if (lane < Gm::TPR) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float2* op = reinterpret_cast<float2*>(p.part_o + (slot * G + g) * D + col);
#pragma unroll
                        for (int v = 0; v < NV; ++v) op[v] = o[g][v];
                    }
                }
                if (lane == 0) {
#pragma unroll
                    for (int g = 0; g < G; ++g) p.part_ml[slot * G + g] = make_float2(m[g], lt[g]);
                }
                if (p.pre_ml != nullptr) {
                    // the combine kernel merges every lane, after this kernel: no counter,
                    // and the kernel boundary orders the partials
                    __syncwarp();
                    cursor_advance(cur, p);
                    continue;
                }
                fence_acq_rel_gpu();   // release: every lane's share of the partial
                __syncwarp();          // before lane 0 counts it
                const int64_t A = cur.first + (int64_t)cur.h * cur.n;   // KV lane's first tile
                const int64_t r_lo = worker_of(A, T_all, R);
                const int64_t r_hi = worker_of(A + cur.n - 1, T_all, R);
                int need;
                if (T_all >= R) {
                    need = (int)(r_hi - r_lo + 1);   // no range is empty
                } else {
                    int c = 0;
                    for (int64_t x = r_lo + lane; x <= r_hi; x += 32)
                        c += (x * T_all) / R != ((x + 1) * T_all) / R;
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
                    need = c;
                }
                int arrived = 0;
                if (p.epoch == 0) {
                    // counters zeroed by the plan kernel of this call
                    if (lane == 0) arrived = (int)atomicAdd(&p.lane_cnt[lane_id], 1ull) + 1;
                } else if (lane == 0) {
                    // counter = epoch << 32 | count, epochs increasing from call to
                    // call: the max resets a counter left by an earlier call (never
                    // one of this call, whose value is at least epoch << 32), then add
                    unsigned long long* c = &p.lane_cnt[lane_id];
                    atomicMax(c, (unsigned long long)p.epoch << 32);
                    arrived = (int)((atomicAdd(c, 1ull) & 0xffffffffull) + 1);
                }
                arrived = __shfl_sync(0xffffffffu, arrived, 0);
                if (arrived == need) {
                    fence_acq_rel_gpu();   // acquire: every counted partial is visible
                    const int64_t K = (int64_t)cur.b * Hk + cur.h;
                    if constexpr (G == 1)
                        merge_query<D, Gm::DPL, G>(p, lane_id, 0, K, sub, r_lo, r_hi, T_all, lane);
                    else
                        merge_lane<D, G>(p, lane_id, K, sub, r_lo, r_hi, T_all, lane);
                }
                __syncwarp();
            }
        }
        cursor_advance(cur, p);
    }
}

// ------------------------------------------------- tensor-core split kernel --
//
// bf16 or fp32 storage, head width 64 or 128.  Same workers, partition, ring,
// fused append, partials and merge as split_decode_kernel; what differs is how a
// staged tile is consumed.  K and V tiles arrive by TMA tensor loads with the
// 128-byte swizzle (each 16-row x 128-byte box lands as 16 rows of 128 bytes
// whose 16-byte chunks are XOR-permuted by row), so the ldmatrix reads below
// hit 32 distinct banks.  The bf16 form follows; the fp32 form (tf32 MMAs on
// split operands) is described in the kernel.  Scores S = Q K^T and the mixture O += P V run on
// mma.sync m16n8k16 (bf16 inputs, fp32 accumulation) with a 16-row A tile:
// row g holds the bf16 rounding of query g (pre-scaled by log2(e)/sqrt(d_h))
// and row g + 8 the bf16 rounding of its remainder, so the two partial products
// sum to the fp32 query's product with ~2^-16 relative error.  The softmax
// weights P are split the same way for O.  Lane l owns query g = l / 4: its
// four scores per tile sit in the accumulator fragment, the quad of lanes
// 4g..4g+3 reduces the tile maximum and sum, and the weights feed the P V
// product straight from registers.


__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A B + D, m16n8k16, bf16 x bf16 -> fp32
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// bf16 rounding of (lo, hi) and of the remainders
__device__ __forceinline__ void split_bf16(float lo, float hi, uint32_t& big, uint32_t& rest) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    big = *reinterpret_cast<const uint32_t*>(&b);
    rest = pack_bf16(lo - __low2float(b), hi - __high2float(b));
}

// D = A B + D, m16n8k8, tf32 x tf32 -> fp32
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// x as big + rest, both tf32 values: big is x with its 13 low mantissa bits
// cleared, rest the cleared part (exact in fp32) with its own 13 low bits cleared,
// so |x - big - rest| < 2^-20 |x|.  Two logic operations and one subtraction.
__device__ __forceinline__ void split_tf32(float x, uint32_t& big, uint32_t& rest) {
    big = __float_as_uint(x) & 0xffffe000u;
    rest = __float_as_uint(x - __uint_as_float(big)) & 0xffffe000u;
}

// Shared-memory tile geometry of the tensor-core kernel for storage type T:
// every 16-row tile of K (and of V) is BOXES boxes of 16 rows x 128 bytes, each
// written by one TMA tensor load with the 128-byte swizzle.
template <typename T, int D>
struct MmaGeo {
    static constexpr int ES = sizeof(T);
    static constexpr int ROW_BYTES = D * ES;
    static constexpr int CHUNKS = ROW_BYTES / 16;         // 16-byte chunks per row
    static constexpr int BOXES = ROW_BYTES / 128;         // 128-byte swizzle boxes per row
    static constexpr int BOX_ELEMS = 128 / ES;            // elements per box row
    static constexpr int BOX_BYTES = kTile * 128;         // one box: 16 rows x 128 bytes
    static constexpr int TILE_BYTES = BOXES * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int KSTEPS = ROW_BYTES / 32;         // k-steps of S = Q K^T (16 bf16 / 8 fp32)
    static constexpr int NB = D / 8;                      // n-blocks of O
#if defined(PKV_MMA_WARPS) && defined(PKV_MMA_STAGES)
    static constexpr int WARPS = PKV_MMA_WARPS;
    static constexpr int STAGES = PKV_MMA_STAGES;
#else
    // bf16: the CUDA-core kernel's geometry for the same bytes per tile.  fp32: as many
    // warps (up to 8) as fit with two stages each (7 at head width 128: the kernel is
    // latency-bound, so warps beat stages), then as many stages as fit (up to 4).
    static constexpr int SMEM_MAX = 227 * 1024 - 1024;   // less the swizzle alignment
    static constexpr int F32_WARPS = SMEM_MAX / (2 * (STAGE_BYTES + 12)) < 8
                                         ? SMEM_MAX / (2 * (STAGE_BYTES + 12)) : 8;
    static constexpr int F32_STAGES = SMEM_MAX / (F32_WARPS * (STAGE_BYTES + 12)) < 4
                                          ? SMEM_MAX / (F32_WARPS * (STAGE_BYTES + 12)) : 4;
    static constexpr int WARPS = ES == 4 ? F32_WARPS : Geo<T, D>::WARPS;
    static constexpr int STAGES = ES == 4 ? F32_STAGES : Geo<T, D>::STAGES;
#endif
    static constexpr int WARP_SMEM = STAGES * STAGE_BYTES;
    // stage rings (1024-byte aligned, as the swizzle requires), then mbarriers and page ids
    static constexpr int CTA_SMEM = 1024 + WARPS * (WARP_SMEM + STAGES * 12);
    static_assert(D == 64 || D == 128, "tensor-core path: head width 64 or 128");
    static_assert(CTA_SMEM <= 227 * 1024, "CTA does not fit an SM");
};

// Cluster lanes of the tensor-core kernel (a single request, bf16): after the rings,
// 8 lane mbarriers and a partial slot -- G rows of (max, sum, o[D]) -- for each warp
// and for each of up to 8 CTAs of a cluster.  Offsets from the 1024-aligned base.
template <typename T, int D, int G>
struct MmaClu {
    using M = MmaGeo<T, D>;
    static constexpr int OFF = (M::WARPS * (M::WARP_SMEM + M::STAGES * 12) + 15) / 16 * 16;
    static constexpr int SLOT = G * (D + 2);               // floats of one partial
    static constexpr int BYTES = 64 + (M::WARPS + 8) * SLOT * 4;
    static constexpr int SMEM = 1024 + OFF + BYTES;         // dynamic shared memory with slots
    static constexpr bool ON = sizeof(T) == 2 && G <= 8 && (M::WARPS == 4 || M::WARPS == 8) &&
                               SMEM <= 227 * 1024;
};

// Byte offset of 16-byte chunk c of row r in a swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)((c >> 3) * (kTile * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Cluster lanes of the tensor-core kernel, after a worker has written its partial
// into its slot and arrived: the lane's first worker (inside one CTA), or warp 0 of
// every CTA of the lane's cluster and then the lead's, wait, merge and write `out`.
// Kept out of line: the split kernel's registers stay those of its streaming loop.
template <typename T, int D, int G>
__device__ __noinline__ void mma_lane_merge(const KParams& p, float* lane_part, uint64_t* lane_bar,
                                            int64_t lane_id, int64_t w, int warp, int lane) {
    using M = MmaGeo<T, D>;
    using C = MmaClu<T, D, G>;
    const int g = lane >> 2, t = lane & 3;
    const bool q_ok = g < G;
    const int kw = p.lane_workers;
    const bool clu = kw > M::WARPS;
    const int j = (int)(w % kw);
    const int bidx = clu ? 0 : warp / kw;
    float Mx = -INFINITY, Lx = 0.f;
    float2 acc[M::NB];
    // n partials from `base` -> row g's common maximum, sum and weighted output
    auto merge = [&](const float* base, int n) {
        const float* rb = base + g * (D + 2);
        Mx = -INFINITY;
        for (int s2 = 0; s2 < n; ++s2) Mx = fmaxf(Mx, rb[s2 * C::SLOT]);
        Lx = 0.f;
#pragma unroll
        for (int nb = 0; nb < M::NB; ++nb) acc[nb] = make_float2(0.f, 0.f);
        for (int s2 = 0; s2 < n; ++s2) {
            const float* ps = rb + s2 * C::SLOT;
            const float ls = ps[1];
            const float ws = ls > 0.f ? exp2f(ps[0] - Mx) : 0.f;
            Lx = fmaf(ls, ws, Lx);
#pragma unroll
            for (int nb = 0; nb < M::NB; ++nb) {
                const float2 x = *reinterpret_cast<const float2*>(ps + 2 + nb * 8 + 2 * t);
                acc[nb] = make_float2(fmaf(ws, x.x, acc[nb].x), fmaf(ws, x.y, acc[nb].y));
            }
        }
    };
    auto write_out = [&]() {
        const float inv = 1.f / Lx;
        float* op = p.out + (lane_id * G + g) * D + 2 * t;
#pragma unroll
        for (int nb = 0; nb < M::NB; ++nb)
            *reinterpret_cast<float2*>(op + nb * 8) =
                make_float2(acc[nb].x * inv, acc[nb].y * inv);
    };
    if (!clu) {
        if (j == 0) {
            if (!mbar_wait_bounded(&lane_bar[bidx], 0, p.wait_ns)) {
                if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            } else if (q_ok) {
                merge(lane_part + warp * C::SLOT, kw);
                write_out();
            }
        }
    } else if (warp == 0) {
        if (!mbar_wait_bounded(&lane_bar[0], 0, p.wait_ns)) {
            if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
        } else {
            const int ctas = kw / M::WARPS;
            const uint32_t rank = (uint32_t)(blockIdx.x % (unsigned)ctas);
            if (q_ok) {
                merge(lane_part, M::WARPS);
                const uint32_t dst = cluster_map(
                    smem_u32(lane_part + (M::WARPS + rank) * C::SLOT + g * (D + 2)), 0);
#pragma unroll
                for (int nb = 0; nb < M::NB; ++nb)
                    st_cluster_v2f32(dst + 4u * (uint32_t)(2 + nb * 8 + 2 * t), acc[nb]);
                if (t == 0) st_cluster_v2f32(dst, make_float2(Mx, Lx));
            }
            // each lane releases its own stores (cluster scope)
            mbar_arrive_cluster(cluster_map(smem_u32(&lane_bar[1]), 0));
            if (rank == 0) {
                if (!mbar_wait_cluster_bounded(&lane_bar[1], 0, p.wait_ns)) {
                    if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
                } else if (q_ok) {
                    merge(lane_part + M::WARPS * C::SLOT, ctas);
                    write_out();
                }
            }
        }
    }
}

template <typename T, int D, int G, bool ROWS = false>
__global__ void __launch_bounds__(MmaGeo<T, D>::WARPS * 32, 1)
split_decode_mma_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv) {
    // ROWS: request b reads page-table row p.table_rows[b], as in split_decode_kernel
    using M = MmaGeo<T, D>;
    // F32: fp32 storage on tf32 MMAs (m16n8k8).  Every fp32 operand is split into two
    // tf32 parts (big + rest, within 2^-20 relative); [big; rest] rows of q (or P) times
    // the big and the rest parts of K (or V) give all four cross products, each exact in
    // fp32, so S and O keep fp32-level accuracy.
    constexpr bool F32 = sizeof(T) == 4;
    static_assert((G >= 1 && G <= 8) || (G == 16 && !F32), "1 to 8 (bf16: or 16) query heads per KV head");
    // WIDE (G = 16): lane l owns queries l / 4 and l / 4 + 8, the A operands are
    // [q_hi rows 0-15] and [q_lo rows 0-15] (two MMAs per product), and each MMA row
    // is a query of its own.  Otherwise rows g and g + 8 of one A operand hold the
    // two bf16 parts of query g.
    constexpr bool WIDE = G == 16;
    constexpr int NQ = WIDE ? 2 : 1;            // queries per lane
    constexpr int NA = WIDE ? 2 : 1;            // A operands per product
    constexpr int NS = WIDE || F32 ? 2 : 1;     // accumulator sets per S block (A or B parts)
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * M::WARPS + warp;
    // cluster lanes: every CTA's lane barriers are initialised before any worker of
    // the cluster can arrive on them (every thread takes part, so before any return)
    using C = MmaClu<T, D, G>;
    uint64_t* lane_bar = reinterpret_cast<uint64_t*>(smem + C::OFF);        // [8]
    float* lane_part = reinterpret_cast<float*>(smem + C::OFF + 64);        // [slots][G][D+2]
    if constexpr (C::ON && !ROWS) {
        if (p.lane_workers > 0) {
            // as in the CUDA-core kernel: inside a CTA one barrier per lane; across a
            // cluster barrier 0 gathers this CTA's warps, barrier 1 (lead) the CTAs
            const uint32_t kw = (uint32_t)p.lane_workers;
            const uint32_t cnt = kw <= (uint32_t)M::WARPS ? 32u * kw
                                 : threadIdx.x == 1 ? 32u * (kw / M::WARPS) : 32u * M::WARPS;
            if (threadIdx.x < 8) mbar_init(&lane_bar[threadIdx.x], cnt);
            if (p.lane_workers > M::WARPS) {
                if (threadIdx.x == 0) fence_mbar_init();
                cluster_sync_all();
            } else {
                __syncthreads();
            }
        }
    }
    if (w >= p.W) return;

    unsigned char* ring = smem + warp * M::WARP_SMEM;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + M::WARPS * M::WARP_SMEM) + warp * M::STAGES;
    int32_t* stage_page =
        reinterpret_cast<int32_t*>(smem + M::WARPS * (M::WARP_SMEM + M::STAGES * 8)) +
        warp * M::STAGES;
    if (lane == 0) {
        for (int s = 0; s < M::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t policy = l2_stream_policy();

    // as in the CUDA-core kernel: a single request reads its page-table entries (and
    // fetches its first tiles into L2) before the wait
    const bool batched = p.seq_lens != nullptr;
    const bool early = !batched && !ROWS;
    if (!batched) pdl_launch_dependents();
    if (!early) pdl_wait_primary();

    // this worker's tiles: range w >> kv_shift, [begin, end) of the flattened (request,
    // KV head, tile) sequence, for sub-lane w & (2^kv_shift - 1) of every KV head in it
    const int sub = (int)(w & ((1 << p.kv_shift) - 1));
    const int Hk = p.H >> p.kv_shift, R = p.W >> p.kv_shift;
    const int64_t T_all = (int64_t)Hk * req_prefix_at(p, p.B);
    const int64_t begin = ((w >> p.kv_shift) * T_all) / R;
    const int64_t end = (((w >> p.kv_shift) + 1) * T_all) / R;
    const int n_work = (int)(end - begin);
    if (n_work <= 0) {
        if (early) pdl_wait_primary();
        return;
    }

    Cursor cur;
    {
        const int b0 = batched ? __ldg(p.worker_req + w) : 0;
        const int64_t pre = req_prefix_at(p, b0);
        cur.b = b0;
        cur.n = (int)(req_prefix_at(p, b0 + 1) - pre);
        cur.first = (int64_t)Hk * pre;
        const int64_t local = begin - cur.first;
        cur.h = (int)(local / cur.n);
        cur.tile = (int)(local % cur.n);
        cur.tile0 = (int)(window_start(p, seq_len_at(p, b0)) / kTile);
        cursor_place(cur, p);
    }
    Cursor prod = cur;

    // Producer step (lane 0): stage tile `prod` into stage s, box by box.
    // page-table entries by warp: lane i holds entry tab_base + i of request tab_b, so
    // a tile's page id is a shuffle and the table is read once per 32 pages
    int tab_b = -1;
    int64_t tab_base = 0;
    int32_t tab_val = -1;
    // armed_only: failure injection -- the barrier expects the stage's bytes but no
    // copy is issued, so the wait on this stage runs out
    auto issue = [&](int s, bool armed_only) {
        if (prod.b != tab_b || prod.page_idx < tab_base || prod.page_idx >= tab_base + 32) {
            tab_b = prod.b;
            tab_base = prod.page_idx;
            const int64_t e = tab_base + lane;
            const int64_t row = ROWS ? (int64_t)__ldg(p.table_rows + tab_b) : (int64_t)tab_b;
            tab_val = e < p.max_pages ? __ldg(p.tables + row * p.max_pages + e) : -1;
        }
        const int32_t page = __shfl_sync(0xffffffffu, tab_val, (int)(prod.page_idx - tab_base));
        if (lane != 0) return;
        stage_page[s] = page;
        if (page < 0 || page >= p.n_pages) {
            atomicOr(p.err, PKV_DEVERR_PAGE_ID);
            mbar_arrive(&bars[s]);
            return;
        }
        const int y = (int)(kv_block(p, page, prod.h) * p.P + prod.slot0);   // pool row
        unsigned char* dst = ring + s * M::STAGE_BYTES;
        mbar_arrive_expect_tx(&bars[s], M::STAGE_BYTES);
        if (armed_only) return;
#pragma unroll
        for (int bx = 0; bx < M::BOXES; ++bx) {
            tma_load_2d(dst + bx * M::BOX_BYTES, &tmk, bx * M::BOX_ELEMS, y, &bars[s], policy);
            tma_load_2d(dst + M::TILE_BYTES + bx * M::BOX_BYTES, &tmv, bx * M::BOX_ELEMS, y, &bars[s],
                        policy);
        }
    };

    const int prologue = n_work < M::STAGES ? n_work : M::STAGES;
    if (early) {
        tab_b = prod.b;
        tab_base = prod.page_idx;
        tab_val = tab_base + lane < p.max_pages ? __ldg(p.tables + (int64_t)tab_b * p.max_pages +
                                                        tab_base + lane) : -1;
        Cursor pf = prod;
        for (int k = 0; k < n_work && k < kEarlyTiles; ++k) {
            if (pf.b != tab_b || pf.page_idx < tab_base || pf.page_idx >= tab_base + 32) break;
            const int32_t page = __shfl_sync(0xffffffffu, tab_val, (int)(pf.page_idx - tab_base));
            if (lane == 0 && page >= 0 && page < p.n_pages) {
                const int64_t off = (kv_block(p, page, pf.h) * p.P + pf.slot0) * D;
                bulk_prefetch_l2(static_cast<const T*>(p.k_pages) + off, M::TILE_BYTES);
                bulk_prefetch_l2(static_cast<const T*>(p.v_pages) + off, M::TILE_BYTES);
            }
            cursor_advance(pf, p);
        }
        asm volatile("" ::"r"(tab_val));   // the entries are in registers before the wait
        pdl_wait_primary();
    }
    for (int s = 0; s < prologue; ++s) {
        issue(s, s == 0 && p.inject_worker == w + 1);
        cursor_advance(prod, p);
    }

    const int g = lane >> 2, t = lane & 3;     // fragment row group and column pair
    bool q_ok = g < G;                          // lanes with g >= G carry zero queries
    // block lanes (table-row form only): this lane's row, and how many positions
    // before the lane's last one its token stops
    const bool blocks = ROWS && p.blk_tok0 != nullptr;
    int64_t q_row = 0;
    int row_short = 0;
    // ldmatrix row addresses: matrix j = lane / 8, row r = lane % 8
    const int mj = lane >> 3, mr = lane & 7;

    uint32_t qa[NA][M::KSTEPS][4];              // A fragments of [q_hi; q_lo] (WIDE: q_hi, q_lo;
                                                // F32: [q_big; q_rest] over 8 features a step)
    float o[M::NB][4];                          // O accumulator fragments
    float m[NQ], l[NQ];                         // running max and this lane's share of the sum
    int piece_first = 0, t_b = 0, w_start = 0;
    int s = 0;
    uint32_t parity = 0;

    for (int k = 0; k < n_work; ++k) {
        const int64_t lane_id = (int64_t)cur.b * p.H + ((cur.h << p.kv_shift) | sub);

        if (k == 0 || cur.tile == 0) {   // a new lane piece starts
            piece_first = cur.tile;
            t_b = (int)seq_len_at(p, cur.b);
            w_start = (int)window_start(p, t_b);
            q_row = lane_id * G + (q_ok ? g : 0);
            if (blocks) {
                const int64_t br = g < G ? block_row(p, cur.b, cur.h, g) : -1;
                q_ok = br >= 0;
                q_row = q_ok ? br : 0;
                row_short = q_ok ? __ldg(p.blk_ntok + cur.b) - 1 - g / p.blk_gp : 0;
            }
            const float* qp = p.q + q_row * D;
#pragma unroll
            for (int ks = 0; ks < M::KSTEPS; ++ks) {
                if constexpr (F32) {
                    // row g: k = t and t + 4 of features 8ks .. 8ks+7; row g + 8: their rests
                    uint32_t b0, r0, b1, r1;
                    split_tf32(qp[ks * 8 + t] * p.qscale, b0, r0);
                    split_tf32(qp[ks * 8 + 4 + t] * p.qscale, b1, r1);
                    qa[0][ks][0] = q_ok ? b0 : 0u;
                    qa[0][ks][1] = q_ok ? r0 : 0u;
                    qa[0][ks][2] = q_ok ? b1 : 0u;
                    qa[0][ks][3] = q_ok ? r1 : 0u;
                    continue;
                }
                const float2 lo = *reinterpret_cast<const float2*>(qp + ks * 16 + 2 * t);
                const float2 hi = *reinterpret_cast<const float2*>(qp + ks * 16 + 8 + 2 * t);
                uint32_t b0, r0, b1, r1;
                split_bf16(lo.x * p.qscale, lo.y * p.qscale, b0, r0);
                split_bf16(hi.x * p.qscale, hi.y * p.qscale, b1, r1);
                if constexpr (WIDE) {
                    // query g + 8 sits 8 rows further on
                    const float2 lo8 = *reinterpret_cast<const float2*>(qp + 8 * D + ks * 16 + 2 * t);
                    const float2 hi8 = *reinterpret_cast<const float2*>(qp + 8 * D + ks * 16 + 8 + 2 * t);
                    uint32_t b2, r2, b3, r3;
                    split_bf16(lo8.x * p.qscale, lo8.y * p.qscale, b2, r2);
                    split_bf16(hi8.x * p.qscale, hi8.y * p.qscale, b3, r3);
                    qa[0][ks][0] = b0, qa[0][ks][1] = b2, qa[0][ks][2] = b1, qa[0][ks][3] = b3;
                    qa[1][ks][0] = r0, qa[1][ks][1] = r2, qa[1][ks][2] = r1, qa[1][ks][3] = r3;
                } else {
                    qa[0][ks][0] = q_ok ? b0 : 0u;   // row g,     k = 2t, 2t+1
                    qa[0][ks][1] = q_ok ? r0 : 0u;   // row g + 8
                    qa[0][ks][2] = q_ok ? b1 : 0u;   // row g,     k = 2t+8, 2t+9
                    qa[0][ks][3] = q_ok ? r1 : 0u;   // row g + 8
                }
            }
#pragma unroll
            for (int nb = 0; nb < M::NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                m[qi] = -INFINITY;
                l[qi] = 0.f;
            }
        }

        if (!mbar_wait_bounded(&bars[s], parity, p.wait_ns)) {
            if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            const int last = (k + M::STAGES - 1 < n_work - 1) ? k + M::STAGES - 1 : n_work - 1;
            int s2 = s;
            uint32_t par2 = parity;
            for (int j = k + 1; j <= last; ++j) {
                if (++s2 == M::STAGES) {
                    s2 = 0;
                    par2 ^= 1u;
                }
                mbar_wait_bounded(&bars[s2], par2, p.wait_ns);
            }
            return;
        }

        unsigned char* Ks = ring + s * M::STAGE_BYTES;
        unsigned char* Vs = Ks + M::TILE_BYTES;
        const int32_t page = stage_page[s];
        const bool page_ok = page >= 0 && page < p.n_pages;
        const bool last_tile = cur.tile == cur.n - 1;
        const int base = (cur.tile0 + cur.tile) * kTile;          // position of the tile's row 0
        const int rem = t_b - base;
        const int rows = !page_ok ? 0 : (rem < kTile ? rem : kTile);
        const int lo = w_start > base ? w_start - base : 0;       // rows before the window


        if (last_tile && page_ok) {
            // fused append: row t_b - 1 from k_new / v_new into the tile and the page
            // (block lanes: every chunk row is already in its page and in the tile);
            // rows past it (stale bytes, possibly not finite) are cleared in V
            const int r = rows - 1;
            constexpr int EPC = 16 / M::ES;               // elements per 16-byte chunk
            if (lane < M::CHUNKS && !blocks) {
                const int64_t src = kv_new_row(p, cur.b, cur.h) * D + lane * EPC;
                const uint4 kb = *reinterpret_cast<const uint4*>(static_cast<const T*>(p.k_new) + src);
                const uint4 vb = *reinterpret_cast<const uint4*>(static_cast<const T*>(p.v_new) + src);
                *reinterpret_cast<uint4*>(Ks + swz(r, lane)) = kb;
                *reinterpret_cast<uint4*>(Vs + swz(r, lane)) = vb;
                const int64_t dst = (kv_block(p, page, cur.h) * p.P + cur.slot0 + r) * D + lane * EPC;
                *reinterpret_cast<uint4*>(static_cast<T*>(p.k_pages) + dst) = kb;
                *reinterpret_cast<uint4*>(static_cast<T*>(p.v_pages) + dst) = vb;
            }
            for (int i = lane; i < (kTile - rows) * M::CHUNKS; i += 32) {
                const int rr = rows + i / M::CHUNKS, c = i % M::CHUNKS;
                *reinterpret_cast<uint4*>(Vs + swz(rr, c)) = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }

        if (rows > 0) {
            // S = [q_hi; q_lo] K^T (WIDE: q_hi K^T and q_lo K^T; F32: [q_big; q_rest] times
            // K_big^T and K_rest^T): 16 x 8 blocks for keys 0-7 (sa) and 8-15 (sb), one
            // accumulator set per A or B part
            float sa[NS][4], sb[NS][4];
#pragma unroll
            for (int a = 0; a < NS; ++a)
                sa[a][0] = sa[a][1] = sa[a][2] = sa[a][3] = sb[a][0] = sb[a][1] = sb[a][2] = sb[a][3] = 0.f;
            const uint32_t kbase = smem_u32(Ks);
#pragma unroll
            for (int ks = 0; ks < M::KSTEPS; ++ks) {
                // matrices: (keys 0-7, chunk 2ks), (keys 0-7, 2ks+1), (keys 8-15, 2ks), (keys 8-15, 2ks+1)
                // (F32: lane 4g+t receives feature 8ks+t, then 8ks+4+t, of key g: B of m16n8k8)
                const int key = ((mj >> 1) << 3) + mr;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + swz(key, 2 * ks + (mj & 1)), b0, b1, b2, b3);
                if constexpr (F32) {
                    uint32_t g0, r0, g1, r1, g2, r2, g3, r3;
                    split_tf32(__uint_as_float(b0), g0, r0);
                    split_tf32(__uint_as_float(b1), g1, r1);
                    split_tf32(__uint_as_float(b2), g2, r2);
                    split_tf32(__uint_as_float(b3), g3, r3);
                    mma_tf32(sa[0], qa[0][ks], g0, g1);
                    mma_tf32(sb[0], qa[0][ks], g2, g3);
                    mma_tf32(sa[1], qa[0][ks], r0, r1);
                    mma_tf32(sb[1], qa[0][ks], r2, r3);
                } else {
#pragma unroll
                    for (int a = 0; a < NA; ++a) {
                        mma_bf16(sa[a], qa[a][ks], b0, b1);
                        mma_bf16(sb[a], qa[a][ks], b2, b3);
                    }
                }
            }
            // scores of query g (WIDE: and g + 8) at keys 2t, 2t+1 (block a) and 8+2t, 9+2t (block b)
            float sc[NQ][4];
            if constexpr (F32) {
                sc[0][0] = (sa[0][0] + sa[1][0]) + (sa[0][2] + sa[1][2]);
                sc[0][1] = (sa[0][1] + sa[1][1]) + (sa[0][3] + sa[1][3]);
                sc[0][2] = (sb[0][0] + sb[1][0]) + (sb[0][2] + sb[1][2]);
                sc[0][3] = (sb[0][1] + sb[1][1]) + (sb[0][3] + sb[1][3]);
            } else if constexpr (WIDE) {
#pragma unroll
                for (int qi = 0; qi < 2; ++qi) {
                    sc[qi][0] = sa[0][2 * qi] + sa[1][2 * qi];
                    sc[qi][1] = sa[0][2 * qi + 1] + sa[1][2 * qi + 1];
                    sc[qi][2] = sb[0][2 * qi] + sb[1][2 * qi];
                    sc[qi][3] = sb[0][2 * qi + 1] + sb[1][2 * qi + 1];
                }
            } else {
                sc[0][0] = sa[0][0] + sa[0][2];
                sc[0][1] = sa[0][1] + sa[0][3];
                sc[0][2] = sb[0][0] + sb[0][2];
                sc[0][3] = sb[0][1] + sb[0][3];
            }
            const int keys[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
            float alpha[NQ], pw[NQ][4];
            bool rescale = false;
            // keys of this lane row in the tile (block lanes: its token ends row_short
            // positions before the lane's last one)
            const int rows_q = rows == 0 ? 0 : (rem - row_short < kTile ? rem - row_short : kTile);
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                float tmax = -INFINITY;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (!q_ok || keys[i] < lo || keys[i] >= rows_q) sc[qi][i] = -INFINITY;
                    tmax = fmaxf(tmax, sc[qi][i]);
                }
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
                const float m_new = q_ok ? fmaxf(m[qi], tmax) : 0.f;
                // a block-lane row with no key yet (its positions end before this
                // piece's tiles) keeps m = -inf: exponents taken from 0, weights 0
                const float mb = m_new == -INFINITY ? 0.f : m_new;
                alpha[qi] = q_ok ? exp2f(m[qi] - mb) : 1.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) pw[qi][i] = q_ok ? exp2f(sc[qi][i] - mb) : 0.f;
                l[qi] = fmaf(l[qi], alpha[qi], (pw[qi][0] + pw[qi][1]) + (pw[qi][2] + pw[qi][3]));
                m[qi] = q_ok ? m_new : m[qi];
                rescale = rescale || alpha[qi] != 1.f;
            }
            if (__any_sync(0xffffffffu, rescale)) {
                // accumulator rows g and g + 8: query g's two parts, or (WIDE) queries g, g + 8
                const float a_g = alpha[0], a_g8 = alpha[NQ - 1];
#pragma unroll
                for (int nb = 0; nb < M::NB; ++nb) {
                    o[nb][0] *= a_g;
                    o[nb][1] *= a_g;
                    o[nb][2] *= a_g8;
                    o[nb][3] *= a_g8;
                }
            }
            if constexpr (F32) {
                // O += [P_big; P_rest] V over two k-steps of 8 keys.  In step kk, k index t
                // stands for key 8kk + 2t and k index t + 4 for key 8kk + 2t + 1 (the keys
                // whose weights this lane holds); V's rows are read in the same order, at
                // feature 8nb + g (the 128-byte swizzle keeps the 32 lanes on 32 banks).
                uint32_t pa[2][4];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    split_tf32(pw[0][2 * kk], pa[kk][0], pa[kk][1]);
                    split_tf32(pw[0][2 * kk + 1], pa[kk][2], pa[kk][3]);
                }
                const unsigned char* vcol = Vs + ((g & 3) << 2);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int r0 = 8 * kk + 2 * t;
#pragma unroll
                    for (int n0 = 0; n0 < M::NB; n0 += 4) {   // 4 n-blocks: independent MMAs in a row
                        uint32_t vg[4][2], vr[4][2];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int c = 2 * (n0 + j) + (g >> 2);   // chunk of feature 8(n0+j) + g
                            split_tf32(*reinterpret_cast<const float*>(vcol + swz(r0, c)), vg[j][0], vr[j][0]);
                            split_tf32(*reinterpret_cast<const float*>(vcol + swz(r0 + 1, c)), vg[j][1],
                                       vr[j][1]);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) mma_tf32(o[n0 + j], pa[kk], vg[j][0], vg[j][1]);
#pragma unroll
                        for (int j = 0; j < 4; ++j) mma_tf32(o[n0 + j], pa[kk], vr[j][0], vr[j][1]);
                    }
                }
            } else {
                // A fragments of [P_hi; P_lo] over the 16 keys (WIDE: P_hi and P_lo of both queries)
                uint32_t pa[NA][4];
                if constexpr (WIDE) {
                    split_bf16(pw[0][0], pw[0][1], pa[0][0], pa[1][0]);   // row g,     keys 2t, 2t+1
                    split_bf16(pw[1][0], pw[1][1], pa[0][1], pa[1][1]);   // row g + 8
                    split_bf16(pw[0][2], pw[0][3], pa[0][2], pa[1][2]);   // row g,     keys 8+2t, 9+2t
                    split_bf16(pw[1][2], pw[1][3], pa[0][3], pa[1][3]);   // row g + 8
                } else {
                    split_bf16(pw[0][0], pw[0][1], pa[0][0], pa[0][1]);
                    split_bf16(pw[0][2], pw[0][3], pa[0][2], pa[0][3]);
                }
                // O += [P_hi; P_lo] V : V[key][dim] as the k x n operand, transposed on load
                const uint32_t vbase = smem_u32(Vs);
#pragma unroll
                for (int np = 0; np < M::NB / 2; ++np) {
                    // matrices: (keys 0-7, chunk 2np), (keys 8-15, 2np), (keys 0-7, 2np+1), (keys 8-15, 2np+1)
                    const int key = ((mj & 1) << 3) + mr;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_trans(vbase + swz(key, 2 * np + (mj >> 1)), b0, b1, b2, b3);
#pragma unroll
                    for (int a = 0; a < NA; ++a) {
                        mma_bf16(o[2 * np], pa[a], b0, b1);
                        mma_bf16(o[2 * np + 1], pa[a], b2, b3);
                    }
                }
            }
        }

        // the stage is free again: hand it to the copy engine for tile k + STAGES
        fence_proxy_async_smem();
        __syncwarp();
        if (k + M::STAGES < n_work) {
            issue(s, false);
            cursor_advance(prod, p);
        }
        if (++s == M::STAGES) {
            s = 0;
            parity ^= 1u;
        }

        if (last_tile || k == n_work - 1) {
            // close the lane piece: quad sums of l; rows g and g + 8 of O add up (WIDE:
            // they are queries g and g + 8)
            float lt[NQ];
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                lt[qi] = l[qi];
                lt[qi] += __shfl_xor_sync(0xffffffffu, lt[qi], 1);
                lt[qi] += __shfl_xor_sync(0xffffffffu, lt[qi], 2);
            }
            auto o_pair = [&](int nb, int qi) {
                return WIDE ? make_float2(o[nb][2 * qi], o[nb][2 * qi + 1])
                            : make_float2(o[nb][0] + o[nb][2], o[nb][1] + o[nb][3]);
            };
            if (piece_first == 0 && last_tile && p.pre_ml == nullptr) {
                if (q_ok) {
#pragma unroll
                    for (int qi = 0; qi < NQ; ++qi) {
                        const float inv = 1.f / lt[qi];
                        float* op = p.out + (blocks ? q_row : lane_id * G + g + 8 * qi) * D + 2 * t;
#pragma unroll
                        for (int nb = 0; nb < M::NB; ++nb) {
                            const float2 x = o_pair(nb, qi);
                            *reinterpret_cast<float2*>(op + nb * 8) = make_float2(x.x * inv, x.y * inv);
                        }
                    }
                }
            } else if (C::ON && !ROWS && p.lane_workers > 0) {
                // cluster lanes, as in the CUDA-core kernel: the lane's kw workers merge
                // their partials (G rows each, in the accumulator layout: this lane holds
                // row g, features 8nb + 2t and + 1) through shared memory, inside one CTA
                // or in two levels across a cluster of kw / WARPS CTAs
                const int kw = p.lane_workers;
                const int bidx = kw > M::WARPS ? 0 : warp / kw;
                if (q_ok) {
                    float* r = lane_part + warp * C::SLOT + g * (D + 2);
#pragma unroll
                    for (int nb = 0; nb < M::NB; ++nb)
                        *reinterpret_cast<float2*>(r + 2 + nb * 8 + 2 * t) = o_pair(nb, 0);
                    if (t == 0) {
                        r[0] = m[0];
                        r[1] = lt[0];
                    }
                }
                mbar_arrive(&lane_bar[bidx]);   // release at CTA scope
                mma_lane_merge<T, D, G>(p, lane_part, lane_bar, lane_id, w, warp, lane);
                __syncwarp();
            } else {
                const int64_t slot =      // partial of KV lane K from range r, this sub-lane
                    ((((int64_t)cur.b * Hk + cur.h) + (w >> p.kv_shift)) << p.kv_shift) | sub;
                if (q_ok) {
#pragma unroll
                    for (int qi = 0; qi < NQ; ++qi) {
                        float* op = p.part_o + (slot * G + g + 8 * qi) * D + 2 * t;
#pragma unroll
                        for (int nb = 0; nb < M::NB; ++nb)
                            *reinterpret_cast<float2*>(op + nb * 8) = o_pair(nb, qi);
                        if (t == 0) p.part_ml[slot * G + g + 8 * qi] = make_float2(m[qi], lt[qi]);
                    }
                }
                if (p.pre_ml != nullptr) {
                    // the combine kernel merges every lane, after this kernel: no counter,
                    // and the kernel boundary orders the partials
                    __syncwarp();
                    cursor_advance(cur, p);
                    continue;
                }
                fence_acq_rel_gpu();   // release: every lane's share of the partial
                __syncwarp();          // before lane 0 counts it
                const int64_t A = cur.first + (int64_t)cur.h * cur.n;   // KV lane's first tile
                const int64_t r_lo = worker_of(A, T_all, R);
                const int64_t r_hi = worker_of(A + cur.n - 1, T_all, R);
                int need;
                if (T_all >= R) {
                    need = (int)(r_hi - r_lo + 1);   // no range is empty
                } else {
                    int c = 0;
                    for (int64_t x = r_lo + lane; x <= r_hi; x += 32)
                        c += (x * T_all) / R != ((x + 1) * T_all) / R;
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
                    need = c;
                }
                int arrived = 0;
                if (p.epoch == 0) {
                    if (lane == 0) arrived = (int)atomicAdd(&p.lane_cnt[lane_id], 1ull) + 1;
                } else if (lane == 0) {
                    unsigned long long* c = &p.lane_cnt[lane_id];
                    atomicMax(c, (unsigned long long)p.epoch << 32);
                    arrived = (int)((atomicAdd(c, 1ull) & 0xffffffffull) + 1);
                }
                arrived = __shfl_sync(0xffffffffu, arrived, 0);
                if (arrived == need) {
                    fence_acq_rel_gpu();   // acquire: every counted partial is visible
                    merge_lane<D, G>(p, lane_id, (int64_t)cur.b * Hk + cur.h, sub, r_lo, r_hi,
                                     T_all, lane);
                }
                __syncwarp();
            }
        }
        cursor_advance(cur, p);
    }
}

// ------------------------------------------------------------------ host --

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WorkspaceLayout workspace_layout(int B, int H, int D, int workers, int G) {
    WorkspaceLayout L{};
    size_t off = 0;
    // lane counters first: their place must not depend on the worker count,
    // because epoch-tagged counters persist from one call to the next
    L.lane_cnt = off;
    off = align_up(off + sizeof(unsigned long long) * (size_t)B * H, 256);
    L.req_prefix = off;
    off = align_up(off + sizeof(int64_t) * ((size_t)B + 1), 256);
    L.worker_req = off;
    off = align_up(off + sizeof(int32_t) * (size_t)workers, 256);
    const size_t slots = (size_t)B * H + (size_t)workers;   // per KV lane and worker
    L.part_ml = off;
    off = align_up(off + sizeof(float2) * slots * (size_t)G, 256);
    L.part_o = off;
    off = align_up(off + sizeof(float) * slots * (size_t)G * (size_t)D, 256);
    L.total = off;
    return L;
}

#ifndef PKV_LANE_MIN_TILES
// cluster lanes: tiles per worker at least.  Their two-level merge through shared
// memory is cheap, so a lane takes as many workers as fit (one tile each at most):
// fewer tiles per worker means fewer copy round trips, and more workers spread a
// lane's copies over more SMs
#define PKV_LANE_MIN_TILES 1
#endif
#ifndef PKV_LANE_MAX_TILES
// ... and at most this many: a longer lane streams at the HBM rate, which the
// global merge's grid over every SM serves better than a lane's cluster of 8 CTAs
#define PKV_LANE_MAX_TILES 4
#endif

// Cluster lanes for a single request (either split kernel): kw workers per lane, a
// power of two below a CTA's warps (lanes inside one CTA) or a multiple of them (one
// cluster of kw / warps CTAs per lane), the largest that fits; every lane has the
// same tiles.  0: this call keeps the global merge.
static int lane_worker_count(const KParams& p, int warps) {
    if (p.seq_lens != nullptr || p.kv_shift != 0 || p.table_rows != nullptr ||
        p.pre_ml != nullptr || p.inject_worker != 0)
        return 0;
    const int64_t t = p.single_t;
    const int64_t ws = (p.window > 0 && t > p.window) ? t - p.window : 0;
    const int64_t n = (t + kTile - 1) / kTile - ws / kTile;    // tiles per lane
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            sms = -1;
    }
    if (sms <= 0) return 0;
    // workers per lane at most: PKV_LANE_MIN_TILES tiles each, a cluster of 8 CTAs,
    // and every lane's CTAs resident at once (one CTA per SM)
    int64_t kmax = (n + PKV_LANE_MIN_TILES - 1) / PKV_LANE_MIN_TILES;
    if (kmax > 8 * warps) kmax = 8 * warps;
    if (kmax > (int64_t)sms * warps / p.H) kmax = (int64_t)sms * warps / p.H;
    // the largest count allowed: a power of two up to warps, then multiples of it
    int64_t k = 0;
    if (kmax >= warps) {
        k = kmax / warps * warps;
    } else if (kmax >= 1) {
        k = 1;
        while (k * 2 <= kmax) k <<= 1;
    }
    return (k >= 1 && k <= n && (n + k - 1) / k <= PKV_LANE_MAX_TILES) ? (int)k : 0;
}
#ifndef PKV_MIN_TILES_PER_WORKER
#define PKV_MIN_TILES_PER_WORKER 4   // below this much work a worker's fixed costs dominate
#endif

int launch_workers(int pool_workers, int B, int H, int64_t max_seq_len, int kv_shift) {
    const int64_t tiles = (int64_t)B * H * ((max_seq_len + kTile - 1) / kTile);
    const int64_t want = (tiles + PKV_MIN_TILES_PER_WORKER - 1) / PKV_MIN_TILES_PER_WORKER;
    const int w = (int)(want < pool_workers ? (want < 1 ? 1 : want) : pool_workers);
    // one worker per sub-lane of each range: a multiple of 2^kv_shift
    const int ns = 1 << kv_shift;
    return w < ns ? ns : w / ns * ns;
}

template <typename T, int D, int G>
static cudaError_t prepare_split() {
    static bool done = false;   // per instantiation
    if (done) return cudaSuccess;
    using Gm = Geo<T, D, G>;
    // room for the cluster-lane barriers and partial slots in single-request launches
    cudaError_t e = cudaFuncSetAttribute(
        split_decode_kernel<T, D, G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        Gm::CLUSTER_LANES && G == 1 ? Gm::CLU_OFF + Gm::CLU_BYTES : Gm::CTA_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(split_decode_kernel<T, D, G, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Geo<T, D, G>::CTA_SMEM);
    if (e == cudaSuccess) done = true;
    return e;
}

template <typename T, int D, int G>
static int resident_workers_t(int num_sms) {
    if (prepare_split<T, D, G>() != cudaSuccess) return 0;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, split_decode_kernel<T, D, G>,
                                                      Geo<T, D, G>::WARPS * 32, Geo<T, D, G>::CTA_SMEM) !=
        cudaSuccess)
        return 0;
    return blocks * num_sms * Geo<T, D, G>::WARPS;
}

template <typename T, int D, int G>
static cudaError_t launch_t(const DecodeArgs& a, KParams& p, cudaStream_t stream) {
    using Gm = Geo<T, D, G>;
    cudaError_t e = prepare_split<T, D, G>();
    if (e != cudaSuccess) return e;
    // the plan (a single request with epoch counters needs none) and, for a
    // shared-prefix call, the prefix kernel; the timing events bracket the attention:
    // the prefix kernel, if any, and the split kernel
    if (a.before_split == nullptr) {
        if (p.epoch == 0 && (e = launch_plan(a, p, stream)) != cudaSuccess) return e;
        if (a.ev_before && (e = cudaEventRecord(a.ev_before, stream)) != cudaSuccess) return e;
    } else {
        if (a.ev_before && (e = cudaEventRecord(a.ev_before, stream)) != cudaSuccess) return e;
        if ((e = launch_plan(a, p, stream)) != cudaSuccess) return e;
    }
    // cluster lanes for a single request on a multi-head pool
    int kw = 0;
    if constexpr (Gm::CLUSTER_LANES && G == 1) kw = lane_worker_count(p, Gm::WARPS);
    if (kw > 0) {
        p.lane_workers = kw;
        p.W = p.H * kw;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)((p.W + Gm::WARPS - 1) / Gm::WARPS));
    cfg.blockDim = dim3(Gm::WARPS * 32);
    cfg.dynamicSmemBytes = kw > 0 ? Gm::CLU_OFF + Gm::CLU_BYTES : Gm::CTA_SMEM;
    cfg.stream = stream;
    // dependent launch: behind this call's own plan kernel, or (a single request)
    // behind whatever came before; the kernel waits for it before reading anything
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (kw > Gm::WARPS) {   // a lane spans the CTAs of one cluster
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)(kw / Gm::WARPS);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    e = p.table_rows != nullptr ? cudaLaunchKernelEx(&cfg, split_decode_kernel<T, D, G, true>, p)
                                : cudaLaunchKernelEx(&cfg, split_decode_kernel<T, D, G, false>, p);
    if (e != cudaSuccess) return e;
    if (p.pre_ml != nullptr) {
        const int64_t rows = (int64_t)p.B * p.H * G;
        combine_kernel<D, G><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.ev_after && (e = cudaEventRecord(a.ev_after, stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

template <typename T, int D, int G>
static cudaError_t prepare_mma() {
    static bool done = false;   // per instantiation
    if (done) return cudaSuccess;
    // with cluster lanes the partial slots follow the rings
    constexpr int smem = MmaClu<T, D, G>::ON && MmaClu<T, D, G>::SMEM > MmaGeo<T, D>::CTA_SMEM
                             ? MmaClu<T, D, G>::SMEM : MmaGeo<T, D>::CTA_SMEM;
    cudaError_t e = cudaFuncSetAttribute(split_decode_mma_kernel<T, D, G, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess && sizeof(T) == 4)   // table rows: fp32 only (the decode-lane prefill)
        e = cudaFuncSetAttribute(split_decode_mma_kernel<T, D, G, sizeof(T) == 4>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, MmaGeo<T, D>::CTA_SMEM);
    if (e == cudaSuccess) done = true;
    return e;
}

template <typename T, int D, int G>
static int resident_workers_mma(int num_sms) {
    if (prepare_mma<T, D, G>() != cudaSuccess) return 0;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, split_decode_mma_kernel<T, D, G, false>,
                                                      MmaGeo<T, D>::WARPS * 32,
                                                      MmaGeo<T, D>::CTA_SMEM) != cudaSuccess)
        return 0;
    return blocks * num_sms * MmaGeo<T, D>::WARPS;
}

template <typename T, int D, int G>
static cudaError_t launch_mma(const DecodeArgs& a, KParams& p, cudaStream_t stream) {
    using M = MmaGeo<T, D>;
    cudaError_t e = prepare_mma<T, D, G>();
    if (e != cudaSuccess) return e;
    // the plan (a single request with epoch counters needs none) and, for a
    // shared-prefix call, the prefix kernel; the timing events bracket the attention:
    // the prefix kernel, if any, and the split kernel
    if (a.before_split == nullptr) {
        if (p.epoch == 0 && (e = launch_plan(a, p, stream)) != cudaSuccess) return e;
        if (a.ev_before && (e = cudaEventRecord(a.ev_before, stream)) != cudaSuccess) return e;
    } else {
        if (a.ev_before && (e = cudaEventRecord(a.ev_before, stream)) != cudaSuccess) return e;
        if ((e = launch_plan(a, p, stream)) != cudaSuccess) return e;
    }
    CUtensorMap tmk, tmv;
    memcpy(&tmk, a.tmap_k, sizeof tmk);
    memcpy(&tmv, a.tmap_v, sizeof tmv);
    // cluster lanes for a single request (bf16, up to 8 query heads per KV head)
    using C = MmaClu<T, D, G>;
    int kw = 0;
    if constexpr (C::ON) kw = lane_worker_count(p, M::WARPS);
    if (kw > 0) {
        p.lane_workers = kw;
        p.W = p.H * kw;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)((p.W + M::WARPS - 1) / M::WARPS));
    cfg.blockDim = dim3(M::WARPS * 32);
    cfg.dynamicSmemBytes = kw > 0 ? C::SMEM : M::CTA_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (kw > M::WARPS) {   // a lane spans the CTAs of one cluster
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)(kw / M::WARPS);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    if (p.table_rows != nullptr && sizeof(T) != 4) return cudaErrorInvalidValue;
    e = p.table_rows != nullptr
            ? cudaLaunchKernelEx(&cfg, split_decode_mma_kernel<T, D, G, sizeof(T) == 4>, p, tmk, tmv)
            : cudaLaunchKernelEx(&cfg, split_decode_mma_kernel<T, D, G, false>, p, tmk, tmv);
    if (e != cudaSuccess) return e;
    if (p.pre_ml != nullptr) {
        const int64_t rows = (int64_t)p.B * p.H * G;
        combine_kernel<D, G><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.ev_after && (e = cudaEventRecord(a.ev_after, stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

// The tensor-core kernel serves grouped-query pools (bf16 on bf16 MMAs, fp32 on
// split tf32 MMAs); for one query head per KV head the CUDA-core kernel is as fast
// (measured on GB300) and is kept.
#define PKV_FOR_EACH_MMA(X) X(__nv_bfloat16, 64, 2) X(__nv_bfloat16, 64, 4) X(__nv_bfloat16, 64, 8) \
    X(__nv_bfloat16, 64, 16) X(__nv_bfloat16, 128, 2) X(__nv_bfloat16, 128, 4)                    \
    X(__nv_bfloat16, 128, 8) X(__nv_bfloat16, 128, 16) X(float, 64, 2) X(float, 64, 4)           \
    X(float, 64, 8) X(float, 128, 2) X(float, 128, 4) X(float, 128, 8)

bool mma_supported(int dtype, int D, int G) {
    if (D != 64 && D != 128) return false;
    if (dtype == PKV_BF16) return G == 2 || G == 4 || G == 8 || G == 16;
    return dtype == PKV_F32 && (G == 2 || G == 4 || G == 8);
}

// Instantiated geometries: every head width for multi-head attention; groups
// of 2, 4 and 8 query heads per KV head at head widths 64 and 128.
#define PKV_FOR_EACH_D(X, T) X(T, 2, 1) X(T, 4, 1) X(T, 8, 1) X(T, 16, 1) X(T, 32, 1) \
    X(T, 64, 1) X(T, 128, 1) X(T, 64, 2) X(T, 64, 4) X(T, 64, 8) X(T, 128, 2) X(T, 128, 4) X(T, 128, 8)

bool decode_supported(int dtype, int D, int G) {
    if (D < 2 || D > 256 || (D & (D - 1)) != 0) return false;
    if (dtype != PKV_F32 && dtype != PKV_BF16) return false;
    if (dtype == PKV_F32 && D > 128) return false;
    if (G == 1) return true;
    return (G == 2 || G == 4 || G == 8) && (D == 64 || D == 128);
}

int resident_workers(int dtype, int D, int G, int num_sms, bool tensor_cores) {
    if (tensor_cores) {
#define PKV_RWM(TT, DD, GG)                                             \
        if (dtype == (sizeof(TT) == 4 ? PKV_F32 : PKV_BF16) && D == DD && G == GG) \
            return resident_workers_mma<TT, DD, GG>(num_sms);
        PKV_FOR_EACH_MMA(PKV_RWM)
#undef PKV_RWM
        return 0;
    }
#define PKV_RW(T, DD, GG) \
    if (D == DD && G == GG) return resident_workers_t<T, DD, GG>(num_sms);
    if (dtype == PKV_F32) {
        PKV_FOR_EACH_D(PKV_RW, float)
    } else if (dtype == PKV_BF16) {
        PKV_FOR_EACH_D(PKV_RW, __nv_bfloat16)
        PKV_RW(__nv_bfloat16, 256, 1)
    }
#undef PKV_RW
    return 0;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    KParams p{};
    p.q = a.q;
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.k_pages = a.k_pages;
    p.v_pages = a.v_pages;
    p.n_pages = a.n_pages;
    p.tables = a.tables;
    p.table_rows = a.table_rows;
    p.allow_empty = a.allow_empty;
    p.max_pages = a.max_pages;
    p.seq_lens = a.seq_lens;
    p.single_t = a.single_t;
    p.max_seq_len = a.max_seq_len;
    p.B = a.B;
    p.H = a.H;
    p.kv_shift = a.kv_shift;
    p.P = a.P;
    p.tiles_per_page = a.P / kTile;
    p.window = a.window;
    p.qscale = 1.4426950408889634f / sqrtf((float)a.D);
    p.out = a.out;
    const WorkspaceLayout L = workspace_layout(a.B, a.H, a.D, a.workers, a.G);
    unsigned char* ws = static_cast<unsigned char*>(a.workspace);
    p.req_prefix = reinterpret_cast<int64_t*>(ws + L.req_prefix);
    p.worker_req = reinterpret_cast<int32_t*>(ws + L.worker_req);
    p.lane_cnt = reinterpret_cast<unsigned long long*>(ws + L.lane_cnt);
    p.epoch = a.epoch;
    p.part_ml = reinterpret_cast<float2*>(ws + L.part_ml);
    p.part_o = reinterpret_cast<float*>(ws + L.part_o);
    p.W = a.workers;
    p.err = a.dev_error;
    p.key_start = a.key_start;
    p.pre_ml = static_cast<const float2*>(a.pre_ml);
    p.pre_o = a.pre_o;
    p.pre_splits = a.pre_splits;
    p.pre_stride = a.pre_stride;
    p.wait_ns = a.wait_limit_ns ? a.wait_limit_ns : kWaitLimitNs;
    p.inject_worker = a.inject_worker;
    p.blk_tok0 = a.blk_tok0;
    p.blk_ntok = a.blk_ntok;
    p.blk_gp = a.blk_gp;
    p.blk_hq = a.blk_hq;
    // block lanes exist only in the tensor-core kernel's table-row form (fp32)
    if (a.blk_tok0 != nullptr &&
        (a.table_rows == nullptr || a.tmap_k == nullptr || a.dtype != PKV_F32 || a.kv_shift != 0))
        return cudaErrorInvalidValue;
    if (a.tmap_k != nullptr && a.tmap_v != nullptr) {
        // table rows on the tensor-core kernel: fp32 pools only (the bf16 pools it
        // serves prefill on the tcgen05 kernel, not through decode lanes)
        if (a.table_rows != nullptr && a.dtype != PKV_F32) return cudaErrorInvalidValue;
#define PKV_LAUNCH_MMA(TT, DD, GG)                                                   \
        if (a.dtype == (sizeof(TT) == 4 ? PKV_F32 : PKV_BF16) && a.D == DD && a.G == GG) \
            return launch_mma<TT, DD, GG>(a, p, stream);
        PKV_FOR_EACH_MMA(PKV_LAUNCH_MMA)
#undef PKV_LAUNCH_MMA
        return cudaErrorInvalidValue;
    }
#define PKV_LAUNCH(T, DD, GG) \
    if (a.D == DD && a.G == GG) return launch_t<T, DD, GG>(a, p, stream);
    if (a.dtype == PKV_F32) {
        PKV_FOR_EACH_D(PKV_LAUNCH, float)
    } else if (a.dtype == PKV_BF16) {
        PKV_FOR_EACH_D(PKV_LAUNCH, __nv_bfloat16)
        PKV_LAUNCH(__nv_bfloat16, 256, 1)
    }
#undef PKV_LAUNCH
    return cudaErrorInvalidValue;
}

// ------------------------------------------------ prefill through decode lanes --

namespace {

struct LaneRowsParams {
    int B;
    int64_t N;
    int H, HQ, D, P, words;       // words: 32-bit words of one K or V head row
    const int32_t* cu_new;        // nullptr: one request of single_n rows
    const int32_t* seq_lens;
    int single_n;
    int64_t single_t;
    const int32_t* tables;
    int max_pages;
    int64_t n_pages;
    const uint32_t* k_new;
    const uint32_t* v_new;
    uint32_t* k_pages;
    uint32_t* v_pages;
    const uint16_t* q_bf16;       // non-null: widen q into q32
    float* q32;
    int32_t* rows;                // nullptr with block lanes (the block plan writes them)
    int32_t* lens;
    unsigned* err;
};

struct BlockPlanParams {
    int B;
    int64_t N;
    int bt;                       // chunk tokens per block
    int64_t X;                    // decode requests of the launch (blocks, then empty ones)
    const int32_t* cu_new;        // nullptr: one request of single_n rows
    const int32_t* seq_lens;
    int single_n;
    int64_t single_t;
    int max_pages, P;
    int32_t* first;               // [B + 1] first block of each request
    int32_t* rows;                // [X] table row (request) of each block
    int32_t* lens;                // [X] length at the block's last token (0: empty)
    int32_t* tok0;                // [X] first chunk row
    int32_t* ntok;                // [X] tokens
    unsigned* err;
};

__device__ __forceinline__ int lr_cu(const LaneRowsParams& p, int b) {
    return p.cu_new ? __ldg(p.cu_new + b) : (b == 0 ? 0 : p.single_n);
}

// One warp per chunk row x: its request b (the last with cu_new[b] <= x); its decode
// length L0_b + i + 1, or 0 when x belongs to no request or the request's lengths
// are bad (those set the error word); its K / V rows stored at position L0_b + i;
// and, for bf16 pools, its query widened to fp32 (exactly).
__global__ void __launch_bounds__(256) lane_rows_kernel(const LaneRowsParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t x = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); x < p.N;
         x += warps) {
        int lo = 0, hi = p.B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (lr_cu(p, mid) <= x) lo = mid;
            else hi = mid;
        }
        const int b = lo;
        const int c0 = lr_cu(p, b), c1 = lr_cu(p, b + 1);
        int64_t t = 0, pos = 0;
        int32_t page = -1;
        if (x >= c0 && x < c1) {
            const int64_t tb = p.seq_lens ? (int64_t)__ldg(p.seq_lens + b) : p.single_t;
            const int64_t L0 = tb - (c1 - c0);
            pos = L0 + (x - c0);
            if (L0 < 0 || tb > (int64_t)p.max_pages * p.P) {
                if (lane == 0) atomicOr(p.err, PKV_DEVERR_SEQ_LEN);
            } else {
                t = pos + 1;
                page = __ldg(p.tables + (int64_t)b * p.max_pages + pos / p.P);
                if (page < 0 || page >= p.n_pages) page = -1;   // the decode kernel reports it
            }
        }
        if (lane == 0 && p.rows != nullptr) {
            p.rows[x] = b;
            p.lens[x] = (int32_t)t;
        }
        if (page >= 0) {
            for (int h = 0; h < p.H; ++h) {
                const int64_t dst = (((int64_t)page * p.H + h) * p.P + pos % p.P) * p.words;
                const int64_t src = (x * p.H + h) * p.words;
                for (int u = lane; u < p.words; u += 32) {
                    p.k_pages[dst + u] = __ldg(p.k_new + src + u);
                    p.v_pages[dst + u] = __ldg(p.v_new + src + u);
                }
            }
        }
        if (p.q_bf16 != nullptr) {
            const int64_t n = (int64_t)p.HQ * p.D;
            for (int64_t e = lane; e < n; e += 32)
                p.q32[x * n + e] = __uint_as_float((uint32_t)__ldg(p.q_bf16 + x * n + e) << 16);
        }
    }
}

// Block lanes: request b's n_b chunk tokens form ceil(n_b / bt) blocks of bt
// consecutive tokens (the last may hold fewer), numbered request by request.  One
// CTA: block counts and their exclusive prefix over requests (first), then every
// decode request x of the launch: its request, first chunk row, token count and
// the length at its last token; x past the last block is empty (length 0).
__global__ void __launch_bounds__(1024) block_plan_kernel(const BlockPlanParams p) {
    __shared__ int warp_sum[32];
    __shared__ int carry_s;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    auto cu = [&](int b) { return p.cu_new ? __ldg(p.cu_new + b) : (b == 0 ? 0 : p.single_n); };
    auto seq = [&](int b) { return p.seq_lens ? (int64_t)__ldg(p.seq_lens + b) : p.single_t; };
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < p.B; base += 1024) {
        const int b = base + tid;
        int nb = 0;
        if (b < p.B) {
            const int c0 = cu(b), c1 = cu(b + 1);
            const int64_t n = (int64_t)c1 - c0, t = seq(b);
            const bool ok = c0 >= 0 && n >= 0 && c1 <= p.N && t - n >= 0 &&
                            t <= (int64_t)p.max_pages * p.P;
            if (!ok) atomicOr(p.err, PKV_DEVERR_SEQ_LEN);
            else nb = (int)((n + p.bt - 1) / p.bt);
        }
        int incl = nb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_sum[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int v = warp_sum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            warp_sum[lane] = v;
        }
        __syncthreads();
        const int carry = carry_s;
        if (b < p.B) p.first[b] = carry + (wid > 0 ? warp_sum[wid - 1] : 0) + incl - nb;
        __syncthreads();
        if (tid == 0) carry_s = carry + warp_sum[31];
        __syncthreads();
    }
    if (tid == 0) p.first[p.B] = carry_s;
    __syncthreads();
    const int total = carry_s;
    for (int64_t x = tid; x < p.X; x += 1024) {
        int32_t row = 0, len = 0, t0 = 0, nt = 0;
        if (x < total) {
            int lo = 0, hi = p.B;                       // last request with first[b] <= x
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (p.first[mid] <= x) lo = mid;
                else hi = mid;
            }
            const int b = lo;
            const int c0 = cu(b), n = cu(b + 1) - c0;
            const int blk = (int)(x - p.first[b]);
            row = b;
            t0 = c0 + blk * p.bt;
            nt = n - blk * p.bt < p.bt ? n - blk * p.bt : p.bt;
            len = (int32_t)(seq(b) - n + (int64_t)blk * p.bt + nt);
        }
        p.rows[x] = row;
        p.lens[x] = len;
        p.tok0[x] = t0;
        p.ntok[x] = nt;
    }
}

}  // namespace

int prefill_block_tokens(int dtype, int D, int G, int kv_shift, int64_t window, bool tmaps) {
    if (dtype != PKV_F32 || !tmaps || window > 0 || kv_shift != 0 || (D != 64 && D != 128))
        return 0;
    return (G == 1 || G == 2 || G == 4) && mma_supported(PKV_F32, D, 8) ? 8 / G : 0;
}

PrefillLanesLayout prefill_lanes_layout(int64_t N, int batch, int block_tokens, int lane_heads,
                                        int D, int workers, int lane_group, int query_heads,
                                        bool widen_q) {
    PrefillLanesLayout L{};
    const bool blocks = block_tokens > 0;
    const int64_t X = blocks ? N / block_tokens + batch : N;
    L.requests = X;
    L.decode = align_up(workspace_layout((int)X, lane_heads, D, workers, blocks ? 8 : lane_group).total,
                        256);
    L.rows = L.decode;
    L.lens = align_up(L.rows + sizeof(int32_t) * (size_t)X, 256);
    L.tok0 = align_up(L.lens + sizeof(int32_t) * (size_t)X, 256);
    L.ntok = blocks ? align_up(L.tok0 + sizeof(int32_t) * (size_t)X, 256) : L.tok0;
    L.first = blocks ? align_up(L.ntok + sizeof(int32_t) * (size_t)X, 256) : L.ntok;
    L.q32 = blocks ? align_up(L.first + sizeof(int32_t) * ((size_t)batch + 1), 256) : L.first;
    L.total = widen_q ? L.q32 + sizeof(float) * (size_t)N * query_heads * D : L.q32;
    return L;
}

cudaError_t launch_prefill_lanes(const PrefillLanesArgs& a, cudaStream_t stream) {
    const bool widen = a.dtype == PKV_BF16;
    const bool blocks = a.block_tokens > 0;
    if (blocks && (widen || a.tmap_k == nullptr || a.kv_shift != 0 || a.window > 0))
        return cudaErrorInvalidValue;
    const int nreq = a.cu_new ? a.batch : 1;
    const PrefillLanesLayout L = prefill_lanes_layout(a.total_new, nreq, a.block_tokens,
                                                      a.lane_heads, a.D, a.workers, a.lane_group,
                                                      a.query_heads, widen);
    unsigned char* ws = static_cast<unsigned char*>(a.workspace);
    LaneRowsParams r{};
    r.B = a.cu_new ? a.batch : 1;
    r.N = a.total_new;
    r.H = a.kv_heads;
    r.HQ = a.query_heads;
    r.D = a.D;
    r.P = a.P;
    r.words = a.D * (a.dtype == PKV_F32 ? 4 : 2) / 4;
    r.cu_new = a.cu_new;
    r.seq_lens = a.seq_lens;
    r.single_n = a.single_n;
    r.single_t = a.single_t;
    r.tables = a.tables;
    r.max_pages = a.max_pages;
    r.n_pages = a.n_pages;
    r.k_new = static_cast<const uint32_t*>(a.k_new);
    r.v_new = static_cast<const uint32_t*>(a.v_new);
    r.k_pages = static_cast<uint32_t*>(a.k_pages);
    r.v_pages = static_cast<uint32_t*>(a.v_pages);
    r.q_bf16 = widen ? static_cast<const uint16_t*>(a.q) : nullptr;
    r.q32 = widen ? reinterpret_cast<float*>(ws + L.q32) : nullptr;
    r.rows = blocks ? nullptr : reinterpret_cast<int32_t*>(ws + L.rows);
    r.lens = blocks ? nullptr : reinterpret_cast<int32_t*>(ws + L.lens);
    r.err = a.dev_error;
    const int64_t want = (a.total_new + 7) / 8;
    lane_rows_kernel<<<(unsigned)(want < 4096 ? (want < 1 ? 1 : want) : 4096), 256, 0, stream>>>(r);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (blocks) {
        BlockPlanParams bp{};
        bp.B = nreq;
        bp.N = a.total_new;
        bp.bt = a.block_tokens;
        bp.X = L.requests;
        bp.cu_new = a.cu_new;
        bp.seq_lens = a.seq_lens;
        bp.single_n = a.single_n;
        bp.single_t = a.single_t;
        bp.max_pages = a.max_pages;
        bp.P = a.P;
        bp.first = reinterpret_cast<int32_t*>(ws + L.first);
        bp.rows = reinterpret_cast<int32_t*>(ws + L.rows);
        bp.lens = reinterpret_cast<int32_t*>(ws + L.lens);
        bp.tok0 = reinterpret_cast<int32_t*>(ws + L.tok0);
        bp.ntok = reinterpret_cast<int32_t*>(ws + L.ntok);
        bp.err = a.dev_error;
        block_plan_kernel<<<1, 1024, 0, stream>>>(bp);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    DecodeArgs d{};
    d.dtype = a.dtype;
    d.B = (int)L.requests;
    d.H = a.lane_heads;
    d.D = a.D;
    d.P = a.P;
    d.G = blocks ? 8 : a.lane_group;
    d.kv_shift = a.kv_shift;
    d.window = a.window;
    d.q = widen ? reinterpret_cast<const float*>(ws + L.q32) : static_cast<const float*>(a.q);
    d.k_new = a.k_new;    // stored again by the decode kernel's append: the same bytes
    d.v_new = a.v_new;
    d.k_pages = a.k_pages;
    d.v_pages = a.v_pages;
    d.n_pages = a.n_pages;
    d.tables = a.tables;
    d.max_pages = a.max_pages;
    d.table_rows = reinterpret_cast<int32_t*>(ws + L.rows);
    d.seq_lens = reinterpret_cast<int32_t*>(ws + L.lens);
    if (blocks) {
        d.blk_tok0 = reinterpret_cast<int32_t*>(ws + L.tok0);
        d.blk_ntok = reinterpret_cast<int32_t*>(ws + L.ntok);
        d.blk_gp = a.lane_group;
        d.blk_hq = a.query_heads;
    }
    d.max_seq_len = (int64_t)a.max_pages * a.P;
    d.out = a.out;
    d.workspace = a.workspace;
    d.workspace_bytes = L.decode;
    d.workers = a.workers;
    d.dev_error = a.dev_error;
    d.ev_before = a.ev_before;
    d.ev_after = a.ev_after;
    d.tmap_k = a.tmap_k;
    d.tmap_v = a.tmap_v;
    d.allow_empty = true;
    return launch_decode(d, stream);
}

}  // namespace pkv
