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
// into slot lane + worker of the workspace (slots never collide: see
// merge_kernel), and the merge kernel combines them:
//     out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s.
//
// The append is fused into the worker that owns the lane's last tile: once that
// tile's copy has landed it overwrites row t_b - 1 of the staged tile with
// k_new / v_new (the pool may still hold stale bytes there) and stores the row
// into the page.  No other worker reads that tile, so nothing races.
//
// Faults are not raised by trapping: bad lengths and page ids, and waits that
// run out, set bits of a device error word and the offending work is skipped.

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "pkv.h"
#include "pkv_internal.h"

namespace pkv {

// ------------------------------------------------------------------ PTX --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async proxy (the bulk-copy engine).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0 && global_timer_ns() - start > limit_ns) return false;
    }
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy accesses (the next bulk copy into the same stage).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

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
    static constexpr int dtype = PKV_F32;
    template <int N>
    __device__ __forceinline__ static void to_float(const void* bits, float* out) {
        const float* f = reinterpret_cast<const float*>(bits);
#pragma unroll
        for (int i = 0; i < N; ++i) out[i] = f[i];
    }
};

template <>
struct Storage<__nv_bfloat16> {
    static constexpr int dtype = PKV_BF16;
    // bf16 is the upper half of an fp32: element 2i is the low half of word i.
    template <int N>
    __device__ __forceinline__ static void to_float(const void* bits, float* out) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(bits);
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

// Warp geometry of one tile for storage type T and head width D.
template <typename T, int D>
struct Geo {
    static constexpr int ES = sizeof(T);
    static constexpr int VEC = (16 / ES) < D ? (16 / ES) : D;  // elements per lane vector
    static constexpr int VBYTES = VEC * ES;                    // 16, 8 or 4
    static constexpr int TPR = D / VEC;                        // lanes sharing one row
    static constexpr int RPI = 32 / TPR;                       // rows per warp step
    static constexpr int ITERS = (kTile + RPI - 1) / RPI;      // warp steps per tile
    static constexpr int TILE_BYTES = kTile * D * ES;          // K (or V) rows of one tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int BUDGET = 24 * 1024;                   // shared memory per worker
    static constexpr int STAGES_RAW = BUDGET / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
    static constexpr int WARP_SMEM = STAGES * STAGE_BYTES;
    static constexpr int CTA_SMEM = kSplitWarps * WARP_SMEM + kSplitWarps * STAGES * 8;
    static_assert(D % VEC == 0 && TPR <= 32 && (TPR & (TPR - 1)) == 0, "unsupported head width");
    static_assert(TILE_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");
};

constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s per bounded wait

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
    const int32_t* seq_lens;    // nullptr: one request of length single_t
    int64_t single_t;
    int64_t single_tiles;
    int64_t max_seq_len;
    int B, H, P, tiles_per_page;
    float qscale;               // log2(e) / sqrt(D)
    float* out;
    int64_t* req_prefix;
    int32_t* worker_req;
    float2* part_ml;
    float* part_o;
    int W;
    unsigned* err;
};

// Tiles-per-lane prefix over requests (written by plan_kernel; closed form for
// a single request).
__device__ __forceinline__ int64_t req_prefix_at(const KParams& p, int b) {
    if (p.seq_lens == nullptr) return b == 0 ? 0 : p.single_tiles;
    return __ldg(p.req_prefix + b);
}

__device__ __forceinline__ int64_t seq_len_at(const KParams& p, int b) {
    return p.seq_lens == nullptr ? p.single_t : (int64_t)__ldg(p.seq_lens + b);
}

// ----------------------------------------------------------- plan kernel --

constexpr int kPlanThreads = 1024;

// Validates lengths, writes the per-request tile prefix and the first request
// of every worker.  One CTA.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const KParams p) {
    __shared__ int64_t warp_sums[kPlanThreads / 32];
    __shared__ int64_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < p.B; base += kPlanThreads) {
        const int i = base + tid;
        int64_t n = 0;
        if (i < p.B) {
            const int64_t t = p.seq_lens[i];
            const int64_t pages = (t + p.P - 1) / p.P;
            if (t < 1 || t > p.max_seq_len || pages > p.max_pages) {
                atomicOr(p.err, PKV_DEVERR_SEQ_LEN);
            } else {
                n = (t + kTile - 1) / kTile;
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
        if (i < p.B) p.req_prefix[i] = carry + before;
        __syncthreads();
        if (tid == 0) carry_s = carry + warp_sums[kPlanThreads / 32 - 1];
        __syncthreads();
    }
    const int64_t total = carry_s;
    if (tid == 0) p.req_prefix[p.B] = total;
    __syncthreads();
    const int64_t T = (int64_t)p.H * total;
    for (int w = tid; w < p.W; w += kPlanThreads) {
        const int64_t x = ((int64_t)w * T) / p.W;
        int lo = 0, hi = p.B - 1;   // largest b with H * prefix[b] <= x
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)p.H * p.req_prefix[mid] <= x) lo = mid; else hi = mid - 1;
        }
        p.worker_req[w] = lo;
    }
}

// ---------------------------------------------------------- split kernel --

// Position of a worker inside the flattened (request, head, tile) sequence.
struct Cursor {
    int b, h;
    int64_t tile;      // tile within the lane
    int64_t n;         // tiles of this lane
    int64_t first;     // H * prefix[b]
};

__device__ __forceinline__ void cursor_advance(Cursor& c, const KParams& p) {
    if (++c.tile < c.n) return;
    c.tile = 0;
    if (++c.h < p.H) return;
    c.h = 0;
    // next request with at least one tile
    int64_t pre = req_prefix_at(p, c.b + 1);
    while (c.b + 1 < p.B) {
        ++c.b;
        const int64_t nxt = req_prefix_at(p, c.b + 1);
        if (nxt > pre) {
            c.n = nxt - pre;
            c.first = (int64_t)p.H * pre;
            return;
        }
        pre = nxt;
    }
    c.b = p.B;   // past the end; never dereferenced
}

template <typename T, int D>
__device__ __forceinline__ int64_t tile_offset(const KParams& p, const Cursor& c, int32_t page) {
    const int64_t slot0 = (c.tile % p.tiles_per_page) * kTile;
    return (((int64_t)page * p.H + c.h) * p.P + slot0) * D;
}

__device__ __forceinline__ int32_t tile_page(const KParams& p, const Cursor& c) {
    return __ldg(p.tables + (int64_t)c.b * p.max_pages + c.tile / p.tiles_per_page);
}

template <typename T, int D>
__global__ void __launch_bounds__(kSplitWarps * 32)
split_decode_kernel(const KParams p) {
    using G = Geo<T, D>;
    using VT = typename VecBits<G::VBYTES>::type;
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * kSplitWarps + warp;
    if (w >= p.W) return;

    // this worker's tiles: [begin, end) of the flattened sequence
    const int64_t T_all = (int64_t)p.H * req_prefix_at(p, p.B);
    const int64_t begin = (w * T_all) / p.W;
    const int64_t end = ((w + 1) * T_all) / p.W;
    const int64_t n_work = end - begin;
    if (n_work <= 0) return;

    unsigned char* ring = smem + warp * G::WARP_SMEM;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSplitWarps * G::WARP_SMEM) + warp * G::STAGES;
    if (lane == 0) {
        for (int s = 0; s < G::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    Cursor cur;
    {
        const int b0 = p.seq_lens == nullptr ? 0 : __ldg(p.worker_req + w);
        const int64_t pre = req_prefix_at(p, b0);
        cur.b = b0;
        cur.n = req_prefix_at(p, b0 + 1) - pre;
        cur.first = (int64_t)p.H * pre;
        const int64_t local = begin - cur.first;
        cur.h = (int)(local / cur.n);
        cur.tile = local % cur.n;
    }
    Cursor prod = cur;
    const uint64_t policy = l2_evict_first_policy();

    // Producer step (lane 0): stage tile `prod` into stage s.
    auto issue = [&](int s) {
        if (lane != 0) return;
        const int32_t page = tile_page(p, prod);
        if (page < 0 || page >= p.n_pages) {
            atomicOr(p.err, PKV_DEVERR_PAGE_ID);
            mbar_arrive(&bars[s]);
            return;
        }
        const int64_t off = tile_offset<T, D>(p, prod, page);
        unsigned char* dst = ring + s * G::STAGE_BYTES;
        mbar_arrive_expect_tx(&bars[s], G::STAGE_BYTES);
        bulk_copy_g2s(dst, static_cast<const T*>(p.k_pages) + off, G::TILE_BYTES, &bars[s], policy);
        bulk_copy_g2s(dst + G::TILE_BYTES, static_cast<const T*>(p.v_pages) + off, G::TILE_BYTES,
                      &bars[s], policy);
    };

    const int prologue = n_work < G::STAGES ? (int)n_work : G::STAGES;
    for (int s = 0; s < prologue; ++s) {
        issue(s);
        cursor_advance(prod, p);
    }

    const int rg = lane / G::TPR;             // row group of this lane
    const int col = (lane % G::TPR) * G::VEC; // first feature of this lane

    float qv[G::VEC];
    float o[G::VEC];
    float m = -INFINITY, l = 0.f;
    int64_t piece_first = 0, t_b = 0;

    for (int64_t k = 0; k < n_work; ++k) {
        const int s = (int)(k % G::STAGES);
        const uint32_t parity = (uint32_t)((k / G::STAGES) & 1);
        const int64_t lane_id = (int64_t)cur.b * p.H + cur.h;

        if (k == 0 || cur.tile == 0) {   // a new lane piece starts
            piece_first = cur.tile;
            t_b = seq_len_at(p, cur.b);
            const float* qp = p.q + lane_id * D + col;
#pragma unroll
            for (int v = 0; v < G::VEC; ++v) {
                qv[v] = qp[v] * p.qscale;
                o[v] = 0.f;
            }
            m = -INFINITY;
            l = 0.f;
        }

        if (!mbar_wait_bounded(&bars[s], parity, kWaitLimitNs)) {
            if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
            // let the copies already issued land before the shared memory goes away
            const int64_t last = (k + G::STAGES - 1 < n_work - 1) ? k + G::STAGES - 1 : n_work - 1;
            for (int64_t j = k + 1; j <= last; ++j)
                mbar_wait_bounded(&bars[j % G::STAGES], (uint32_t)((j / G::STAGES) & 1), kWaitLimitNs);
            return;
        }

        T* Ks = reinterpret_cast<T*>(ring + s * G::STAGE_BYTES);
        T* Vs = Ks + kTile * D;
        const int32_t page = tile_page(p, cur);
        const bool page_ok = page >= 0 && page < p.n_pages;
        const bool last_tile = cur.tile == cur.n - 1;
        const int64_t rem = t_b - cur.tile * kTile;
        const int rows = !page_ok ? 0 : (rem < kTile ? (int)rem : kTile);

        if (last_tile && page_ok) {
            // fused append: row t_b - 1 comes from k_new / v_new, into the tile and the page
            const int r = rows - 1;
            if (lane < G::TPR) {
                const int64_t src = lane_id * D + col;
                const VT kb = *reinterpret_cast<const VT*>(static_cast<const T*>(p.k_new) + src);
                const VT vb = *reinterpret_cast<const VT*>(static_cast<const T*>(p.v_new) + src);
                *reinterpret_cast<VT*>(Ks + r * D + col) = kb;
                *reinterpret_cast<VT*>(Vs + r * D + col) = vb;
                const int64_t dst = tile_offset<T, D>(p, cur, page) + (int64_t)r * D + col;
                *reinterpret_cast<VT*>(static_cast<T*>(p.k_pages) + dst) = kb;
                *reinterpret_cast<VT*>(static_cast<T*>(p.v_pages) + dst) = vb;
            }
            __syncwarp();
        }

        if (rows > 0) {
            float sc[G::ITERS];
#pragma unroll
            for (int it = 0; it < G::ITERS; ++it) {
                const int row = it * G::RPI + rg;
                float acc = 0.f;
                if (row < kTile) {
                    float kf[G::VEC];
                    const VT kb = *reinterpret_cast<const VT*>(Ks + row * D + col);
                    Storage<T>::template to_float<G::VEC>(&kb, kf);
#pragma unroll
                    for (int v = 0; v < G::VEC; ++v) acc = fmaf(qv[v], kf[v], acc);
                }
                sc[it] = acc;
            }
#pragma unroll
            for (int it = 0; it < G::ITERS; ++it) {
#pragma unroll
                for (int off = G::TPR / 2; off >= 1; off >>= 1)
                    sc[it] += __shfl_xor_sync(0xffffffffu, sc[it], off);
            }
            float tmax = -INFINITY;
#pragma unroll
            for (int it = 0; it < G::ITERS; ++it) {
                const int row = it * G::RPI + rg;
                if (row >= rows) sc[it] = -INFINITY;
                tmax = fmaxf(tmax, sc[it]);
            }
#pragma unroll
            for (int off = G::TPR; off < 32; off <<= 1)
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            const float m_new = fmaxf(m, tmax);
            const float alpha = exp2f(m - m_new);
            l *= alpha;
#pragma unroll
            for (int v = 0; v < G::VEC; ++v) o[v] *= alpha;
#pragma unroll
            for (int it = 0; it < G::ITERS; ++it) {
                const int row = it * G::RPI + rg;
                if (row < rows) {
                    const float pw = exp2f(sc[it] - m_new);
                    l += pw;
                    float vf[G::VEC];
                    const VT vb = *reinterpret_cast<const VT*>(Vs + row * D + col);
                    Storage<T>::template to_float<G::VEC>(&vb, vf);
#pragma unroll
                    for (int v = 0; v < G::VEC; ++v) o[v] = fmaf(pw, vf[v], o[v]);
                }
            }
            m = m_new;
        }

        // the stage is free again: hand it to the copy engine for tile k + STAGES
        fence_proxy_async_smem();
        __syncwarp();
        if (k + G::STAGES < n_work) {
            issue(s);
            cursor_advance(prod, p);
        }

        if (last_tile || k == n_work - 1) {
            // close the lane piece: sum the row groups
            float lt = l;
#pragma unroll
            for (int off = G::TPR; off < 32; off <<= 1) {
                lt += __shfl_xor_sync(0xffffffffu, lt, off);
#pragma unroll
                for (int v = 0; v < G::VEC; ++v) o[v] += __shfl_xor_sync(0xffffffffu, o[v], off);
            }
            if (piece_first == 0 && last_tile) {
                if (lane < G::TPR) {
                    const float inv = 1.f / lt;
                    float* op = p.out + lane_id * D + col;
#pragma unroll
                    for (int v = 0; v < G::VEC; ++v) op[v] = o[v] * inv;
                }
            } else {
                const int64_t slot = lane_id + w;
                if (lane < G::TPR) {
                    float* op = p.part_o + slot * D + col;
#pragma unroll
                    for (int v = 0; v < G::VEC; ++v) op[v] = o[v];
                }
                if (lane == 0) p.part_ml[slot] = make_float2(m, lt);
            }
        }
        cursor_advance(cur, p);
    }
}

// ---------------------------------------------------------- merge kernel --

constexpr int kMergeWarps = 8;

// One warp per lane.  Lane (b, h) covers flattened tiles [A, A + n); tile x
// belongs to worker floor(((x + 1) W - 1) / T) (the inverse of
// begin(w) = floor(w T / W)).  A lane covered by one worker is already final.
// When T < W some workers own no tile; those between the lane's first and last
// worker wrote nothing and are skipped.  Partial slots lane + w are disjoint
// across lanes because the first worker of lane i + 1 is at least the last
// worker of lane i.
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const KParams p) {
    constexpr int DPL = D >= 32 ? D / 32 : 1;   // features per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t lane_id = (int64_t)blockIdx.x * kMergeWarps + warp;
    if (lane_id >= (int64_t)p.B * p.H) return;
    const int b = (int)(lane_id / p.H), h = (int)(lane_id % p.H);
    const int64_t pre = req_prefix_at(p, b);
    const int64_t n = req_prefix_at(p, b + 1) - pre;
    if (n <= 0) return;
    const int64_t T_all = (int64_t)p.H * req_prefix_at(p, p.B);
    const int64_t A = (int64_t)p.H * pre + (int64_t)h * n;
    const int64_t w_lo = ((A + 1) * p.W - 1) / T_all;
    const int64_t w_hi = ((A + n) * p.W - 1) / T_all;
    if (w_lo == w_hi) return;

    auto owns_tiles = [&](int64_t w) { return (w * T_all) / p.W != ((w + 1) * T_all) / p.W; };
    float M = -INFINITY;
    for (int64_t w = w_lo + lane; w <= w_hi; w += 32)
        if (owns_tiles(w)) M = fmaxf(M, p.part_ml[lane_id + w].x);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

    float L = 0.f;
    for (int64_t w = w_lo + lane; w <= w_hi; w += 32) {
        if (!owns_tiles(w)) continue;
        const float2 ml = p.part_ml[lane_id + w];
        L += ml.y * exp2f(ml.x - M);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);

    if (lane * DPL >= D) return;
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    for (int64_t w = w_lo; w <= w_hi; ++w) {
        if (!owns_tiles(w)) continue;
        const int64_t slot = lane_id + w;
        const float sc = exp2f(p.part_ml[slot].x - M);
        const float* op = p.part_o + slot * D + lane * DPL;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = fmaf(sc, op[i], acc[i]);
    }
    const float inv = 1.f / L;
    float* out = p.out + lane_id * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) out[i] = acc[i] * inv;
}

// ------------------------------------------------------------------ host --

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WorkspaceLayout workspace_layout(int B, int H, int D, int workers) {
    WorkspaceLayout L{};
    size_t off = 0;
    L.req_prefix = off;
    off = align_up(off + sizeof(int64_t) * ((size_t)B + 1), 256);
    L.worker_req = off;
    off = align_up(off + sizeof(int32_t) * (size_t)workers, 256);
    const size_t slots = (size_t)B * H + (size_t)workers;
    L.part_ml = off;
    off = align_up(off + sizeof(float2) * slots, 256);
    L.part_o = off;
    off = align_up(off + sizeof(float) * slots * (size_t)D, 256);
    L.total = off;
    return L;
}

int launch_workers(int pool_workers, int B, int H, int64_t max_seq_len) {
    const int64_t tiles = (int64_t)B * H * ((max_seq_len + kTile - 1) / kTile);
    return (int)(tiles < pool_workers ? (tiles < 1 ? 1 : tiles) : pool_workers);
}

template <typename T, int D>
static int split_smem() { return Geo<T, D>::CTA_SMEM; }

template <typename T, int D>
static cudaError_t prepare_split() {
    static bool done = false;   // per instantiation; attribute is per device-function
    if (done) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(split_decode_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Geo<T, D>::CTA_SMEM);
    if (e == cudaSuccess) done = true;
    return e;
}

template <typename T, int D>
static int resident_workers_t(int num_sms) {
    if (prepare_split<T, D>() != cudaSuccess) return 0;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, split_decode_kernel<T, D>,
                                                      kSplitWarps * 32, Geo<T, D>::CTA_SMEM) !=
        cudaSuccess)
        return 0;
    return blocks * num_sms * kSplitWarps;
}

template <typename T, int D>
static cudaError_t launch_t(const DecodeArgs& a, KParams& p, cudaStream_t stream) {
    cudaError_t e = prepare_split<T, D>();
    if (e != cudaSuccess) return e;
    if (a.seq_lens != nullptr) {
        plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int grid = (p.W + kSplitWarps - 1) / kSplitWarps;
    if (a.ev_before && (e = cudaEventRecord(a.ev_before, stream)) != cudaSuccess) return e;
    split_decode_kernel<T, D><<<grid, kSplitWarps * 32, Geo<T, D>::CTA_SMEM, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.ev_after && (e = cudaEventRecord(a.ev_after, stream)) != cudaSuccess) return e;
    const int64_t lanes = (int64_t)p.B * p.H;
    const int mgrid = (int)((lanes + kMergeWarps - 1) / kMergeWarps);
    merge_kernel<D><<<mgrid, kMergeWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

#define PKV_FOR_EACH_D(X, T) X(T, 2) X(T, 4) X(T, 8) X(T, 16) X(T, 32) X(T, 64) X(T, 128)

bool decode_supported(int dtype, int D) {
    if (D < 2 || D > 256 || (D & (D - 1)) != 0) return false;
    if (dtype == PKV_F32) return D <= 128;
    if (dtype == PKV_BF16) return D <= 256;
    return false;
}

int resident_workers(int dtype, int D, int num_sms) {
#define PKV_RW(T, DD) \
    if (D == DD) return resident_workers_t<T, DD>(num_sms);
    if (dtype == PKV_F32) {
        PKV_FOR_EACH_D(PKV_RW, float)
    } else if (dtype == PKV_BF16) {
        PKV_FOR_EACH_D(PKV_RW, __nv_bfloat16)
        PKV_RW(__nv_bfloat16, 256)
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
    p.max_pages = a.max_pages;
    p.seq_lens = a.seq_lens;
    p.single_t = a.single_t;
    p.single_tiles = (a.single_t + kTile - 1) / kTile;
    p.max_seq_len = a.max_seq_len;
    p.B = a.B;
    p.H = a.H;
    p.P = a.P;
    p.tiles_per_page = a.P / kTile;
    p.qscale = 1.4426950408889634f / sqrtf((float)a.D);
    p.out = a.out;
    const WorkspaceLayout L = workspace_layout(a.B, a.H, a.D, a.workers);
    unsigned char* ws = static_cast<unsigned char*>(a.workspace);
    p.req_prefix = reinterpret_cast<int64_t*>(ws + L.req_prefix);
    p.worker_req = reinterpret_cast<int32_t*>(ws + L.worker_req);
    p.part_ml = reinterpret_cast<float2*>(ws + L.part_ml);
    p.part_o = reinterpret_cast<float*>(ws + L.part_o);
    p.W = a.workers;
    p.err = a.dev_error;
#define PKV_LAUNCH(T, DD) \
    if (a.D == DD) return launch_t<T, DD>(a, p, stream);
    if (a.dtype == PKV_F32) {
        PKV_FOR_EACH_D(PKV_LAUNCH, float)
    } else if (a.dtype == PKV_BF16) {
        PKV_FOR_EACH_D(PKV_LAUNCH, __nv_bfloat16)
        PKV_LAUNCH(__nv_bfloat16, 256)
    }
#undef PKV_LAUNCH
    return cudaErrorInvalidValue;
}

}  // namespace pkv
