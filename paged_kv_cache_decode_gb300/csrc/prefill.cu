// Batched prefill into the paged KV cache, on the sm_103a tensor cores.
//
// What is computed ("Incremental Serving", section "Paged KV-cache layout": a
// batched prefill may run a FlashAttention-style tiled computation while it
// writes the same paged cache that paged decode attention reads).  Request b
// holds L0 = seq_lens[b] - n_b cached tokens and appends the n_b rows
// cu_new[b] .. cu_new[b+1]-1 of the batch.  Chunk token i sits at position
// L0 + i: its key and value rows are stored there, and its output is the
// softmax attention of its query over positions 0 .. L0 + i (the last `window`
// of them with a sliding window) -- what n_b successive decode steps give.
//
// Three launches per call:
//   1. plan (one CTA): validates lengths and lists the work units request by
//      request, the heaviest (last) unit of each request first;
//   2. append: copies every new key / value row into its page;
//   3. attention: one CTA per (work unit, KV head).
//
// Attention CTA.  A query tile is 128 rows: 128/G consecutive tokens times the
// G query heads that share one KV head, so every key tile serves all of them.
// A work unit is two consecutive query tiles, A and B, which share every K / V
// tile the CTA loads.  Key tiles are 128 positions, loaded as 8 groups of 16
// rows (a group never straddles a page) by TMA tensor copies with the 128-byte
// swizzle into a ring of slots, K and V of a tile in consecutive slots.  Per key
// tile and query tile:
//     S  = Q K^T               tcgen05.mma, M=128 N=128 K=d_h, fp32 in TMEM
//     P  = 2^(c S - c m)       softmax warps: TMEM -> registers -> bf16 hi + lo
//                              back into TMEM over the S columns already read
//     O += P_hi V + P_lo V     tcgen05.mma with A = P from TMEM, M=128 N=d_h K=128,
//                              twice: each weight carried to ~2^-16, not bf16's 2^-9
// with c = log2(e) / sqrt(d_h).  Warp roles (320 threads):
//   warps 0-3, 4-7  softmax of tiles A, B: warp w reads TMEM lanes 32(w%4) ..
//              32(w%4)+31, one query row per thread; they stage Q, write P,
//              rescale O and store the output;
//   warp 8     producer: eight lanes issue the K / V tile copies, one 16-row
//              group each;
//   warp 9     MMA: allocates TMEM, one thread issues the MMAs and commits.
// The MMA order P V_A(j), S_A(j+1), P V_B(j), S_B(j+1) ... keeps the tensor cores
// on one tile while the other tile's softmax runs.  MMAs of one thread run in
// issue order, so S_A(j+1) overwrites P_A(j) only after P V_A(j) has read it, and
// a commit after S_A(j+1) also covers P V_A(j): when tile A's softmax sees S it
// may rescale O_A.

// Exponent base.  Row m only moves when the row's maximum grows by more than 8
// in log2 units; O and the row sum l are then scaled by 2^(c (m_old - m_new)).
// Until then every weight is at most 2^8, which bf16 and the fp32 accumulators
// hold as well as any other; O / l uses the same m in both, so the result is the
// softmax whatever m is.
//
// Faults are not raised by trapping: bad lengths and page ids set bits of the
// device error word (a bad page reads as zeros), and a wait that runs out sets
// the timeout bit and ends the CTA's work; later CTAs of a pool whose error word
// holds the timeout bit return at once.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "pkv.h"
#include "pkv_internal.h"
#include "ptx.cuh"
#include "tc05.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;                  // query rows per tile = TMEM lanes
constexpr int kKeys = 128;                  // key positions per key tile
constexpr int kPfThreads = 320;             // 8 softmax warps, producer, MMA
constexpr int kPlanThreads = 1024;          // one request per plan thread
constexpr uint64_t kPfWaitLimitNs = kTcWaitLimitNs;

template <int D>
struct PfGeo {
    static constexpr int CHUNKS = D / 64;                    // 128-byte swizzle columns of Q, K, V
    static constexpr int COL_BYTES = kRows * 128;            // one such column of a 128-row tile
    static constexpr int Q_BYTES = CHUNKS * COL_BYTES;       // one query tile
    static constexpr int KV_BYTES = CHUNKS * kKeys * 128;    // one K or V tile = one ring slot
    static constexpr int BAR_BYTES = 256;
    static constexpr int FIXED = 1024 + 2 * Q_BYTES + BAR_BYTES;
    static constexpr int SLOTS_FIT = (227 * 1024 - FIXED) / KV_BYTES;
    static constexpr int SLOTS = SLOTS_FIT < 8 ? SLOTS_FIT : 8;
    static constexpr int SMEM = FIXED + SLOTS * KV_BYTES;
    static constexpr uint32_t S_COL = 0;                     // S of tiles A and B: columns 0, 128
    static constexpr uint32_t O_COL = 256;                   // O of tiles A and B: 256, 256 + D
    // P_hi and P_lo (bf16 pairs, 64 columns each) overwrite their tile's S columns
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(D == 64 || D == 128, "prefill: head width 64 or 128");
    static_assert(SLOTS >= 3, "ring too small");
    static_assert(SMEM <= 227 * 1024, "prefill CTA does not fit an SM");
    static_assert(2 * SLOTS * 8 + 7 * 8 + 8 <= BAR_BYTES, "barrier area");
};

struct PfParams {
    int B, H, G, P, max_pages;
    int64_t window;
    int64_t n_pages;
    int pool_rows;                 // rows of one layer's 2-D pool view (pages * H * P)
    const __nv_bfloat16* q;        // [N][H*G][D]
    const __nv_bfloat16* k_new;    // [N][H][D]
    const __nv_bfloat16* v_new;
    __nv_bfloat16* k_pages;        // [pages][H][P][D]
    __nv_bfloat16* v_pages;
    const int32_t* cu_new;         // [B + 1]; nullptr: one request of single_n rows
    const int32_t* seq_lens;       // [B]; nullptr: single_t
    int single_n;
    int64_t single_t;
    const int32_t* tables;         // [B][max_pages]
    float* out;                    // [N][H*G][D]
    int2* items;                   // query tiles (request, tile), in launch order
    int* n_items;
    int max_items;                 // capacity of items (the launch's CTAs / H)
    int64_t total_new;             // N
    float scale_log2;              // log2(e) / sqrt(D)
    unsigned* dev_error;
};

// Row offset of request b's chunk and its length after the chunk.
__device__ __forceinline__ int cu_at(const PfParams& p, int b) {
    return p.cu_new ? p.cu_new[b] : (b == 0 ? 0 : p.single_n);
}

__device__ __forceinline__ int64_t seq_len_at(const PfParams& p, int b) {
    return p.seq_lens ? (int64_t)p.seq_lens[b] : p.single_t;
}

// ------------------------------------------------------------------ plan --

__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const PfParams p) {
    __shared__ int warp_sum[kPlanThreads / 32];
    const int b = threadIdx.x;
    const int T = 2 * kRows / p.G;                // tokens of one work unit (two query tiles)
    int tiles = 0;
    if (b < p.B) {
        const int c0 = cu_at(p, b), c1 = cu_at(p, b + 1);
        const int64_t n = (int64_t)c1 - c0;
        const int64_t t = seq_len_at(p, b);
        const bool ok = c0 >= 0 && n >= 0 && c1 <= p.total_new && t - n >= 0 &&
                        t <= (int64_t)p.max_pages * p.P;
        if (!ok) atomicOr(p.dev_error, PKV_DEVERR_SEQ_LEN);
        else tiles = (int)((n + T - 1) / T);
    }
    // exclusive prefix of tiles over requests
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += v;
        }
        warp_sum[lane] = w;               // inclusive over warps
    }
    __syncthreads();
    const int first = (warp > 0 ? warp_sum[warp - 1] : 0) + incl - tiles;
    // requests whose row ranges overlap can hold more tiles than the launch has CTAs for
    const int total = warp_sum[kPlanThreads / 32 - 1];
    if (total > p.max_items && threadIdx.x == 0) atomicOr(p.dev_error, PKV_DEVERR_SEQ_LEN);
    for (int k = 0; k < tiles && first + k < p.max_items; ++k)
        p.items[first + k] = make_int2(b, tiles - 1 - k);
    if (threadIdx.x == 0) *p.n_items = total < p.max_items ? total : p.max_items;
}

// ---------------------------------------------------------------- append --

// Every new key / value row into its page: one thread per 16-byte piece.
template <int D>
__global__ void __launch_bounds__(256) prefill_append_kernel(const PfParams p) {
    constexpr int U = D / 8;
    const int64_t total = p.total_new * p.H * U;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t x = idx / (p.H * U);
        const int rem = (int)(idx - x * p.H * U);
        const int h = rem / U, u = rem - (rem / U) * U;
        int lo = 0, hi = p.B;                       // last request with cu_new[b] <= x
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu_at(p, mid) <= x) lo = mid;
            else hi = mid;
        }
        const int b = lo;
        const int c0 = cu_at(p, b), c1 = cu_at(p, b + 1);
        if (x < c0 || x >= c1) continue;
        const int64_t t = seq_len_at(p, b);
        const int64_t L0 = t - (c1 - c0);
        if (L0 < 0 || t > (int64_t)p.max_pages * p.P) continue;      // the plan reports it
        const int64_t pos = L0 + (x - c0);
        const int32_t page = p.tables[(int64_t)b * p.max_pages + pos / p.P];
        if (page < 0 || page >= p.n_pages) {
            atomicOr(p.dev_error, PKV_DEVERR_PAGE_ID);
            continue;
        }
        const int64_t dst = (((int64_t)page * p.H + h) * p.P + pos % p.P) * D + u * 8;
        const int64_t src = (x * p.H + h) * D + u * 8;
        *reinterpret_cast<uint4*>(p.k_pages + dst) = *reinterpret_cast<const uint4*>(p.k_new + src);
        *reinterpret_cast<uint4*>(p.v_pages + dst) = *reinterpret_cast<const uint4*>(p.v_new + src);
    }
}

// ------------------------------------------------------------- attention --

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1)
prefill_attention_kernel(const __grid_constant__ PfParams p, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
    using M = PfGeo<D>;
    const int item = blockIdx.x / p.H;
    const int h = blockIdx.x - item * p.H;
    if (item >= *p.n_items) return;
    if (*reinterpret_cast<volatile unsigned*>(p.dev_error) & PKV_DEVERR_TIMEOUT) return;

    const int2 it = p.items[item];
    const int b = it.x, unit = it.y;
    const int G = p.G, T = kRows / G;                         // tokens per query tile
    const int c0 = cu_at(p, b);
    const int n = cu_at(p, b + 1) - c0;
    const int64_t t_b = seq_len_at(p, b);
    const int64_t L0 = t_b - n;
    const int i0 = unit * 2 * T;                              // tile A: tokens i0 .. i0+T-1
    const int i_end = min(n, i0 + 2 * T);                     // the unit's tokens end here
    const int64_t pos_last = L0 + i_end - 1;
    const int64_t lo_first =
        p.window > 0 ? (L0 + i0 - p.window + 1 > 0 ? L0 + i0 - p.window + 1 : 0) : 0;
    const int64_t kt0 = lo_first / kKeys;
    const int ntiles = (int)(pos_last / kKeys - kt0 + 1);

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* Qs = sm;                                   // tiles A, B
    unsigned char* ring = Qs + 2 * M::Q_BYTES;                // SLOTS K or V tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + M::SLOTS * M::KV_BYTES);
    uint64_t* slot_full = bars;                  // per slot: copy landed
    uint64_t* slot_empty = bars + M::SLOTS;      //           MMAs reading it done
    uint64_t* s_full = bars + 2 * M::SLOTS;      // per tile A, B: S computed
    uint64_t* p_full = s_full + 2;               //                P written
    uint64_t* o_done = p_full + 2;               // last P V of both tiles done
    uint64_t* q_ready = o_done + 1;
    uint64_t* drain = q_ready + 1;               // MMA completion on the abort path
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < M::SLOTS; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 128);
        }
        mbar_init(o_done, 1);
        mbar_init(q_ready, 256);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) tmem_alloc(tmem_slot, M::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 8) {
        // ------------------------------------------------------ softmax --
        const int x = warp >> 2;                              // query tile A (0) or B (1)
        const int r = threadIdx.x & 127;                      // row of the tile = TMEM lane
        const int g = r % G;
        const int i = i0 + x * T + r / G;
        const bool valid = i < i_end;
        const int HQ = p.H * G;
        const int64_t row_x = (int64_t)c0 + i;
        const int qh = h * G + g;
        unsigned char* Qx = Qs + x * M::Q_BYTES;
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.q + (row_x * HQ + qh) * D);
#pragma unroll
            for (int u = 0; u < D / 8; ++u) {
                const uint4 v = valid ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(Qx + sw_off(r, u)) = v;
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(q_ready);

        const int64_t pos = L0 + i;
        const int64_t hi = valid ? pos : -1;                  // keys lo .. hi
        const int64_t lo = p.window > 0 ? (pos - p.window + 1 > 0 ? pos - p.window + 1 : 0) : 0;
        const float c = p.scale_log2;
        const uint32_t t_s = tmem + ((uint32_t)((warp & 3) * 32) << 16) + M::S_COL + x * kKeys;
        const uint32_t t_o = tmem + ((uint32_t)((warp & 3) * 32) << 16) + M::O_COL + x * D;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            if (!pf_warp_wait(&s_full[x], j & 1, abort_flag, p.dev_error)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // keys e_lo .. e_hi of the tile are this row's (none when e_lo > e_hi)
            const int64_t k0 = (kt0 + j) * kKeys;
            const bool full = k0 >= lo && k0 + kKeys - 1 <= hi;
            const int e_lo = full ? 0 : (int)(lo - k0 > 0 ? (lo - k0 < kKeys ? lo - k0 : kKeys) : 0);
            const int e_hi = full ? kKeys - 1
                                  : (int)(hi - k0 < kKeys - 1 ? (hi - k0 > -1 ? hi - k0 : -1)
                                                              : kKeys - 1);
            // The tile's row maximum first, from 1.5 reads of S: keys 64..127 for their
            // maximum only, then keys 0..63 kept in registers.  With m settled (and O
            // rescaled if it moved), the weights 2^(c s - c m) of keys 0..63 from those
            // registers, then of keys 64..127 from a second read.  Each weight w is
            // split into bf16 hi = rn(w) and lo = rn(w - hi) (w - hi is exact in fp32),
            // so P_hi V + P_lo V carries w to about 2^-16 instead of bf16's 2^-9.  The
            // pairs go back over the S columns of their own half, already read: keys
            // 64hh + 2i, 2i+1 -> P_hi column 64hh + i, P_lo column 64hh + 32 + i.
            const float2 c2 = make_float2(c, c);
            float m2[2] = {-INFINITY, -INFINITY};
            {
                uint32_t sv[64];
                tmem_ld32(t_s + 64, sv);
                tmem_ld32(t_s + 96, sv + 32);
                tmem_wait_ld();
                if (!full) {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (64 + e < e_lo || 64 + e > e_hi) sv[e] = 0xff800000u;
                }
#pragma unroll
                for (int e = 0; e < 64; e += 4) {
                    m2[0] = fmax3(m2[0], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                    m2[1] = fmax3(m2[1], __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]));
                }
            }
            uint32_t s0[64];                                  // S of keys 0..63
            tmem_ld32(t_s, s0);
            tmem_ld32(t_s + 32, s0 + 32);
            tmem_wait_ld();
            if (!full) {
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    if (e < e_lo || e > e_hi) s0[e] = 0xff800000u;
            }
#pragma unroll
            for (int e = 0; e < 64; e += 4) {
                m2[0] = fmax3(m2[0], __uint_as_float(s0[e]), __uint_as_float(s0[e + 1]));
                m2[1] = fmax3(m2[1], __uint_as_float(s0[e + 2]), __uint_as_float(s0[e + 3]));
            }
            const float mx = fmaxf(m2[0], m2[1]);
            float alpha = 1.f;
            if (mx > m_used && (m_used == -INFINITY || (mx - m_used) * c > 8.f)) {
                alpha = m_used == -INFINITY ? 0.f : ex2((m_used - mx) * c);
                m_used = mx;
                l *= alpha;
            }
            // S of this tile was committed after P V of the previous one, so that P V
            // is complete: O may be rescaled
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    tmem_ld32(t_o + cc * 32, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    tmem_st32(t_o + cc * 32, ov);
                }
                tmem_wait_st();
            }
            const float mb = m_used == -INFINITY ? 0.f : m_used * c;
            const float2 nmb2 = make_float2(-mb, -mb);
            float2 acc[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) acc[k] = make_float2(0.f, 0.f);
            // weights of 64 keys -> 32 P_hi pairs at column `col`, 32 P_lo pairs at col + 32
            auto weights = [&](const uint32_t* sv, uint32_t col) {
                uint32_t phi[32], plo[32];
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 xe = __ffma2_rn(
                        make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, nmb2);
                    const float2 pr = make_float2(ex2(xe.x), ex2(xe.y));
                    acc[(e >> 1) & 1] = __fadd2_rn(acc[(e >> 1) & 1], pr);
                    const __nv_bfloat162 hb = __floats2bfloat162_rn(pr.x, pr.y);
                    const __nv_bfloat162 lb =
                        __floats2bfloat162_rn(pr.x - __low2float(hb), pr.y - __high2float(hb));
                    phi[e >> 1] = *reinterpret_cast<const uint32_t*>(&hb);
                    plo[e >> 1] = *reinterpret_cast<const uint32_t*>(&lb);
                }
                tmem_st32(t_s + col, phi);
                tmem_st32(t_s + col + 32, plo);
            };
            weights(s0, 0);
            {
                uint32_t sv[64];
                tmem_ld32(t_s + 64, sv);
                tmem_ld32(t_s + 96, sv + 32);
                tmem_wait_ld();
                if (!full) {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (64 + e < e_lo || 64 + e > e_hi) sv[e] = 0xff800000u;
                }
                weights(sv, 64);
            }
            tmem_wait_st();
            const float2 a = __fadd2_rn(acc[0], acc[1]);
            l += a.x + a.y;
            tc_fence_before();
            mbar_arrive(&p_full[x]);
        }
        if (ok && pf_warp_wait(o_done, 0, abort_flag, p.dev_error)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float4* dst = reinterpret_cast<float4*>(p.out + (row_x * HQ + qh) * D);
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                tmem_ld32(t_o + cc * 32, ov);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        dst[(cc * 32 + e) / 4] = make_float4(
                            __uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv,
                            __uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
                }
            }
        }
    } else if (warp == 8) {
        // ----------------------------------------------------- producer --
        // loads in order: K of tile j is load 2j, V of tile j load 2j+1, into slot
        // load % SLOTS once the MMAs that read the slot's previous tile are done.
        // Lane gi < 8 looks up the page of the tile's 16-row group gi and issues its
        // boxes; lane 0 arms the slot's barrier first.
        const uint64_t pol = l2_normal_policy();
        const int32_t* table = p.tables + (int64_t)b * p.max_pages;
        const int gi = lane & 7;
        int issued = 0;
        bool aborted = false;
        for (int j = 0; j < ntiles && !aborted; ++j) {
            const int64_t key = (kt0 + j) * kKeys + 16 * gi;
            int y = p.pool_rows;                                    // past the pool: reads zeros
            if (lane < 8 && key <= pos_last) {
                const int32_t page = table[key / p.P];
                if (page >= 0 && page < p.n_pages)
                    y = (int)(((int64_t)page * p.H + h) * p.P + key % p.P);
                else
                    atomicOr(p.dev_error, PKV_DEVERR_PAGE_ID);
            }
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                const int ld = 2 * j + kv, s = ld % M::SLOTS;
                if (ld >= M::SLOTS && !pf_warp_wait(&slot_empty[s], ((ld / M::SLOTS) - 1) & 1,
                                                    abort_flag, p.dev_error)) {
                    aborted = true;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&slot_full[s], M::KV_BYTES);
                __syncwarp();
                if (lane < 8) {
                    unsigned char* dst = ring + s * M::KV_BYTES + gi * 2048;
                    const CUtensorMap* map = kv ? &tmv : &tmk;
#pragma unroll
                    for (int cc = 0; cc < M::CHUNKS; ++cc)
                        tma_load_2d(dst + cc * kKeys * 128, map, cc * 64, y, &slot_full[s], pol);
                }
                ++issued;
            }
        }
        if (lane == 0 && (aborted || *abort_flag)) {
            // let the copies in flight land before the CTA's shared memory goes away
            for (int ld = issued - M::SLOTS > 0 ? issued - M::SLOTS : 0; ld < issued; ++ld)
                mbar_wait_bounded(&slot_full[ld % M::SLOTS], (ld / M::SLOTS) & 1, kPfWaitLimitNs);
        }
    } else {
        // ---------------------------------------------------------- MMA --
        // S_A(0) S_B(0) | P V_A(j) S_A(j+1) P V_B(j) S_B(j+1) | ... : while one
        // tile's softmax runs, the tensor cores work on the other tile
        constexpr uint32_t idS = idesc_bf16(kKeys, false);
        constexpr uint32_t idO = idesc_bf16(D, true);
        // V is MN-major: 64-column swizzle atoms kKeys * 128 bytes apart, 8-row groups
        // 1024 bytes apart.  With D = 64 there is a single atom column, and the atom
        // stride is set equal to the group stride.
        constexpr uint32_t kVLbo = D == 64 ? 1024u : (uint32_t)(kKeys * 128);
        const uint32_t q_addr = smem_u32(Qs), ring_addr = smem_u32(ring);
        auto wait_slot = [&](int ld) {
            return pf_warp_wait(&slot_full[ld % M::SLOTS], (ld / M::SLOTS) & 1, abort_flag,
                                p.dev_error);
        };
        // descriptors are built once per group: a k-step only moves the start address,
        // by a constant (shared-memory addresses stay below 2^18, so no field overflows)
        auto issue_s = [&](int j, int x) {
            const uint32_t k_addr = ring_addr + ((2 * j) % M::SLOTS) * M::KV_BYTES;
            const uint64_t da = sw128_desc(q_addr + x * M::Q_BYTES, 16, 1024);
            const uint64_t db = sw128_desc(k_addr, 16, 1024);
            const uint32_t d = tmem + M::S_COL + x * kKeys;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint64_t dk = (uint64_t)(((k >> 2) * (kRows * 128) + (k & 3) * 32) >> 4);
                umma_bf16(d, da + dk, db + dk, idS, k > 0);
            }
            umma_commit(&s_full[x]);
        };
        auto issue_pv = [&](int j, int x) {
            const uint32_t v_addr = ring_addr + ((2 * j + 1) % M::SLOTS) * M::KV_BYTES;
            const uint64_t dv = sw128_desc(v_addr, kVLbo, 1024);
            // P in TMEM: keys 16k .. 16k+15 are P_hi columns 64(k/4) + 8(k%4) .. +7 and the
            // P_lo columns 32 further on
            const uint32_t pa = tmem + M::S_COL + x * kKeys;
            const uint32_t o = tmem + M::O_COL + x * D;
#pragma unroll
            for (int k = 0; k < kKeys / 16; ++k) {
                const uint64_t dvk = dv + (uint64_t)((k * 16 * 128) >> 4);
                const uint32_t ph = pa + (k >> 2) * 64 + (k & 3) * 8;
                umma_bf16_tmem_a(o, ph, dvk, idO, (j > 0 || k > 0) ? 1u : 0u);
                umma_bf16_tmem_a(o, ph + 32, dvk, idO, 1u);
            }
        };
        bool ok = pf_warp_wait(q_ready, 0, abort_flag, p.dev_error) && wait_slot(0);
        bool issued_any = false;
        if (ok) {
            tc_fence_after();
            if (lane == 0) {
                issue_s(0, 0);
                issue_s(0, 1);
                umma_commit(&slot_empty[0]);
            }
            issued_any = true;
            __syncwarp();
        }
        for (int j = 0; ok && j < ntiles; ++j) {
            const bool more = j + 1 < ntiles;
            if (!pf_warp_wait(&p_full[0], j & 1, abort_flag, p.dev_error) || !wait_slot(2 * j + 1)) {
                ok = false;
                break;
            }
            if (j == ntiles - 1) {
                // rows at positions >= t_b of the last loaded group hold stale bytes,
                // possibly not finite: clear them in V (their weights are 0)
                unsigned char* Vs = ring + ((2 * j + 1) % M::SLOTS) * M::KV_BYTES;
                const int64_t k0 = (kt0 + j) * kKeys;
                const int r0 = (int)(t_b - k0);
                const int r1 = (int)(((pos_last - k0) / 16 + 1) * 16);
                for (int idx = lane; idx < (r1 - r0) * M::CHUNKS * 8; idx += 32) {
                    const int row = r0 + idx / (M::CHUNKS * 8);
                    const int piece = idx % (M::CHUNKS * 8);
                    *reinterpret_cast<uint4*>(Vs + (piece >> 3) * kKeys * 128 + row * 128 +
                                              (piece & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) issue_pv(j, 0);
            __syncwarp();
            if (more) {
                if (!wait_slot(2 * j + 2)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) issue_s(j + 1, 0);
                __syncwarp();
            }
            if (!pf_warp_wait(&p_full[1], j & 1, abort_flag, p.dev_error)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                issue_pv(j, 1);
                umma_commit(&slot_empty[(2 * j + 1) % M::SLOTS]);
                if (more) {
                    issue_s(j + 1, 1);
                    umma_commit(&slot_empty[(2 * j + 2) % M::SLOTS]);
                } else {
                    umma_commit(o_done);
                }
            }
            __syncwarp();
        }
        if (issued_any && *abort_flag) {
            // MMAs still in flight read shared memory and write TMEM: let them finish
            if (lane == 0) {
                umma_commit(drain);
                mbar_wait_bounded(drain, 0, kPfWaitLimitNs);
            }
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, M::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host --

template <int D>
cudaError_t launch_prefill_t(const PrefillArgs& a, const PfParams& p, cudaStream_t stream) {
    using M = PfGeo<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_attention_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, M::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
    const int64_t pieces = a.total_new * a.H * (D / 8);
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (pieces + 255) / 256;
    const int append_blocks = (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
    prefill_append_kernel<D><<<append_blocks, 256, 0, stream>>>(p);
    const int64_t blocks = prefill_max_tiles(a.B, a.G, a.total_new) * a.H;
    CUtensorMap tmk, tmv;
    std::memcpy(&tmk, a.tmap_k, sizeof tmk);
    std::memcpy(&tmv, a.tmap_v, sizeof tmv);
    if (a.ev_before) cudaEventRecord(a.ev_before, stream);
    prefill_attention_kernel<D><<<(unsigned)blocks, kPfThreads, M::SMEM, stream>>>(p, tmk, tmv);
    if (a.ev_after) cudaEventRecord(a.ev_after, stream);
    return cudaGetLastError();
}

}  // namespace

int64_t prefill_max_tiles(int B, int G, int64_t total_new) {
    return total_new / (2 * kRows / G) + B;
}

size_t prefill_workspace_bytes(int B, int G, int64_t total_new) {
    return 256 + (size_t)prefill_max_tiles(B, G, total_new) * sizeof(int2);
}

bool prefill_supported(int dtype, int D, int G) {
    return dtype == PKV_BF16 && (D == 64 || D == 128) && G >= 1 && G <= kRows && kRows % G == 0;
}

int prefill_max_batch() { return kPlanThreads; }

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    PfParams p{};
    p.B = a.B;
    p.H = a.H;
    p.G = a.G;
    p.P = a.P;
    p.max_pages = a.max_pages;
    p.window = a.window;
    p.n_pages = a.n_pages;
    p.pool_rows = (int)(a.n_pages * a.H * a.P);
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
    p.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
    p.k_pages = static_cast<__nv_bfloat16*>(a.k_pages);
    p.v_pages = static_cast<__nv_bfloat16*>(a.v_pages);
    p.cu_new = a.cu_new;
    p.seq_lens = a.seq_lens;
    p.single_n = (int)a.single_n;
    p.single_t = a.single_t;
    p.tables = a.tables;
    p.out = a.out;
    p.n_items = static_cast<int*>(a.workspace);
    p.max_items = (int)prefill_max_tiles(a.B, a.G, a.total_new);
    p.items = reinterpret_cast<int2*>(static_cast<char*>(a.workspace) + 256);
    p.total_new = a.total_new;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a.D));
    p.dev_error = a.dev_error;
    switch (a.D) {
        case 64: return launch_prefill_t<64>(a, p, stream);
        case 128: return launch_prefill_t<128>(a, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
