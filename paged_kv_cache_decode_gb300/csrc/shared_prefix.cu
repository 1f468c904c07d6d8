// Shared-prefix decode attention: the shared part, on the sm_103a tensor cores.
//
// What is computed.  In a batch whose requests all map their first S positions
// to the same physical pages (a prompt shared by forked requests; "Incremental
// Serving", section "Current scope", names page sharing between requests), the
// decode attention of every query splits exactly into the S shared keys and the
// request's own keys S .. t_b - 1:
//     out = (2^(m1-M) o1 + 2^(m2-M) o2) / (2^(m1-M) l1 + 2^(m2-M) l2),  M = max(m1, m2),
// where (m, l, o) are the running maximum (log2 units), sum and unnormalised
// output of a softmax over each part.  This kernel computes the shared part for
// all requests at once: per KV head, the rows (request, query head) of the batch
// against the S shared keys read once — a dense contraction, run as tcgen05 MMAs.
// The split decode kernel then runs over positions S .. t_b - 1 only and merges
// these partials into its result.
//
// Work: one CTA per (KV head, tile of 128 rows, key split).  The rows of a tile
// are 128/G requests times the G query heads of the KV head.  A key split is a
// range of whole 128-key tiles of the shared prefix, so the grid fills the GPU
// once.  Each CTA writes one partial (m, l, o[d_h]) per row.
//
// Precision.  The decode query is fp32 and the decode path is held to fp32-level
// accuracy, so q is split into bf16 hi + lo (S = Q_hi K^T + Q_lo K^T) and the
// softmax weights likewise (O += P_hi V + P_lo V): each product then carries the
// fp32 value to ~2^-16.
//
// Per key tile j (128 keys), with S double-buffered in TMEM:
//     S(j)  = Q_hi K_j^T + Q_lo K_j^T          16 MMAs, M=128 N=128 K=16, fp32 in TMEM
//     P(j)  = 2^(c S - c m) -> P_hi, P_lo       softmax warps, bf16 pairs back into
//                                               the S(j) columns (P_hi 0-63, P_lo 64-127)
//     O    += P_hi V_j + P_lo V_j               16 MMAs, A from TMEM, B = V MN-major
// MMA order S(0) | S(j+1), P V(j) | ...: S of the next tile runs while the
// softmax works on this one.  Warp roles (192 threads): warps 0-3 softmax (one
// row per thread), warp 4 producer (eight lanes issue the TMA copies of one
// 16-row group each), warp 5 MMA (TMEM allocation, one issuing thread).
//
// Faults are not raised by trapping: a wait that runs out sets the timeout bit
// of the device error word and ends the CTA's work.

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

constexpr int kSpRows = 128;                 // rows per tile = TMEM lanes
constexpr int kSpKeys = 128;                 // keys per key tile
constexpr int kSpThreads = 192;

template <int D>
struct SpGeo {
    static constexpr int CHUNKS = D / 64;
    static constexpr int Q_BYTES = CHUNKS * kSpRows * 128;   // one bf16 query tile (hi or lo)
    static constexpr int KV_BYTES = CHUNKS * kSpKeys * 128;  // one K or V tile = one ring slot
    static constexpr int BAR_BYTES = 256;
    static constexpr int FIXED = 1024 + 2 * Q_BYTES + BAR_BYTES;
    static constexpr int SLOTS_FIT = (227 * 1024 - FIXED) / KV_BYTES;
    static constexpr int SLOTS = SLOTS_FIT < 8 ? SLOTS_FIT : 8;
    static constexpr int SMEM = FIXED + SLOTS * KV_BYTES;
    static constexpr uint32_t S_COL = 0;                     // S buffers at columns 0 and 128
    static constexpr uint32_t O_COL = 256;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(D == 64 || D == 128, "shared prefix: head width 64 or 128");
    static_assert(SLOTS >= 4, "ring too small");
    static_assert(SMEM <= 227 * 1024, "CTA does not fit an SM");
    static_assert(2 * SLOTS * 8 + 10 * 8 + 8 <= BAR_BYTES, "barrier area");
};

struct SpParams {
    int B, H, G, P, max_pages;
    int64_t window;
    int64_t n_pages;
    int pool_rows;                   // rows of one layer's 2-D pool view (pages * H * P)
    const float* q;                  // [B][H*G][D] fp32
    const int32_t* tables;           // [B][max_pages]; request 0's row holds the prefix
    const int32_t* seq_lens;         // [B]
    int64_t shared_len;              // S, a multiple of the page size
    int64_t split_len;               // keys per split, a multiple of kSpKeys
    int row_tiles;
    float2* pre_ml;                  // [splits][B*H*G]
    float* pre_o;                    // [splits][B*H*G][D]
    float scale_log2;                // log2(e) / sqrt(D)
    unsigned* dev_error;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(kSpThreads, 1)
shared_prefix_kernel(const __grid_constant__ SpParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
    using M = SpGeo<D>;
    pdl_launch_dependents();            // the split kernel may launch; it waits for our writes
    if (*reinterpret_cast<volatile unsigned*>(p.dev_error) & PKV_DEVERR_TIMEOUT) return;
    const int h = blockIdx.x % p.H;
    const int rest = blockIdx.x / p.H;
    const int rt = rest % p.row_tiles;
    const int ks = rest / p.row_tiles;
    const int64_t k_begin = (int64_t)ks * p.split_len;
    const int64_t k_end = k_begin + p.split_len < p.shared_len ? k_begin + p.split_len : p.shared_len;
    const int ntiles = (int)((k_end - k_begin + kSpKeys - 1) / kSpKeys);
    const int G = p.G, HQ = p.H * G;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* Qhi = sm;
    unsigned char* Qlo = Qhi + M::Q_BYTES;
    unsigned char* ring = Qlo + M::Q_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + M::SLOTS * M::KV_BYTES);
    uint64_t* slot_full = bars;
    uint64_t* slot_empty = bars + M::SLOTS;
    uint64_t* s_full = bars + 2 * M::SLOTS;      // per S buffer
    uint64_t* p_full = s_full + 2;               // per S buffer (the softmax may run a tile ahead)
    uint64_t* pv_done = p_full + 2;              // per S buffer: P V of tiles b, b+2, ... done
    uint64_t* o_done = pv_done + 2;              // the last P V
    uint64_t* q_ready = o_done + 1;
    uint64_t* drain = q_ready + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < M::SLOTS; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
        }
        mbar_init(&pv_done[0], 1);
        mbar_init(&pv_done[1], 1);
        mbar_init(o_done, 1);
        mbar_init(q_ready, 128);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(tmem_slot, M::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        // ------------------------------------------------------ softmax --
        const int r = threadIdx.x;                            // row = TMEM lane
        const int b = rt * (kSpRows / G) + r / G;
        const int g = r % G;
        const bool valid = b < p.B;
        const int64_t row = (int64_t)b * HQ + h * G + g;      // query row of the batch
        {
            // q (fp32) -> bf16 hi + lo, 128-byte swizzled, K-major
            const float4* src = reinterpret_cast<const float4*>(p.q + row * D);
#pragma unroll
            for (int u = 0; u < D / 8; ++u) {
                float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
                if (valid) {
                    x0 = __ldg(src + 2 * u);
                    x1 = __ldg(src + 2 * u + 1);
                }
                const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 hb = __floats2bfloat162_rn(xs[2 * k], xs[2 * k + 1]);
                    hi[k] = *reinterpret_cast<const uint32_t*>(&hb);
                    lo[k] = pack_bf16x2(xs[2 * k] - __low2float(hb), xs[2 * k + 1] - __high2float(hb));
                }
                *reinterpret_cast<uint4*>(Qhi + sw_off(r, u)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(Qlo + sw_off(r, u)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(q_ready);
        if (valid && g == 0 && b > 0) {
            // the prefix pages of this split must be request 0's in every request
            const int64_t pg0 = k_begin / p.P, pg1 = (k_end + p.P - 1) / p.P;
            bool differs = false;
            for (int64_t j = pg0; j < pg1; ++j)
                differs |= __ldg(p.tables + (int64_t)b * p.max_pages + j) != __ldg(p.tables + j);
            if (differs) atomicOr(p.dev_error, PKV_DEVERR_SHARED);
        }

        const int64_t t_b = valid ? (int64_t)p.seq_lens[b] : 0;
        const int64_t lo = p.window > 0 ? (t_b - p.window > 0 ? t_b - p.window : 0) : 0;
        const int64_t hi = valid ? k_end - 1 : -1;            // keys lo .. hi of this split
        const float c = p.scale_log2;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t t_o = tmem + lane_base + M::O_COL;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const uint32_t t_s = tmem + lane_base + M::S_COL + (j & 1) * kSpKeys;
            if (!pf_warp_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, p.dev_error)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int64_t k0 = k_begin + (int64_t)j * kSpKeys;
            const bool full = k0 >= lo && k0 + kSpKeys - 1 <= hi;
            const int e_lo = full ? 0 : (int)(lo - k0 > 0 ? (lo - k0 < kSpKeys ? lo - k0 : kSpKeys) : 0);
            const int e_hi = full ? kSpKeys - 1
                                  : (int)(hi - k0 < kSpKeys - 1 ? (hi - k0 > -1 ? hi - k0 : -1)
                                                                : kSpKeys - 1);
            // pass 1: row maximum over this row's keys, eight chains
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t sv[64];
                tmem_ld32(t_s + hh * 64, sv);
                tmem_ld32(t_s + hh * 64 + 32, sv + 32);
                tmem_wait_ld();
                if (!full) {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (hh * 64 + e < e_lo || hh * 64 + e > e_hi) sv[e] = 0xff800000u;
                }
#pragma unroll
                for (int e = 0; e < 64; ++e) m8[e & 7] = fmaxf(m8[e & 7], __uint_as_float(sv[e]));
            }
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            float alpha = 1.f;
            if (mx > m_used && (m_used == -INFINITY || (mx - m_used) * c > 8.f)) {
                alpha = m_used == -INFINITY ? 0.f : ex2((m_used - mx) * c);
                m_used = mx;
                l *= alpha;
            }
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // O holds P V of tiles 0 .. j-1 once P V(j-1) is complete.  Its barrier
                // cannot run a phase past it: the next, P V(j+1), needs P(j+1)
                if (!pf_warp_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag,
                                  p.dev_error)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
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
            // pass 2: weights, split into bf16 hi + lo, into TMEM over the S columns
            // already read: P_hi of keys 2i, 2i+1 -> column i, P_lo -> column 64 + i
            const float mb = m_used == -INFINITY ? 0.f : m_used * c;
            const float2 c2 = make_float2(c, c), nmb2 = make_float2(-mb, -mb);
            float2 acc[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.f, 0.f);
            uint32_t plo0[32];                                // P_lo of keys 0..63, stored last
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t sv[64];
                tmem_ld32(t_s + hh * 64, sv);
                tmem_ld32(t_s + hh * 64 + 32, sv + 32);
                tmem_wait_ld();
                if (!full) {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (hh * 64 + e < e_lo || hh * 64 + e > e_hi) sv[e] = 0xff800000u;
                }
                uint32_t phi[32], plo[32];
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 xe = __ffma2_rn(
                        make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, nmb2);
                    const float2 pr = make_float2(ex2(xe.x), ex2(xe.y));
                    acc[(e >> 1) & 3] = __fadd2_rn(acc[(e >> 1) & 3], pr);
                    const __nv_bfloat162 hb = __floats2bfloat162_rn(pr.x, pr.y);
                    phi[e >> 1] = *reinterpret_cast<const uint32_t*>(&hb);
                    plo[e >> 1] = pack_bf16x2(pr.x - __low2float(hb), pr.y - __high2float(hb));
                }
                tmem_st32(t_s + hh * 32, phi);
                if (hh == 0) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) plo0[k] = plo[k];
                } else {
                    tmem_st32(t_s + 64, plo0);
                    tmem_st32(t_s + 96, plo);
                }
            }
            tmem_wait_st();
            const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
            const float2 a = __fadd2_rn(a01, a23);
            l += a.x + a.y;
            tc_fence_before();
            mbar_arrive(&p_full[j & 1]);
        }
        if (ok && pf_warp_wait(o_done, 0, abort_flag, p.dev_error)) {
            tc_fence_after();
            const int64_t slot = (int64_t)ks * p.B * HQ + row;
            float4* dst = reinterpret_cast<float4*>(p.pre_o + slot * D);
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                tmem_ld32(t_o + cc * 32, ov);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        dst[(cc * 32 + e) / 4] =
                            make_float4(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1]),
                                        __uint_as_float(ov[e + 2]), __uint_as_float(ov[e + 3]));
                }
            }
            if (valid)
                p.pre_ml[slot] = l > 0.f ? make_float2(m_used * c, l) : make_float2(-INFINITY, 0.f);
        }
    } else if (warp == 4) {
        // ----------------------------------------------------- producer --
        // K of tile j is load 2j, V load 2j+1, into slot load % SLOTS; lane gi < 8
        // issues the boxes of 16-row group gi (the prefix pages are request 0's)
        const uint64_t pol = l2_normal_policy();
        const int gi = lane & 7;
        int issued = 0;
        bool aborted = false;
        for (int j = 0; j < ntiles && !aborted; ++j) {
            const int64_t key = k_begin + (int64_t)j * kSpKeys + 16 * gi;
            int y = p.pool_rows;                                    // past the pool: reads zeros
            if (lane < 8 && key < k_end) {
                const int32_t page = p.tables[key / p.P];
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
                        tma_load_2d(dst + cc * kSpKeys * 128, map, cc * 64, y, &slot_full[s], pol);
                }
                ++issued;
            }
        }
        if (lane == 0 && (aborted || *abort_flag)) {
            for (int ld = issued - M::SLOTS > 0 ? issued - M::SLOTS : 0; ld < issued; ++ld)
                mbar_wait_bounded(&slot_full[ld % M::SLOTS], (ld / M::SLOTS) & 1, kTcWaitLimitNs);
        }
    } else {
        // ---------------------------------------------------------- MMA --
        constexpr uint32_t idS = idesc_bf16(kSpKeys, false);
        constexpr uint32_t idO = idesc_bf16(D, true);
        constexpr uint32_t kVLbo = D == 64 ? 1024u : (uint32_t)(kSpKeys * 128);
        const uint32_t qhi_addr = smem_u32(Qhi), qlo_addr = smem_u32(Qlo);
        const uint32_t ring_addr = smem_u32(ring);
        auto wait_slot = [&](int ld) {
            return pf_warp_wait(&slot_full[ld % M::SLOTS], (ld / M::SLOTS) & 1, abort_flag,
                                p.dev_error);
        };
        // descriptors are built once per group; a k-step only moves the start address
        auto issue_s = [&](int j) {
            const uint32_t k_addr = ring_addr + ((2 * j) % M::SLOTS) * M::KV_BYTES;
            const uint32_t d = tmem + M::S_COL + (j & 1) * kSpKeys;
            const uint64_t db = sw128_desc(k_addr, 16, 1024);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const uint64_t da = sw128_desc(part ? qlo_addr : qhi_addr, 16, 1024);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t dk = (uint64_t)(((k >> 2) * (kSpRows * 128) + (k & 3) * 32) >> 4);
                    umma_bf16(d, da + dk, db + dk, idS, (part > 0 || k > 0) ? 1u : 0u);
                }
            }
            umma_commit(&s_full[j & 1]);
            umma_commit(&slot_empty[(2 * j) % M::SLOTS]);
        };
        auto issue_pv = [&](int j) {
            const uint32_t v_addr = ring_addr + ((2 * j + 1) % M::SLOTS) * M::KV_BYTES;
            const uint32_t pa = tmem + M::S_COL + (j & 1) * kSpKeys;
            const uint64_t dv = sw128_desc(v_addr, kVLbo, 1024);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int k = 0; k < kSpKeys / 16; ++k)
                    umma_bf16_tmem_a(tmem + M::O_COL, pa + part * 64 + k * 8,
                                     dv + (uint64_t)((k * 16 * 128) >> 4), idO,
                                     (j > 0 || part > 0 || k > 0) ? 1u : 0u);
            umma_commit(&slot_empty[(2 * j + 1) % M::SLOTS]);
            umma_commit(&pv_done[j & 1]);
            if (j == ntiles - 1) umma_commit(o_done);
        };
        bool ok = pf_warp_wait(q_ready, 0, abort_flag, p.dev_error) && wait_slot(0);
        bool issued_any = false;
        if (ok) {
            tc_fence_after();
            if (lane == 0) issue_s(0);
            issued_any = true;
            __syncwarp();
        }
        for (int j = 0; ok && j < ntiles; ++j) {
            if (j + 1 < ntiles) {
                if (!wait_slot(2 * j + 2)) break;
                tc_fence_after();
                if (lane == 0) issue_s(j + 1);
                __syncwarp();
            }
            if (!pf_warp_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag, p.dev_error) ||
                !wait_slot(2 * j + 1))
                break;
            tc_fence_after();
            if (lane == 0) issue_pv(j);
            __syncwarp();
        }
        if (issued_any && *abort_flag) {
            if (lane == 0) {
                umma_commit(drain);
                mbar_wait_bounded(drain, 0, kTcWaitLimitNs);
            }
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, M::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_shared_prefix_t(const SharedPrefixArgs& a, const SpParams& p, int ctas,
                                   cudaStream_t stream) {
    using M = SpGeo<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(shared_prefix_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, M::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    CUtensorMap tmk, tmv;
    std::memcpy(&tmk, a.tmap_k, sizeof tmk);
    std::memcpy(&tmv, a.tmap_v, sizeof tmv);
    shared_prefix_kernel<D><<<(unsigned)ctas, kSpThreads, M::SMEM, stream>>>(p, tmk, tmv);
    return cudaGetLastError();
}

}  // namespace

SharedPrefixPlan shared_prefix_plan(int B, int H, int G, int64_t shared_len, int num_sms) {
    SharedPrefixPlan s{};
    s.row_tiles = (B * G + kSpRows - 1) / kSpRows;
    const int64_t tiles = (shared_len + kSpKeys - 1) / kSpKeys;
    int64_t want = num_sms / ((int64_t)H * s.row_tiles);
    if (want < 1) want = 1;
    if (want > tiles) want = tiles;
    const int64_t per = (tiles + want - 1) / want;            // key tiles per split
    s.split_len = per * kSpKeys;
    s.splits = (int)((shared_len + s.split_len - 1) / s.split_len);
    return s;
}

bool shared_prefix_supported(int dtype, int D, int G) {
    return dtype == PKV_BF16 && (D == 64 || D == 128) && G >= 1 && kSpRows % G == 0;
}

cudaError_t launch_shared_prefix(const SharedPrefixArgs& a, cudaStream_t stream) {
    SpParams p{};
    p.B = a.B;
    p.H = a.H;
    p.G = a.G;
    p.P = a.P;
    p.max_pages = a.max_pages;
    p.window = a.window;
    p.n_pages = a.n_pages;
    p.pool_rows = (int)(a.n_pages * a.H * a.P);
    p.q = a.q;
    p.tables = a.tables;
    p.seq_lens = a.seq_lens;
    p.shared_len = a.shared_len;
    p.split_len = a.plan.split_len;
    p.row_tiles = a.plan.row_tiles;
    p.pre_ml = a.pre_ml;
    p.pre_o = a.pre_o;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a.D));
    p.dev_error = a.dev_error;
    const int ctas = a.H * a.plan.row_tiles * a.plan.splits;
    switch (a.D) {
        case 64: return launch_shared_prefix_t<64>(a, p, ctas, stream);
        case 128: return launch_shared_prefix_t<128>(a, p, ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_shared_prefix_hook(const void* ctx, cudaStream_t stream) {
    return launch_shared_prefix(*static_cast<const SharedPrefixArgs*>(ctx), stream);
}

}  // namespace pkv
