/*
 * Seeded synthetic inputs for paged decode attention workloads.
 *
 * This file is shared input plumbing: both the fp64 oracle and the device
 * harness take their q / k / v / history values from it, so that the two
 * sides see the same bytes.  It holds none of the attention arithmetic.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), evaluated counter-style.  The i-th output
 * (0-based) of a SplitMix64 stream whose state starts at `s` is
 * mix(s + (i + 1) * GAMMA), so any element can be computed independently.
 *
 * Value distribution: an approximately standard normal value built from one
 * 64-bit output as the Irwin-Hall sum of its four 16-bit fields, centred and
 * divided by its exact standard deviation.  Integer work plus one IEEE fp64
 * multiply and one rounding to fp32, so the value is identical on every host.
 *
 * bf16 storage values are the fp32 value rounded to nearest, ties to even.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define SM64_GAMMA 0x9e3779b97f4a7c15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

/* i-th output (0-based) of the SplitMix64 stream seeded with `seed`. */
uint64_t synth_splitmix64_at(uint64_t seed, uint64_t i) {
    return sm64_mix(seed + (i + 1) * SM64_GAMMA);
}

/* Seed of an independent sub-stream, e.g. one (layer, kind, request). */
uint64_t synth_stream_seed(uint64_t seed, uint64_t stream) {
    return sm64_mix(seed ^ sm64_mix(stream + SM64_GAMMA));
}

/* Irwin-Hall(4) of 16-bit uniforms: sum in [0, 4*65535], mean 2*65535,
 * variance 4*(65536^2-1)/12.  Returned centred and scaled to unit variance. */
static inline float normal_from_bits(uint64_t x) {
    int64_t s = (int64_t)(x & 0xffff) + (int64_t)((x >> 16) & 0xffff) +
                (int64_t)((x >> 32) & 0xffff) + (int64_t)(x >> 48);
    /* 2*s - 4*65535 is an exact even-centred integer; divide by 2*sd. */
    const double inv_two_sd = 1.0 / (2.0 * sqrt(4.0 * (65536.0 * 65536.0 - 1.0) / 12.0));
    return (float)((double)(2 * s - 4 * 65535) * inv_two_sd);
}

uint16_t synth_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u) {           /* inf / nan */
        uint16_t h = (uint16_t)(u >> 16);
        if (u & 0x007fffffu) h |= 0x0040u;              /* keep nan quiet */
        return h;
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

float synth_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Key of one element of a (head, token, feature) row stream.  Tokens of one
 * head are consecutive, so rows are consecutive keys. */
static inline uint64_t row_key(int64_t head, int64_t token, int64_t d, int64_t D) {
    return ((uint64_t)head << 44) + (uint64_t)token * (uint64_t)D + (uint64_t)d;
}

/* out[r*D + d] = value of (head, token0 + r, d), for r < nrows.
 * dtype 0: fp32 written to out (float*); dtype 1: bf16 bits (uint16_t*). */
void synth_rows(uint64_t seed, uint64_t stream, int64_t head, int64_t token0,
                int64_t nrows, int64_t D, int dtype, void* out) {
    uint64_t s = synth_stream_seed(seed, stream);
    #pragma omp parallel for schedule(static) if (nrows * D > (1 << 16))
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t d = 0; d < D; ++d) {
            float v = normal_from_bits(synth_splitmix64_at(s, row_key(head, token0 + r, d, D)));
            if (dtype == 0) ((float*)out)[r * D + d] = v;
            else ((uint16_t*)out)[r * D + d] = synth_f32_to_bf16(v);
        }
    }
}

/*
 * Fill history pages of one request in physical layout.
 * out has shape [n_pages][H][P][D] in the storage dtype and holds logical pages
 * first_page .. first_page + n_pages - 1.  Logical token j of head h goes to
 * page j / P, slot j % P.  Tokens j < n_tokens get the value of (stream, head h,
 * token j); all other slots are zero.
 */
void synth_history_pages_from(uint64_t seed, uint64_t stream, int64_t first_page, int64_t n_pages,
                              int64_t H, int64_t P, int64_t D, int64_t n_tokens, int dtype,
                              void* out) {
    uint64_t s = synth_stream_seed(seed, stream);
    int64_t es = dtype == 0 ? 4 : 2;
    #pragma omp parallel for schedule(static) collapse(2)
    for (int64_t pg = 0; pg < n_pages; ++pg) {
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t slot = 0; slot < P; ++slot) {
                int64_t j = (first_page + pg) * P + slot;
                int64_t base = ((pg * H + h) * P + slot) * D;
                if (j >= n_tokens) {
                    memset((char*)out + base * es, 0, (size_t)(D * es));
                    continue;
                }
                for (int64_t d = 0; d < D; ++d) {
                    float v = normal_from_bits(synth_splitmix64_at(s, row_key(h, j, d, D)));
                    if (dtype == 0) ((float*)out)[base + d] = v;
                    else ((uint16_t*)out)[base + d] = synth_f32_to_bf16(v);
                }
            }
        }
    }
}

void synth_history_pages(uint64_t seed, uint64_t stream, int64_t n_pages, int64_t H,
                         int64_t P, int64_t D, int64_t n_tokens, int dtype, void* out) {
    synth_history_pages_from(seed, stream, 0, n_pages, H, P, D, n_tokens, dtype, out);
}

/* n fp32 -> bf16 bits, round to nearest even. */
void synth_f32_to_bf16_array(const float* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = synth_f32_to_bf16(in[i]);
}

int synth_max_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
