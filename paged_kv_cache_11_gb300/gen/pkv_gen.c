/*
 * pkv_gen.c -- seeded synthetic inputs shared by the tests, the bench and
 * the oracle's callers.
 *
 * This file holds no attention arithmetic.  It turns (seed, stream, index)
 * into numbers:
 *
 *   - a counter-based SplitMix64 stream (Steele, Lea and Flood, "Fast
 *     splittable pseudorandom number generators", OOPSLA 2014): element i of
 *     a stream with key k is the SplitMix64 finaliser applied to
 *     k + (i + 1) * 0x9E3779B97F4A7C15;
 *   - N(0,1) samples by the Box-Muller transform (Box and Muller, 1958) on
 *     pairs of uniforms, computed in double and rounded once to fp32;
 *   - IEEE-754 round-to-nearest-even from that fp32 value to bfloat16 or to
 *     binary16.
 *
 * Every element is a pure function of (seed, stream, index), so any slice of
 * a tensor can be produced on its own and the work splits across threads
 * without changing a single bit.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define PKVGEN_BF16 0
#define PKVGEN_FP16 1
#define PKVGEN_FP32 2

static uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* element i of the stream keyed by `key` */
static uint64_t sm64_at(uint64_t key, uint64_t i) {
    return sm64_mix(key + (i + 1ULL) * 0x9E3779B97F4A7C15ULL);
}

uint64_t pkvgen_stream_key(uint64_t seed, uint64_t stream) {
    return sm64_mix(sm64_mix(seed) ^ (stream * 0xD1B54A32D192ED03ULL + 0x8CB92BA72F3D8DD7ULL));
}

uint64_t pkvgen_u64(uint64_t seed, uint64_t stream, uint64_t i) {
    return sm64_at(pkvgen_stream_key(seed, stream), i);
}

/* the Box-Muller pair (elements 2*pair and 2*pair + 1 of the stream) */
static void normal_pair(uint64_t key, uint64_t pair, float* z0, float* z1) {
    /* u1 in (0, 1], u2 in [0, 1): 53 random bits each */
    double u1 = ((double)(sm64_at(key, 2 * pair) >> 11) + 1.0) * (1.0 / 9007199254740992.0);
    double u2 = (double)(sm64_at(key, 2 * pair + 1) >> 11) * (1.0 / 9007199254740992.0);
    double r = sqrt(-2.0 * log(u1));
    double t = 6.283185307179586476925286766559 * u2;
    *z0 = (float)(r * cos(t));
    *z1 = (float)(r * sin(t));
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x0040u);
    uint32_t lsb = (b >> 16) & 1u;
    return (uint16_t)((b + 0x7FFFu + lsb) >> 16);
}

static uint16_t f32_to_fp16_rne(float f) {
    double x = (double)f;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return 0x7E00u;
    if (a == 0.0) return sign;
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (a < 6.103515625e-05) { /* below 2^-14: subnormal grid of 2^-24 */
        double q = rint(a * 16777216.0);
        return (uint16_t)(sign | (uint16_t)q); /* q == 1024 lands on the smallest normal */
    }
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    m *= 2.0;
    e -= 1;                  /* a = m * 2^e, m in [1, 2) */
    double q = rint((m - 1.0) * 1024.0);
    if (q >= 1024.0) { q = 0.0; e += 1; }
    if (e + 15 >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)q);
}

typedef struct {
    uint64_t key, offset;
    int64_t begin, end;
    int dtype;
    void* out;
} job_t;

static void put(const job_t* j, int64_t i, float v) {
    if (j->dtype == PKVGEN_BF16)
        ((uint16_t*)j->out)[i] = f32_to_bf16_rne(v);
    else if (j->dtype == PKVGEN_FP16)
        ((uint16_t*)j->out)[i] = f32_to_fp16_rne(v);
    else
        ((float*)j->out)[i] = v;
}

static void run_job(const job_t* j) {
    for (int64_t i = j->begin; i < j->end;) {
        uint64_t e = j->offset + (uint64_t)i; /* stream element */
        float z0, z1;
        normal_pair(j->key, e >> 1, &z0, &z1);
        if ((e & 1) == 0) {
            put(j, i++, z0);
            if (i < j->end) put(j, i++, z1);
        } else {
            put(j, i++, z1);
        }
    }
}

static void* job_thread(void* p) {
    run_job((const job_t*)p);
    return 0;
}

/*
 * Fill out[0..n) with elements offset..offset+n of the N(0,1) stream
 * (seed, stream), stored as dtype (0 bf16, 1 fp16, 2 fp32).  Returns 0, or -1
 * for a bad argument.
 */
int pkvgen_normal(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, int dtype, void* out,
                  int nthreads) {
    if (n < 0 || (n > 0 && !out) || dtype < 0 || dtype > 2) return -1;
    if (n == 0) return 0;
    uint64_t key = pkvgen_stream_key(seed, stream);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < 65536) nthreads = 1;
    job_t jobs[256];
    pthread_t th[256];
    int64_t chunk = (n + nthreads - 1) / nthreads;
    chunk = (chunk + 1) & ~(int64_t)1;
    int launched = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t b = (int64_t)t * chunk, e = b + chunk;
        if (b >= n) break;
        if (e > n) e = n;
        jobs[t].key = key;
        jobs[t].offset = offset;
        jobs[t].begin = b;
        jobs[t].end = e;
        jobs[t].dtype = dtype;
        jobs[t].out = out;
        ++launched;
    }
    int started[256] = {0};
    for (int t = 1; t < launched; ++t) started[t] = pthread_create(&th[t], 0, job_thread, &jobs[t]) == 0;
    run_job(&jobs[0]);
    for (int t = 1; t < launched; ++t) {
        if (started[t])
            pthread_join(th[t], 0);
        else
            run_job(&jobs[t]);
    }
    return 0;
}

/* The RNE conversions above, exposed so that the tests can pin them. */
void pkvgen_round_f32(const float* in, int64_t n, int dtype, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = dtype == PKVGEN_BF16 ? f32_to_bf16_rne(in[i]) : f32_to_fp16_rne(in[i]);
}

/* out[i] = element offset + i of the raw 64-bit stream (seed, stream). */
void pkvgen_u64_fill(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint64_t* out) {
    uint64_t key = pkvgen_stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = sm64_at(key, offset + (uint64_t)i);
}
