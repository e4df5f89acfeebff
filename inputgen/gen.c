/*
 * Seeded synthetic inputs for the MoE token-dispatch + expert-GEMM path.
 *
 * This file produces INPUTS ONLY: activations x, expert weights W and routed
 * top-k expert indices. It holds none of the dispatch or GEMM arithmetic, and
 * both the CPU oracle and the CUDA path consume exactly the bytes it writes.
 *
 * Random numbers are counter based so that any slice (one expert's weight
 * matrix, one token's logits) can be produced on its own, in parallel:
 *   u64(seed, stream, i) = i-th output of a splitmix64 sequence whose state
 *                          starts at key(seed, stream)
 *                        = mix(key + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix is Steele, Lea and Flood's splitmix64 finaliser (OOPSLA 2014,
 * "Fast splittable pseudorandom number generators").
 * Normals use the Box-Muller transform on pairs (2p, 2p+1) of uniforms in
 * (0, 1]: element 2p takes the cosine branch and element 2p+1 the sine branch.
 * bf16 values are made by float64 -> float32 (round to nearest even, C cast)
 * -> bf16 (round to nearest even on the float32 bit pattern).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* Key of one stream: two rounds of mixing over the seed and the stream id. */
uint64_t ig_stream_key(uint64_t seed, uint64_t stream) {
    return sm64_mix(sm64_mix(seed + GOLDEN) ^ (stream * 0xD1B54A32D192ED03ull));
}

/* i-th raw 64-bit output of the splitmix64 sequence that starts at `state`. */
uint64_t ig_splitmix64_at(uint64_t state, uint64_t i) {
    return sm64_mix(state + (i + 1) * GOLDEN);
}

static inline double u01(uint64_t key, uint64_t i) {
    /* 53 random bits, shifted into (0, 1] so that log() is finite. */
    return (double)((ig_splitmix64_at(key, i) >> 11) + 1) * (1.0 / 9007199254740992.0);
}

double ig_normal_at(uint64_t key, uint64_t i) {
    const uint64_t p = i >> 1;
    const double u1 = u01(key, 2 * p), u2 = u01(key, 2 * p + 1);
    const double r = sqrt(-2.0 * log(u1));
    const double th = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * sin(th) : r * cos(th);
}

uint16_t ig_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ---- bf16 normal fill, threaded over contiguous ranges ---------------- */
typedef struct {
    uint64_t key, start, n;
    double scale;
    uint16_t* out;
} fill_job;

static void* fill_worker(void* arg) {
    fill_job* j = (fill_job*)arg;
    for (uint64_t i = 0; i < j->n; ++i) {
        double z = j->scale * ig_normal_at(j->key, j->start + i);
        j->out[i] = ig_f32_to_bf16((float)z);
    }
    return NULL;
}

/* out[i] = bf16(float(scale * N(0,1)[start + i])) for i in [0, n). */
int ig_fill_normal_bf16(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n,
                        double scale, uint16_t* out, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((uint64_t)nthreads > n / 4096 + 1) nthreads = (int)(n / 4096 + 1);
    const uint64_t key = ig_stream_key(seed, stream);
    pthread_t th[256];
    fill_job jobs[256];
    const uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
    int launched = 0;
    for (int t = 0; t < nthreads; ++t) {
        uint64_t b = (uint64_t)t * per, e = b + per;
        if (b >= n) break;
        if (e > n) e = n;
        jobs[t].key = key; jobs[t].start = start + b; jobs[t].n = e - b;
        jobs[t].scale = scale; jobs[t].out = out + b;
        if (t == nthreads - 1 || pthread_create(&th[t], NULL, fill_worker, &jobs[t]) != 0) {
            fill_worker(&jobs[t]);
            th[t] = 0;
        }
        launched = t + 1;
    }
    for (int t = 0; t < launched; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    return 0;
}

/* ---- routing: top-k of per-token router logits ------------------------- */
/*
 * logit[t][e] = N(0,1)[t*E + e] (stream `stream`) + bias[e], with
 * bias[e] = -zipf_s * ln(e + 1) when zipf_s > 0 (a Zipf(s) rank weight for
 * expert e, so expert 0 is the most popular). Slot s of token t holds the
 * expert with the s-th largest logit; equal logits go to the lower expert.
 * The k experts of a token are therefore distinct.
 */
typedef struct {
    uint64_t key;
    int64_t t0, t1, E, k;
    double zipf_s;
    int32_t* topk;
    double* scratch;
    unsigned char* taken;
} topk_job;

static void* topk_worker(void* arg) {
    topk_job* j = (topk_job*)arg;
    for (int64_t t = j->t0; t < j->t1; ++t) {
        for (int64_t e = 0; e < j->E; ++e) {
            double v = ig_normal_at(j->key, (uint64_t)(t * j->E + e));
            if (j->zipf_s > 0.0) v -= j->zipf_s * log((double)(e + 1));
            j->scratch[e] = v;
            j->taken[e] = 0;
        }
        for (int64_t s = 0; s < j->k; ++s) {
            int64_t best = -1;
            for (int64_t e = 0; e < j->E; ++e) {
                if (j->taken[e]) continue;
                if (best < 0 || j->scratch[e] > j->scratch[best]) best = e;
            }
            j->taken[best] = 1;
            j->topk[t * j->k + s] = (int32_t)best;
        }
    }
    return NULL;
}

int ig_topk_routing(uint64_t seed, uint64_t stream, int64_t T, int64_t E, int64_t k,
                    double zipf_s, int32_t* topk, int nthreads) {
    if (k < 1 || k > E || T < 0) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > T) nthreads = T > 0 ? (int)T : 1;
    const uint64_t key = ig_stream_key(seed, stream);
    double* scratch = (double*)malloc(sizeof(double) * (size_t)(E * nthreads));
    unsigned char* taken = (unsigned char*)malloc((size_t)(E * nthreads));
    if (!scratch || !taken) { free(scratch); free(taken); return 2; }
    pthread_t th[256];
    topk_job jobs[256];
    const int64_t per = (T + nthreads - 1) / nthreads;
    int launched = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t b = (int64_t)t * per, e = b + per;
        if (b >= T) break;
        if (e > T) e = T;
        jobs[t].key = key; jobs[t].t0 = b; jobs[t].t1 = e; jobs[t].E = E; jobs[t].k = k;
        jobs[t].zipf_s = zipf_s; jobs[t].topk = topk;
        jobs[t].scratch = scratch + (size_t)t * (size_t)E;
        jobs[t].taken = taken + (size_t)t * (size_t)E;
        if (t == nthreads - 1 || pthread_create(&th[t], NULL, topk_worker, &jobs[t]) != 0) {
            topk_worker(&jobs[t]);
            th[t] = 0;
        }
        launched = t + 1;
    }
    for (int t = 0; t < launched; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    free(scratch);
    free(taken);
    return 0;
}

/* ---- router logits and combine gates ----------------------------------- */
/* logits[t][e] = float32(N(0,1)[t*E + e] - zipf_s * ln(e + 1)), the same
 * stream and bias as the routing above (rounded to float32). */
int ig_logits_f32(uint64_t seed, uint64_t stream, int64_t T, int64_t E, double zipf_s,
                  float* out) {
    const uint64_t key = ig_stream_key(seed, stream);
    for (int64_t t = 0; t < T; ++t)
        for (int64_t e = 0; e < E; ++e) {
            double v = ig_normal_at(key, (uint64_t)(t * E + e));
            if (zipf_s > 0.0) v -= zipf_s * log((double)(e + 1));
            out[t * E + e] = (float)v;
        }
    return 0;
}

/* Positive weights that sum to one per token: u[t][s] uniform in (0, 1],
 * divided by the token's sum, rounded to float32. */
int ig_weights_f32(uint64_t seed, uint64_t stream, int64_t T, int64_t k, float* out) {
    const uint64_t key = ig_stream_key(seed, stream);
    for (int64_t t = 0; t < T; ++t) {
        double sum = 0.0;
        for (int64_t s = 0; s < k; ++s) sum += u01(key, (uint64_t)(t * k + s));
        for (int64_t s = 0; s < k; ++s)
            out[t * k + s] = (float)(u01(key, (uint64_t)(t * k + s)) / sum);
    }
    return 0;
}
