/*
 * synth_host.c -- the seeded input generator of synth/__init__.py in plain C
 * for the host, split over threads, for weight tensors too large to draw
 * with numpy.  Same counter arithmetic (fmix32 words), same Irwin-Hall(12)
 * sum, one binary32 multiply by sigma: identical bits to the numpy
 * definition and to the CUDA twin.  Test infrastructure: it draws numbers
 * and holds none of the method's arithmetic.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared -pthread.
 */
#include <pthread.h>
#include <stdint.h>

static uint32_t fmix32(uint32_t h)
{
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

typedef struct {
    uint32_t key;
    uint64_t offset, begin, end;
    float sigma;
    float *out;
} job_t;

static void *run(void *p)
{
    const job_t *j = (const job_t *)p;
    for (uint64_t e = j->begin; e < j->end; ++e) {
        const uint32_t i = (uint32_t)(j->offset + e);
        const uint32_t a = fmix32(i ^ j->key);
        int32_t s = 0;
        for (uint32_t k = 0; k < 6; ++k) {
            const uint32_t w = fmix32(a + (k + 1u) * 0x9E3779B9u);
            s += (int32_t)(w & 0xFFFFu) + (int32_t)(w >> 16);
        }
        const float z = (float)(s - 393210) / 65536.0f; /* exact: |s - 393210| < 2^24 */
        j->out[e] = z * j->sigma;
    }
    return 0;
}

/* out[e] = N(0, sigma) draw of element offset + e of stream `seed`, for
 * e < count; counters are 32-bit (offset + count <= 2^32).  Returns 0, or
 * 3 for counters out of range. */
int synth_normal_f32_host(uint32_t seed, uint64_t offset, uint64_t count, float sigma, float *out,
                          int threads)
{
    if (count == 0) return 0;
    if (offset + count > (1ull << 32)) return 3;
    if (threads < 1) threads = 1;
    if (threads > 64) threads = 64;
    if ((uint64_t)threads > count) threads = (int)count;
    job_t jobs[64];
    pthread_t tid[64];
    const uint32_t key = fmix32(seed);
    for (int t = 0; t < threads; ++t) {
        jobs[t].key = key;
        jobs[t].offset = offset;
        jobs[t].begin = count * (uint64_t)t / (uint64_t)threads;
        jobs[t].end = count * (uint64_t)(t + 1) / (uint64_t)threads;
        jobs[t].sigma = sigma;
        jobs[t].out = out;
    }
    int started = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tid[t], 0, run, &jobs[t]) != 0) break;
        started = t;
    }
    run(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], 0);
    for (int t = started + 1; t < threads; ++t) run(&jobs[t]); /* threads that did not start */
    return 0;
}
