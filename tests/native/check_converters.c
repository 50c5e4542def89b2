/*
 * Exhaustive check of an oracle library's binary32 -> fp16 / bf16 rounding
 * against the compiler's own conversions (_Float16 and __bf16 casts, which
 * round to nearest, ties to even).  Every one of the 2^32 binary32 bit
 * patterns is converted both ways; NaN inputs only need a NaN result.
 *
 * usage: check_converters <liboracle.so> f16|bf16
 * prints the number of mismatches and the first few; exit status 0 iff none.
 */
#include <dlfcn.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

typedef uint16_t (*conv_fn)(float);

static conv_fn oracle_conv;
static int use_bf16;
#define THREADS 16

typedef struct { uint64_t begin, end, mismatches; uint32_t first[4]; } job;

static uint16_t reference(float f) {
    uint16_t out;
    if (use_bf16) { __bf16 b = (__bf16)f; memcpy(&out, &b, 2); }
    else { _Float16 h = (_Float16)f; memcpy(&out, &h, 2); }
    return out;
}

static int is_nan16(uint16_t h) {
    return use_bf16 ? ((h & 0x7f80u) == 0x7f80u && (h & 0x7fu)) : ((h & 0x7c00u) == 0x7c00u && (h & 0x3ffu));
}

static void* run(void* p) {
    job* j = (job*)p;
    for (uint64_t u = j->begin; u < j->end; ++u) {
        uint32_t bits = (uint32_t)u;
        float f;
        memcpy(&f, &bits, 4);
        uint16_t a = oracle_conv(f), b = reference(f);
        int same = (a == b) || (is_nan16(a) && is_nan16(b));
        if (!same) {
            if (j->mismatches < 4) j->first[j->mismatches] = bits;
            j->mismatches++;
        }
    }
    return NULL;
}

int main(int argc, char** argv) {
    if (argc != 3) return 2;
    void* h = dlopen(argv[1], RTLD_NOW);
    if (!h) { fprintf(stderr, "%s\n", dlerror()); return 2; }
    use_bf16 = strcmp(argv[2], "bf16") == 0;
    oracle_conv = (conv_fn)dlsym(h, use_bf16 ? "oracle_f32_to_bf16" : "oracle_f32_to_f16");
    if (!oracle_conv) return 2;
    pthread_t th[THREADS];
    job jobs[THREADS];
    uint64_t total = 1ull << 32, step = total / THREADS;
    for (int i = 0; i < THREADS; ++i) {
        memset(&jobs[i], 0, sizeof jobs[i]);
        jobs[i].begin = i * step;
        jobs[i].end = (i == THREADS - 1) ? total : (i + 1) * step;
        pthread_create(&th[i], NULL, run, &jobs[i]);
    }
    uint64_t mismatches = 0;
    for (int i = 0; i < THREADS; ++i) {
        pthread_join(th[i], NULL);
        for (uint64_t k = 0; k < jobs[i].mismatches && k < 4; ++k)
            printf("mismatch at 0x%08x\n", jobs[i].first[k]);
        mismatches += jobs[i].mismatches;
    }
    printf("mismatches %llu\n", (unsigned long long)mismatches);
    return mismatches == 0 ? 0 : 1;
}
