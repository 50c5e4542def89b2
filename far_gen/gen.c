/*
 * Seeded synthetic inputs for fused residual-add + RMSNorm.
 *
 * This file holds random-number generation only: no step of the
 * normalisation (no sums, no rounding to 16-bit formats, no division by
 * the row RMS) lives here.  It serves the CPU oracle and the CUDA path alike,
 * so that both read the same bytes; neither side's arithmetic is in it.
 *
 * Generator: Philox4x32-10, a counter-based generator (Salmon, Moraes, Dror,
 * Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11).  A value is
 * a pure function of (seed, stream, index), so any row range can be produced
 * alone, by any number of threads, with the same result.
 *
 * Normals: Box-Muller in binary64 (one Philox block of four 32-bit words gives
 * four standard normals).  The result is rounded once to binary32 by the C
 * cast; callers round that to the storage format they need.
 */
#include <math.h>
#include <stdint.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

typedef struct { uint32_t v[4]; } block4;

static block4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                            uint32_t k0, uint32_t k1) {
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)PHILOX_M0 * c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += PHILOX_W0;
        k1 += PHILOX_W1;
    }
    block4 b = {{c0, c1, c2, c3}};
    return b;
}

static block4 draw(uint64_t seed, uint32_t stream, uint64_t counter) {
    return philox4x32_10((uint32_t)counter, (uint32_t)(counter >> 32), stream, 0u,
                         (uint32_t)seed, (uint32_t)(seed >> 32));
}

/* uniform in the open interval (0, 1) from one 32-bit word */
static double open_unit(uint32_t w) { return ((double)w + 0.5) * (1.0 / 4294967296.0); }

/* standard normal number `index` of (seed, stream) */
static double normal_at(uint64_t seed, uint32_t stream, uint64_t index) {
    block4 b = draw(seed, stream, index >> 2);
    unsigned lane = (unsigned)(index & 3u);
    unsigned pair = lane >> 1;
    double u1 = open_unit(b.v[2 * pair]);
    double u2 = open_unit(b.v[2 * pair + 1]);
    double radius = sqrt(-2.0 * log(u1));
    double angle = 6.283185307179586476925286766559 * u2;
    return (lane & 1u) ? radius * sin(angle) : radius * cos(angle);
}

/* out[i] = (float)(mean + sd * Z(index start + i)) */
void fargen_normal_f32(uint64_t seed, uint32_t stream, int64_t start, int64_t n,
                       double mean, double sd, float* out) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(mean + sd * normal_at(seed, stream, (uint64_t)(start + i)));
}

/* four consecutive standard normals: indices 4*block .. 4*block + 3 of (seed, stream) */
static void normals_of_block(uint64_t seed, uint32_t stream, uint64_t block, double z[4]) {
    block4 b = draw(seed, stream, block);
    for (unsigned pair = 0; pair < 2; ++pair) {
        double u1 = open_unit(b.v[2 * pair]);
        double u2 = open_unit(b.v[2 * pair + 1]);
        double radius = sqrt(-2.0 * log(u1));
        double angle = 6.283185307179586476925286766559 * u2;
        z[2 * pair] = radius * cos(angle);
        z[2 * pair + 1] = radius * sin(angle);
    }
}

/*
 * Rows [row0, row0 + rows) of a [*, hidden] matrix whose element (t, h) is
 * sd * row_scale[t - row0] * Z(index t * hidden + h); out is rows x hidden.
 * Same values as normal_at(); computed a Philox block at a time.
 */
void fargen_rows_f32(uint64_t seed, uint32_t stream, int64_t row0, int64_t rows,
                     int64_t hidden, const double* row_scale, double sd, float* out) {
    for (int64_t t = 0; t < rows; ++t) {
        double scale = sd * row_scale[t];
        uint64_t base = (uint64_t)(row0 + t) * (uint64_t)hidden;
        float* dst = out + t * hidden;
        int64_t h = 0;
        while (h < hidden) {
            uint64_t index = base + (uint64_t)h;
            double z[4];
            normals_of_block(seed, stream, index >> 2, z);
            for (unsigned lane = (unsigned)(index & 3u); lane < 4u && h < hidden; ++lane, ++h)
                dst[h] = (float)(scale * z[lane]);
        }
    }
}

/* out[i] = uniform in (0, 1), index start + i of (seed, stream); a Philox block at a time */
void fargen_uniform_f64(uint64_t seed, uint32_t stream, int64_t start, int64_t n, double* out) {
    int64_t i = 0;
    while (i < n) {
        uint64_t index = (uint64_t)(start + i);
        block4 b = draw(seed, stream, index >> 2);
        for (unsigned lane = (unsigned)(index & 3u); lane < 4u && i < n; ++lane, ++i)
            out[i] = open_unit(b.v[lane]);
    }
}

/* out[i] = uniform in (0, 1) at index idx[i] of (seed, stream) */
void fargen_uniform_at_f64(uint64_t seed, uint32_t stream, const int64_t* idx, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) {
        uint64_t index = (uint64_t)idx[i];
        block4 b = draw(seed, stream, index >> 2);
        out[i] = open_unit(b.v[index & 3u]);
    }
}

/* the raw Philox block for a counter: exposed so tests can check the generator itself */
void fargen_philox_block(uint64_t seed, uint32_t stream, uint64_t counter, uint32_t* out4) {
    block4 b = draw(seed, stream, counter);
    for (int i = 0; i < 4; ++i) out4[i] = b.v[i];
}

/* raw Philox4x32-10 on an explicit counter and key (for the published test vectors) */
void fargen_philox_raw(const uint32_t* ctr4, const uint32_t* key2, uint32_t* out4) {
    block4 b = philox4x32_10(ctr4[0], ctr4[1], ctr4[2], ctr4[3], key2[0], key2[1]);
    for (int i = 0; i < 4; ++i) out4[i] = b.v[i];
}
