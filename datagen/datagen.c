/*
 * Seeded synthetic inputs for the quantized-weight GEMV library and its tests.
 *
 * This file is input preparation only.  It draws the fp32 weights and
 * activations that the workloads describe, and it packs the weights into the
 * block formats that the GPU kernels and the CPU oracle both read.  It holds
 * none of the arithmetic of the hot path: no activation quantisation, no dot
 * products, no transform, no soft-cap, no argmax.  Both the oracle and the
 * CUDA path consume the bytes written here; the oracle decodes them with its
 * own, independent code.
 *
 * Random numbers.  Every value is a pure function of (seed, stream, index):
 *   key(seed, stream) = mix64(seed + G * (stream + 1))
 *   u64(seed, stream, i) = mix64(key + G * (i + 1))
 * where mix64 is the SplitMix64 output function (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014) and G is its
 * golden-gamma increment 0x9E3779B97F4A7C15.
 *   uniform(i) = ((u64(i) >> 11) + 0.5) * 2^-53          in (0, 1)
 *   normal(i)  = Box-Muller on the uniform pair (2*(i/2), 2*(i/2)+1):
 *                r = sqrt(-2 ln u0), cos(2 pi u1) for even i, sin for odd i.
 * Normals are formed in double and rounded once to float after scaling.
 *
 * Block weight formats (blocks of 32 consecutive weights along K, row-major
 * over rows; a row of K weights has K/32 blocks):
 *   Q4: codes u8 [N][K/2]; block byte j (0..15) holds code j in bits 0-3 and
 *       code j+16 in bits 4-7.  scale f16 [N][K/32], min f16 [N][K/32].
 *   Q6: lo u8 [N][K/2] with the low 4 code bits in the Q4 byte order;
 *       hi u8 [N][K/4], 8 bytes per block, byte t (0..7) holding the top 2
 *       code bits of codes t, t+8, t+16, t+24 in bits 0-1, 2-3, 4-5, 6-7.
 *   A weight decodes as  w = scale * code + min.
 *   Q2: codes u8 [N][K/4], 8 bytes per block, byte t (0..7) holding codes t, t+8,
 *       t+16, t+24 in bits 0-1, 2-3, 4-5, 6-7; scale f16 [N][K/32]; no min plane:
 *       a weight decodes as w = scale * (code - 2) (zero point 2).
 * Asymmetric block quantiser used to make the packed inputs: lo = min(w),
 * hi = max(w) over the block; d = (hi - lo) / qmax in float (qmax 15 or 63);
 * scale = f16(d), min = f16(lo) (round to nearest even);
 * code = clamp(rint((w - min) / scale), 0, qmax) in float with the stored
 * half values; code = 0 when scale == 0.
 * Q2 quantiser: scale = f16(max(hi, -lo / 2)) so that the codes 0..3 (values
 * -2, -1, 0, 1 times the scale) cover the block; code = clamp(rint(w / scale) + 2,
 * 0, 3) in float with the stored half; code = 2 when scale == 0.
 *   CQ: idx u8 [N][K/2]; element 2j in bits 0-3 of byte j, element 2j+1 in
 *       bits 4-7; codebook f16 [16]; row scale f16 [N].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define DG_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed + DG_GAMMA * (stream + 1));
}

static inline uint64_t keyed_u64(uint64_t key, uint64_t i) {
    return mix64(key + DG_GAMMA * (i + 1));
}

static inline double keyed_uniform(uint64_t key, uint64_t i) {
    return ((double)(keyed_u64(key, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static const double DG_TWO_PI = 6.283185307179586476925286766559;

/* normal(i) for a whole aligned pair at once: out0 = normal(2p), out1 = normal(2p+1) */
static inline void keyed_normal_pair(uint64_t key, uint64_t p, double* out0, double* out1) {
    double u0 = keyed_uniform(key, 2 * p);
    double u1 = keyed_uniform(key, 2 * p + 1);
    double r = sqrt(-2.0 * log(u0));
    double a = DG_TWO_PI * u1;
    *out0 = r * cos(a);
    *out1 = r * sin(a);
}

static inline double keyed_normal(uint64_t key, uint64_t i) {
    double a, b;
    keyed_normal_pair(key, i >> 1, &a, &b);
    return (i & 1) ? b : a;
}

uint64_t dg_u64(uint64_t seed, uint64_t stream, uint64_t i) {
    return keyed_u64(stream_key(seed, stream), i);
}

double dg_uniform(uint64_t seed, uint64_t stream, uint64_t i) {
    return keyed_uniform(stream_key(seed, stream), i);
}

double dg_normal(uint64_t seed, uint64_t stream, uint64_t i) {
    return keyed_normal(stream_key(seed, stream), i);
}

/* out[j] = (float)(mean + sigma * normal(offset + j)), j < n */
void dg_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double mean,
                   double sigma, float* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t j = 0; j < n; ++j) out[j] = (float)(mean + sigma * keyed_normal(key, offset + (uint64_t)j));
}

/* out[j] = (float)(lo + (hi - lo) * uniform(offset + j)) */
void dg_uniform_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double lo, double hi,
                    float* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t j = 0; j < n; ++j) out[j] = (float)(lo + (hi - lo) * keyed_uniform(key, offset + (uint64_t)j));
}

/* ---- fp16 packing (round to nearest even, via the compiler's _Float16) ---- */
static inline uint16_t f32_to_f16_bits(float f) {
    _Float16 h = (_Float16)f;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

static inline float f16_bits_to_f32(uint16_t b) {
    _Float16 h;
    memcpy(&h, &b, 2);
    return (float)h;
}

void dg_f32_to_f16(const float* in, int64_t n, uint16_t* out) {
    for (int64_t j = 0; j < n; ++j) out[j] = f32_to_f16_bits(in[j]);
}

/* ---- block quantiser and packers ---- */

/* quantise one block of 32 floats to codes in [0, qmax]; writes scale/min bits */
static void quantize_block(const float* w, int qmax, uint8_t* q, uint16_t* scale_bits, uint16_t* min_bits) {
    float lo = w[0], hi = w[0];
    for (int i = 1; i < 32; ++i) {
        if (w[i] < lo) lo = w[i];
        if (w[i] > hi) hi = w[i];
    }
    float d = (hi - lo) / (float)qmax;
    uint16_t db = f32_to_f16_bits(d);
    uint16_t mb = f32_to_f16_bits(lo);
    float d16 = f16_bits_to_f32(db);
    float m16 = f16_bits_to_f32(mb);
    for (int i = 0; i < 32; ++i) {
        int c = 0;
        if (d16 != 0.0f) {
            float t = rintf((w[i] - m16) / d16);
            if (t < 0.0f) t = 0.0f;
            if (t > (float)qmax) t = (float)qmax;
            c = (int)t;
        }
        q[i] = (uint8_t)c;
    }
    *scale_bits = db;
    *min_bits = mb;
}

static void pack_q4_block(const uint8_t* q, uint8_t* codes16) {
    for (int j = 0; j < 16; ++j) codes16[j] = (uint8_t)((q[j] & 15) | ((q[j + 16] & 15) << 4));
}

static void pack_q6_block(const uint8_t* q, uint8_t* lo16, uint8_t* hi8) {
    for (int j = 0; j < 16; ++j) lo16[j] = (uint8_t)((q[j] & 15) | ((q[j + 16] & 15) << 4));
    for (int t = 0; t < 8; ++t)
        hi8[t] = (uint8_t)(((q[t] >> 4) & 3) | (((q[t + 8] >> 4) & 3) << 2) | (((q[t + 16] >> 4) & 3) << 4) |
                           (((q[t + 24] >> 4) & 3) << 6));
}

static void quantize_block_q2(const float* w, uint8_t* q, uint16_t* scale_bits) {
    float lo = w[0], hi = w[0];
    for (int i = 1; i < 32; ++i) {
        if (w[i] < lo) lo = w[i];
        if (w[i] > hi) hi = w[i];
    }
    float d = hi > -lo / 2.0f ? hi : -lo / 2.0f;
    if (d < 0.0f) d = 0.0f;
    uint16_t db = f32_to_f16_bits(d);
    float d16 = f16_bits_to_f32(db);
    for (int i = 0; i < 32; ++i) {
        int c = 2;
        if (d16 != 0.0f) {
            float t = rintf(w[i] / d16) + 2.0f;
            if (t < 0.0f) t = 0.0f;
            if (t > 3.0f) t = 3.0f;
            c = (int)t;
        }
        q[i] = (uint8_t)c;
    }
    *scale_bits = db;
}

static void pack_q2_block(const uint8_t* q, uint8_t* c8) {
    for (int t = 0; t < 8; ++t)
        c8[t] = (uint8_t)((q[t] & 3) | ((q[t + 8] & 3) << 2) | ((q[t + 16] & 3) << 4) | ((q[t + 24] & 3) << 6));
}

void dg_pack_q2_codes(const uint8_t* q, int64_t n, int64_t k, uint8_t* codes) {
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < k / 32; ++b) pack_q2_block(q + r * k + b * 32, codes + r * (k / 4) + b * 8);
}

/* Pack caller-chosen codes (values 0..15 / 0..63) for [n][k]; used by tests to
 * build exact cases.  q is row-major [n][k]. */
void dg_pack_q4_codes(const uint8_t* q, int64_t n, int64_t k, uint8_t* codes) {
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < k / 32; ++b) pack_q4_block(q + r * k + b * 32, codes + r * (k / 2) + b * 16);
}

void dg_pack_q6_codes(const uint8_t* q, int64_t n, int64_t k, uint8_t* lo, uint8_t* hi) {
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < k / 32; ++b)
            pack_q6_block(q + r * k + b * 32, lo + r * (k / 2) + b * 16, hi + r * (k / 4) + b * 8);
}

/* Quantise a caller-supplied fp32 matrix [n][k]. hi may be NULL for bits == 4. */
void dg_quantize_matrix(int bits, const float* w, int64_t n, int64_t k, uint8_t* lo, uint8_t* hi,
                        uint16_t* scale, uint16_t* min) {
    int qmax = bits == 4 ? 15 : 63;
    uint8_t q[32];
    int64_t nb = k / 32;
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            if (bits == 2) {
                quantize_block_q2(w + r * k + b * 32, q, scale + r * nb + b);
                pack_q2_block(q, lo + r * (k / 4) + b * 8);
                continue;
            }
            quantize_block(w + r * k + b * 32, qmax, q, scale + r * nb + b, min + r * nb + b);
            if (bits == 4)
                pack_q4_block(q, lo + r * (k / 2) + b * 16);
            else
                pack_q6_block(q, lo + r * (k / 2) + b * 16, hi + r * (k / 4) + b * 8);
        }
    }
}

/* ---- seeded random quantised matrices, multi-threaded over rows ---- */
typedef struct {
    int bits;
    uint64_t key;
    int64_t k;
    double sigma;
    int64_t row0, row1;
    uint8_t* lo;
    uint8_t* hi;
    uint16_t* scale;
    uint16_t* min;
} qjob;

/* the fp32 weight of element (r, c): (float)(sigma * normal(r*k + c)) */
static void weights_row(uint64_t key, int64_t r, int64_t k, double sigma, float* row) {
    uint64_t base = (uint64_t)r * (uint64_t)k; /* k is even, so pairs never straddle rows */
    for (int64_t c = 0; c < k; c += 2) {
        double a, b;
        keyed_normal_pair(key, (base + (uint64_t)c) >> 1, &a, &b);
        row[c] = (float)(sigma * a);
        row[c + 1] = (float)(sigma * b);
    }
}

static void* qjob_run(void* arg) {
    qjob* j = (qjob*)arg;
    float* row = (float*)malloc(sizeof(float) * (size_t)j->k);
    int qmax = j->bits == 4 ? 15 : 63;
    int64_t nb = j->k / 32;
    uint8_t q[32];
    for (int64_t r = j->row0; r < j->row1; ++r) {
        weights_row(j->key, r, j->k, j->sigma, row);
        for (int64_t b = 0; b < nb; ++b) {
            if (j->bits == 2) {
                quantize_block_q2(row + b * 32, q, j->scale + r * nb + b);
                pack_q2_block(q, j->lo + r * (j->k / 4) + b * 8);
                continue;
            }
            quantize_block(row + b * 32, qmax, q, j->scale + r * nb + b, j->min + r * nb + b);
            if (j->bits == 4)
                pack_q4_block(q, j->lo + r * (j->k / 2) + b * 16);
            else
                pack_q6_block(q, j->lo + r * (j->k / 2) + b * 16, j->hi + r * (j->k / 4) + b * 8);
        }
    }
    free(row);
    return NULL;
}

/* W[r][c] = (float)(sigma * normal(seed, stream, r*k + c)), quantised to Q4/Q6.
 * Returns 0 on success. */
int dg_make_quantized(int bits, uint64_t seed, uint64_t stream, int64_t n, int64_t k, double sigma, uint8_t* lo,
                      uint8_t* hi, uint16_t* scale, uint16_t* min, int nthreads) {
    if ((bits != 2 && bits != 4 && bits != 6) || k % 32 != 0 || n < 0) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < (int64_t)nthreads * 4) nthreads = 1;
    qjob jobs[256];
    pthread_t th[256];
    uint64_t key = stream_key(seed, stream);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].bits = bits;
        jobs[t].key = key;
        jobs[t].k = k;
        jobs[t].sigma = sigma;
        jobs[t].row0 = n * t / nthreads;
        jobs[t].row1 = n * (t + 1) / nthreads;
        jobs[t].lo = lo;
        jobs[t].hi = hi;
        jobs[t].scale = scale;
        jobs[t].min = min;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, qjob_run, &jobs[t]) != 0) break;
        started = t;
    }
    qjob_run(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) qjob_run(&jobs[t]); /* threads that failed to start */
    return 0;
}

/* The unquantised fp32 weights of rows [row0, row0 + nrows) of the same matrix. */
void dg_weights_f32(uint64_t seed, uint64_t stream, int64_t row0, int64_t nrows, int64_t k, double sigma,
                    float* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t r = 0; r < nrows; ++r) weights_row(key, row0 + r, k, sigma, out + r * k);
}

/* CQ matrix: idx uniform on 0..15 (low 4 bits of u64(stream_idx, element)),
 * packed two per byte, element 2j in the low nibble. */
void dg_make_cq_indices(uint64_t seed, uint64_t stream, int64_t n, int64_t k, uint8_t* idx) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t r = 0; r < n; ++r)
        for (int64_t j = 0; j < k / 2; ++j) {
            uint64_t e = (uint64_t)(r * k + 2 * j);
            uint8_t a = (uint8_t)(keyed_u64(key, e) & 15);
            uint8_t b = (uint8_t)(keyed_u64(key, e + 1) & 15);
            idx[r * (k / 2) + j] = (uint8_t)(a | (b << 4));
        }
}
