/*
 * CPU oracle for the quantized-weight GEMV library.  TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, scalar C that states what the hot path computes, in fp64
 * wherever the method does not fix the precision.  It shares no code, header,
 * table or constant with the CUDA library: it decodes the packed bytes with its
 * own bit extraction, written from the layout statement below.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * Layouts read here (blocks of 32 consecutive weights along K, rows row-major):
 *   Q4: codes byte (r, 16*b + j) holds code 32*b + j in bits 0-3 and code
 *       32*b + j + 16 in bits 4-7.
 *   Q6: lo plane as Q4 for the low 4 bits; hi plane 8 bytes per block, byte
 *       (r, 8*b + t) holding the top 2 bits of codes 32*b + t, +8, +16, +24
 *       in bits 0-1, 2-3, 4-5, 6-7.
 *   scale / min: one IEEE binary16 per block; a weight is scale*code + min.
 *   Q2: codes byte (r, 8*b + t) holds the 2-bit codes 32*b + t, +8, +16, +24 in bits
 *       0-1, 2-3, 4-5, 6-7; one binary16 scale per block, no min: a weight is
 *       scale*(code - 2), the int2 zero point 2 of the Gemma WebGPU Engine ("Roadmap").
 *   CQ: byte (r, j) holds index 2j in bits 0-3 and index 2j+1 in bits 4-7.
 *
 * Where the pages leave a step open, the reading taken is stated at the
 * function that takes it.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* IEEE binary16 bits -> double, exactly: sign, 5-bit exponent (bias 15),
 * 10-bit fraction; exponent 0 is subnormal (no implicit 1), 31 is inf/NaN. */
double or_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/*
 * Per-block int8 activation quantisation (the "q8_1" activation shared by the
 * decode GEMVs: genie-ai-runtime v1.1 -> v1.3.1, "v1.2.0 - a decode
 * optimization cycle"; oxinfer README, "How it works", per-matmul activation
 * quantization; Gemma WebGPU Engine, "Roadmap", SRQ activation and sumA).
 * For each block b of 32 values:
 *   amax = max |x_i|;  s_b = amax / 127 (fp32);
 *   xq_i = clamp(round_half_even(x_i / s_b), -127, 127)  (fp32 division);
 *   S_b  = sum_i xq_i.
 * The scale is fp32 by the workload statement ("fp32 absmax scale"), and the
 * integer decision is taken in that precision.  Reading: when s_b == 0 the
 * block is all zero codes (no division by zero).
 */
void or_quantize_act(const float* x, int64_t k, int8_t* xq, float* s, int32_t* S) {
    for (int64_t b = 0; b < k / 32; ++b) {
        const float* xb = x + 32 * b;
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        float sb = amax / 127.0f;
        int32_t sum = 0;
        for (int i = 0; i < 32; ++i) {
            int q = 0;
            if (sb != 0.0f) {
                float t = nearbyintf(xb[i] / sb);
                if (t > 127.0f) t = 127.0f;
                if (t < -127.0f) t = -127.0f;
                q = (int)t;
            }
            xq[32 * b + i] = (int8_t)q;
            sum += q;
        }
        s[b] = sb;
        S[b] = sum;
    }
}

/* code i (0..k-1) of one Q4 row */
int or_q4_code(const uint8_t* row_codes, int64_t i) {
    int64_t b = i / 32, e = i % 32;
    uint8_t byte = row_codes[16 * b + (e % 16)];
    return e < 16 ? (byte & 15) : (byte >> 4);
}

/* code i of one Q6 row: low 4 bits from lo, top 2 bits from hi */
int or_q6_code(const uint8_t* row_lo, const uint8_t* row_hi, int64_t i) {
    int64_t b = i / 32, e = i % 32;
    int low = or_q4_code(row_lo, i);
    uint8_t hbyte = row_hi[8 * b + (e % 8)];
    int high = (hbyte >> (2 * (e / 8))) & 3;
    return low | (high << 4);
}

/* code i of one Q2 row */
int or_q2_code(const uint8_t* row_codes, int64_t i) {
    int64_t b = i / 32, e = i % 32;
    return (row_codes[8 * b + (e % 8)] >> (2 * (e / 8))) & 3;
}

static int code_at(int bits, const uint8_t* lo, const uint8_t* hi, int64_t k, int64_t r, int64_t i) {
    if (bits == 2) return or_q2_code(lo + r * (k / 4), i);
    if (bits == 4) return or_q4_code(lo + r * (k / 2), i);
    return or_q6_code(lo + r * (k / 2), hi + r * (k / 4), i);
}

/* all codes of rows [row0, row0+nrows) as integers [nrows][k] */
void or_codes(int bits, const uint8_t* lo, const uint8_t* hi, int64_t k, int64_t row0, int64_t nrows, int32_t* out) {
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t i = 0; i < k; ++i) out[r * k + i] = code_at(bits, lo, hi, k, row0 + r, i);
}

/* dequantised weights w = scale*code + min in fp64 for rows [row0, row0+nrows) */
void or_dequant_rows(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min,
                     int64_t k, int64_t row0, int64_t nrows, double* out) {
    int64_t nb = k / 32;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t rr = row0 + r;
        for (int64_t i = 0; i < k; ++i) {
            double d = or_half_to_double(scale[rr * nb + i / 32]);
            if (bits == 2) {
                out[r * k + i] = d * (double)(code_at(bits, lo, hi, k, rr, i) - 2);
                continue;
            }
            double m = or_half_to_double(min[rr * nb + i / 32]);
            out[r * k + i] = d * (double)code_at(bits, lo, hi, k, rr, i) + m;
        }
    }
}

/*
 * Integer block dots D[r][b] = sum_{i<32} code(r, 32b+i) * xq(32b+i), the
 * int8 x int4/int6 dot products of the dp4a MMVQ path (genie-ai-runtime,
 * "The decode arc": dp4a int8 MMVQ for Q4_K and Q6_K; oxinfer README,
 * "How it works": int8 SDOT over blocks).  Exact integers.
 */
void or_blockdots(int bits, const uint8_t* lo, const uint8_t* hi, int64_t n, int64_t k, const int8_t* xq,
                  int32_t* D) {
    int64_t nb = k / 32;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            int64_t acc = 0;
            for (int i = 0; i < 32; ++i) acc += (int64_t)code_at(bits, lo, hi, k, r, 32 * b + i) * xq[32 * b + i];
            D[r * nb + b] = (int32_t)acc;
        }
}

/*
 * y_r = sum_i w_deq(r, i) * x_deq(i) over rows [row0, row0+nrows), in fp64:
 * dequantise the weights to fp64 and dot them with the int8-dequantised
 * activation x_deq(i) = s_b * xq(i).  Reading: the oracle's input is the
 * quantised activation, because the method quantises x before the dot
 * (sources as for or_quantize_act); the weights decode as scale*code + min.
 */
void or_gemv(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min, int64_t k,
             const float* x, int64_t row0, int64_t nrows, double* y, int8_t* xq_work, float* s_work,
             int32_t* S_work) {
    or_quantize_act(x, k, xq_work, s_work, S_work);
    int64_t nb = k / 32;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t rr = row0 + r;
        double acc = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            double d = or_half_to_double(scale[rr * nb + i / 32]);
            double w = bits == 2 ? d * (double)(code_at(bits, lo, hi, k, rr, i) - 2)
                                 : d * (double)code_at(bits, lo, hi, k, rr, i) +
                                       or_half_to_double(min[rr * nb + i / 32]);
            double xd = (double)s_work[i / 32] * (double)xq_work[i];
            acc += w * xd;
        }
        y[r] = acc;
    }
}

/* Same, for an explicit list of rows (sampled checks at full size). */
void or_gemv_rows(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min,
                  int64_t k, const float* x, const int64_t* rows, int64_t nrows, double* y, int8_t* xq_work,
                  float* s_work, int32_t* S_work) {
    for (int64_t j = 0; j < nrows; ++j)
        or_gemv(bits, lo, hi, scale, min, k, x, rows[j], 1, y + j, xq_work, s_work, S_work);
}

/*
 * Final-logit soft-capping, l = c * tanh(z / c) (genie-ai-runtime, "What
 * Gemma 4 E2B actually is": final-logit soft-capping; oxinfer README, "How
 * it works": tied softcapped LM head).  Reading: c <= 0 means no cap.
 */
double or_softcap(double z, double c) {
    if (c <= 0.0) return z;
    return c * tanh(z / c);
}

void or_softcap_vec(const double* z, int64_t n, double c, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_softcap(z[i], c);
}

/*
 * Deterministic argmax (Gemma WebGPU Engine, "Roadmap": two deterministic
 * argmax dispatches).  Reading: the lowest index among the maxima; a NaN is
 * never greater than anything; if every value is NaN the result is 0.
 */
int64_t or_argmax_f64(const double* v, int64_t n) {
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(v[i])) continue;
        if (best < 0 || v[i] > v[best]) best = i;
    }
    return best < 0 ? 0 : best;
}

int64_t or_argmax_f32(const float* v, int64_t n) {
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(v[i])) continue;
        if (best < 0 || v[i] > v[best]) best = i;
    }
    return best < 0 ? 0 : best;
}

/*
 * Normalised Walsh-Hadamard transform of one group of g values (g a power of
 * two): u_i = g^(-1/2) * sum_j (-1)^popcount(i & j) x_j (needle.js "Inference
 * backends", "Pure TypeScript": the CQ kernel applies a normalised fast
 * Walsh-Hadamard transform to each activation group).  Written as the
 * explicit O(g^2) sum over the Sylvester-ordered Hadamard matrix, not as a
 * butterfly.  Reading: natural (Sylvester) order, scale applied once.
 */
void or_wht(const double* x, int64_t g, double* u) {
    double scale = 1.0 / sqrt((double)g);
    for (int64_t i = 0; i < g; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < g; ++j) {
            int sign = __builtin_popcountll((unsigned long long)(i & j)) & 1;
            acc += sign ? -x[j] : x[j];
        }
        u[i] = scale * acc;
    }
}

/*
 * CQ matvec over the selected rows [row_start, row_start + row_count):
 *   u = WHT of each group of x;  y_j = scale_r * sum_i codebook[idx(r, i)] * u_i,
 * r = row_start + j (needle.js "Inference backends": "Pure TypeScript" for
 * the transform then packed codebook-index decode inside the dot product;
 * "Custom backend" for the selected-row range).  fp64 throughout.
 */
void or_cq_matvec(const uint8_t* idx, const uint16_t* codebook, const uint16_t* row_scale, int64_t k, int64_t group,
                  int64_t row_start, int64_t row_count, const float* x, double* y, double* xwork, double* uwork) {
    for (int64_t i = 0; i < k; ++i) xwork[i] = (double)x[i];
    for (int64_t g0 = 0; g0 < k; g0 += group) or_wht(xwork + g0, group, uwork + g0);
    double cb[16];
    for (int c = 0; c < 16; ++c) cb[c] = or_half_to_double(codebook[c]);
    for (int64_t j = 0; j < row_count; ++j) {
        int64_t r = row_start + j;
        const uint8_t* row = idx + r * (k / 2);
        double acc = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            uint8_t byte = row[i / 2];
            int c = (i % 2 == 0) ? (byte & 15) : (byte >> 4);
            acc += cb[c] * uwork[i];
        }
        y[j] = or_half_to_double(row_scale[r]) * acc;
    }
}

/*
 * log sum_i exp(v_i) over all n values, in fp64 (max-shifted).  The full-vocabulary
 * normaliser of the selected token's log-probability (needle.js "Inference
 * backends", "Resident layers": the selected ID is returned with its
 * full-vocabulary log probability).  Reading: NaN values are skipped.
 */
double or_logsumexp(const double* v, int64_t n) {
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
        if (!isnan(v[i]) && v[i] > m) m = v[i];
    if (m == -INFINITY) return -INFINITY;
    if (m == INFINITY) return INFINITY; /* exp(+inf) dominates the sum */
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i)
        if (!isnan(v[i])) s += exp(v[i] - m);
    return m + log(s);
}

/*
 * Constrained selection (needle.js "Resident layers": grammar-allowed token IDs
 * uploaded as an ascending list, the selected ID and its full-vocabulary log
 * probability returned).  Reading: the selected ID is the allowed ID of the
 * largest value, the lowest ID among equals, NaN never selected; allowed == NULL
 * means every ID.  Returns the ID (-1 if nothing can be selected) and writes
 * v[id] - logsumexp(v) to *logprob.
 */
int64_t or_select(const double* v, int64_t n, const int32_t* allowed, int64_t n_allowed, double* logprob) {
    int64_t best = -1;
    const int64_t cnt = allowed ? n_allowed : n;
    for (int64_t j = 0; j < cnt; ++j) {
        const int64_t id = allowed ? (int64_t)allowed[j] : j;
        if (id < 0 || id >= n || isnan(v[id])) continue;
        if (best < 0 || v[id] > v[best] || (v[id] == v[best] && id < best)) best = id;
    }
    *logprob = best < 0 ? NAN : v[best] - or_logsumexp(v, n);
    return best;
}
