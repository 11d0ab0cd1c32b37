// Shared device helpers of the quantized-weight GEMV kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qgemv.h"

namespace qg {

// Codes OR-ed into the device error word (its address is a kernel parameter) by a
// kernel whose bounded wait ran out (1, 2, 4, 8), or by a CTA of the persistent chain
// that stopped on the chain's abort word (16).  Host side: qg_device_error() reads and
// clears it.
enum : unsigned { ERR_WAIT_FULL = 1u, ERR_WAIT_EMPTY = 2u, ERR_WAIT_DRAIN = 4u, ERR_WAIT_GRID = 8u, ERR_ABORTED = 16u };

constexpr int WARP = 32;
// 1 s: far beyond any legitimate wait of these kernels, short enough to keep the context alive.
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ unsigned short ldg_stream2(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float half_bits_to_float(unsigned short b) {
    return __half2float(__ushort_as_half(b));
}

// ---------------------------------------------------------------- activation quantisation
// One block of 32 values held one per lane: s = max|x| / 127 (IEEE fp32 division),
// q = clamp(round-half-even(x / s), -127, 127), q = 0 when s == 0.  Returns q; s and
// the block sum S are returned through references (valid in every lane).
// clamp(round-half-even(fl32(x / s)), -127, 127) for s > 0, the quotient correctly
// rounded as an fp32 division gives it.  inv = 1/s correctly rounded: t = x * inv is
// then within 2^-23 |x/s| <= 1.6e-5 of x/s, and fl32(x/s) within 2^-24 |x/s|, so the
// two can round to different integers only when t lies within ~2.3e-5 of a
// half-integer.  Outside 1/4096 of one, rint(t) is the answer; inside (and for a NaN
// or infinite t) the exact quotient decides.
// The nearest integer to t comes from fp32 adds: t + 1.5*2^23 rounds to an integer
// (round-half-even, |t| < 2^22) whose value sits in the low mantissa bits.
__device__ __forceinline__ int quant_code(float x, float s, float inv) {
    constexpr float MAGIC = 12582912.0f;  // 1.5 * 2^23
    const float t = x * inv;
    const float r = __fadd_rn(t, MAGIC);
    const float qf = __fsub_rn(r, MAGIC);
    int q;
    if (fabsf(t - qf) < 0.5f - (1.0f / 4096.0f))
        q = __float_as_int(r) - 0x4B400000;
    else
        q = __float2int_rn(__fdiv_rn(x, s));
    return max(-127, min(127, q));
}

__device__ __forceinline__ int quantize_lane(float x, float& s, int& S) {
    float a = fabsf(x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    s = __fdiv_rn(a, 127.0f);
    int q = 0;
    if (s != 0.0f) q = quant_code(x, s, __frcp_rn(s));
    int t = q;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    S = t;
    return q;
}

// Shared-memory image of a quantised activation column with nb blocks:
//   lo[nb][16] int8 : elements 0..15 of each block;  hi[nb][16] int8 : elements 16..31;
//   s[nb] fp32 ; S[nb] fp32 (block sums, exact in fp32).
// The split halves let a lane fetch the 16 activations that meet the low (or high)
// nibbles of its 16-byte code block with one conflict-free 128-bit load.
struct XqView {
    int8_t* lo;
    int8_t* hi;
    float* s;
    float* S;
};
__device__ __forceinline__ XqView xq_view(unsigned char* base, int nb) {
    XqView v;
    v.lo = reinterpret_cast<int8_t*>(base);
    v.hi = reinterpret_cast<int8_t*>(base + 16 * nb);
    v.s = reinterpret_cast<float*>(base + 32 * nb);
    v.S = reinterpret_cast<float*>(base + 36 * nb);
    return v;
}
__host__ __device__ constexpr int xq_bytes(int nb) { return 40 * nb; }

// Cooperative quantisation of `batch` activation columns x[c][k] into per-column
// XqViews (column c at base + c * stride) by NT threads (t = 0..NT-1, whole warps).
// The columns' runs of V consecutive values (V = 4 or 8) form one index space; thread
// t takes run i*NT + t, so 32/V consecutive lanes hold one block of 32 of one column
// and a block's max and sum take log2(32/V) shuffles.  All CHUNK loads of a round are
// issued before any is used, so the prologue costs about one L2 round trip per round.
// L2ONLY reads x with ld.global.cg: for a vector other SMs wrote during the same
// launch, which the non-coherent (and L1) path may hold stale.  (What a preceding
// kernel wrote is visible to every read issued after griddepcontrol.wait.)
template <int NT, bool L2ONLY, int V>
__device__ __forceinline__ void quantize_runs(const float* __restrict__ x, int k, int batch, unsigned char* base,
                                              int stride, int t) {
    constexpr int F = V / 4;         // float4s per run
    constexpr int CHUNK = 8 / F;     // runs per thread per round (8 float4 loads in flight)
    constexpr int LPB = 32 / V;      // lanes per block
    const int nb = k >> 5;
    const int nrun = k / V;          // runs per column
    const int total = batch * nrun;
    const int m = t & (LPB - 1);     // run within the block
    // column of run idx: idx / nrun, a shift when nrun is a power of two (k = 2^j)
    const int nrun_log2 = (nrun & (nrun - 1)) == 0 ? __ffs(nrun) - 1 : -1;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    for (int r0 = 0; r0 < total; r0 += NT * CHUNK) {
        float4 r[CHUNK][F];
#pragma unroll
        for (int i = 0; i < CHUNK; ++i) {
            const int idx = r0 + i * NT + t;
#pragma unroll
            for (int f = 0; f < F; ++f)
                r[i][f] = idx < total ? (L2ONLY ? __ldcg(x4 + F * idx + f) : __ldg(x4 + F * idx + f))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < CHUNK; ++i) {
            if (r0 + i * NT >= total) break;  // the same for every thread: nothing left in this round
            const int idx = r0 + i * NT + t;
            float a = 0.0f;
#pragma unroll
            for (int f = 0; f < F; ++f)
                a = fmaxf(a, fmaxf(fmaxf(fabsf(r[i][f].x), fabsf(r[i][f].y)), fmaxf(fabsf(r[i][f].z), fabsf(r[i][f].w))));
#pragma unroll
            for (int o = 1; o < LPB; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            const float s = __fdiv_rn(a, 127.0f);
            int q[V];
#pragma unroll
            for (int e = 0; e < V; ++e) q[e] = 0;
            if (s != 0.0f) {
                const float inv = __frcp_rn(s);
#pragma unroll
                for (int f = 0; f < F; ++f) {
                    q[4 * f + 0] = quant_code(r[i][f].x, s, inv);
                    q[4 * f + 1] = quant_code(r[i][f].y, s, inv);
                    q[4 * f + 2] = quant_code(r[i][f].z, s, inv);
                    q[4 * f + 3] = quant_code(r[i][f].w, s, inv);
                }
            }
            int S = 0;
            uint32_t packed[F];
#pragma unroll
            for (int f = 0; f < F; ++f) {
                S += (q[4 * f] + q[4 * f + 1]) + (q[4 * f + 2] + q[4 * f + 3]);
                packed[f] = (uint32_t)(q[4 * f] & 255) | ((uint32_t)(q[4 * f + 1] & 255) << 8) |
                            ((uint32_t)(q[4 * f + 2] & 255) << 16) | ((uint32_t)(q[4 * f + 3] & 255) << 24);
            }
#pragma unroll
            for (int o = 1; o < LPB; o <<= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
            if (idx < total) {
                const int c = batch == 1 ? 0 : nrun_log2 >= 0 ? idx >> nrun_log2 : idx / nrun;
                const int b = (idx - c * nrun) / LPB;
                const XqView v = xq_view(base + (size_t)c * stride, nb);
                int8_t* dst = m < LPB / 2 ? v.lo + 16 * b + V * m : v.hi + 16 * b + V * (m - LPB / 2);
                if constexpr (F == 2)
                    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
                else
                    *reinterpret_cast<uint32_t*>(dst) = packed[0];
                if (m == 0) {
                    v.s[b] = s;
                    v.S[b] = (float)S;
                }
            }
        }
    }
}

// Runs of 8 values when every thread gets at least one (the scale, its reciprocal
// and the shuffles then serve 8 values), else runs of 4 (more threads in the one round).
template <int NT, bool L2ONLY = false>
__device__ __forceinline__ void quantize_x_cols(const float* __restrict__ x, int k, int batch, unsigned char* base,
                                                int stride, int t) {
    if (batch * k >= 8 * NT)
        quantize_runs<NT, L2ONLY, 8>(x, k, batch, base, stride, t);
    else
        quantize_runs<NT, L2ONLY, 4>(x, k, batch, base, stride, t);
}

// ---------------------------------------------------------------- dp4a block dots
// 16 code bytes of a Q4 block: word w (bytes 4w..4w+3) carries codes 4w..4w+3 in its
// low nibbles and codes 16+4w..16+4w+3 in its high nibbles.

// dp4a with unsigned bytes in a and signed bytes in b
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Q4 block dot straight from the 16 code bytes: the low nibbles are masked out
// (values 0..15), the high nibbles are masked in place (16 * code, 0..240) and dotted
// as unsigned bytes, so the second sum is exactly 16x the high-half dot.
__device__ __forceinline__ int block_dot_q4(uint4 c, uint4 xlo, uint4 xhi) {
    int a = __dp4a((int)(c.x & 0x0F0F0F0Fu), (int)xlo.x, 0);
    int b = dp4a_us(c.x & 0xF0F0F0F0u, xhi.x, 0);
    a = __dp4a((int)(c.y & 0x0F0F0F0Fu), (int)xlo.y, a);
    b = dp4a_us(c.y & 0xF0F0F0F0u, xhi.y, b);
    a = __dp4a((int)(c.z & 0x0F0F0F0Fu), (int)xlo.z, a);
    b = dp4a_us(c.z & 0xF0F0F0F0u, xhi.z, b);
    a = __dp4a((int)(c.w & 0x0F0F0F0Fu), (int)xlo.w, a);
    b = dp4a_us(c.w & 0xF0F0F0F0u, xhi.w, b);
    return a + (b >> 4);
}

// Q2 block dot from its 8 code bytes (word h0 = bytes 0..3, h1 = bytes 4..7; byte t
// holds codes t, t+8, t+16, t+24 at bit pairs 0..3).  Bit pair s of h0 / h1 meets the
// activation word 2s / 2s+1 of the block (elements 8s..8s+3 / 8s+4..8s+7), i.e. words
// of the low half for s < 2 and of the high half for s >= 2.  Every pair is masked in
// place (4^s x code, at most 192 as an unsigned byte) and the pairs are summed from the
// top, the running sum shifted right by two before the next pair: after pair 3 it is a
// multiple of 64, after pair 2 of 16, after pair 1 of 4, so each shift divides exactly
// and pair 0 leaves the plain dot.  A seed of 64 t (added before the first shift) comes
// out as t: the zero-point term -2 S_b of the Q2 format rides along at no cost.
// |sum| <= 64 (|t| + 2 * 4 * 3 * 127) stays far inside int32 for |t| < 2^20.
__device__ __forceinline__ int block_dot_q2(uint2 c, uint4 xlo, uint4 xhi, int seed64 = 0) {
    int a = dp4a_us(c.x & 0xC0C0C0C0u, xhi.z, seed64);
    a = dp4a_us(c.y & 0xC0C0C0C0u, xhi.w, a);
    a >>= 2;
    a = dp4a_us(c.x & 0x30303030u, xhi.x, a);
    a = dp4a_us(c.y & 0x30303030u, xhi.y, a);
    a >>= 2;
    a = dp4a_us(c.x & 0x0C0C0C0Cu, xlo.z, a);
    a = dp4a_us(c.y & 0x0C0C0C0Cu, xlo.w, a);
    a >>= 2;
    a = __dp4a((int)(c.x & 0x03030303u), (int)xlo.x, a);
    return __dp4a((int)(c.y & 0x03030303u), (int)xlo.y, a);
}

// block dot of any format from its raw words: Q4 cw; Q6 cw and hw; Q2 hw (8 code bytes)
template <int BITS>
__device__ __forceinline__ int qdot(uint4 cw, uint2 hw, uint4 xlo, uint4 xhi) {
    if constexpr (BITS == 2) {
        (void)cw;
        return block_dot_q2(hw, xlo, xhi);
    } else if constexpr (BITS == 4) {
        (void)hw;
        return block_dot_q4(cw, xlo, xhi);
    } else {
        // Q6 = low nibbles (the Q4 plane) + 16 x the high bit pairs (the Q2 plane layout):
        // by linearity the dot is the Q4 dot of the low plane plus 16 x the Q2 dot of the
        // high plane, exact in int32
        return block_dot_q4(cw, xlo, xhi) + (block_dot_q2(hw, xlo, xhi) << 4);
    }
}

// s_b * (scale * D + min * S_b) in fp32
__device__ __forceinline__ float block_combine(int D, float d, float m, float s, float S) {
    return s * fmaf(d, (float)D, m * S);
}

// Q2 (w = scale * (code - 2)): s_b * scale * (D - 2 S_b), the integer factor exact in
// fp32 (|D|, |S_b| < 2^14)
__device__ __forceinline__ float block_combine_q2(int D, float d, float s, float S) {
    return (s * d) * fmaf(-2.0f, S, (float)D);
}

// the combine of a format from the block's binary16 scale (and min) bits
template <int BITS>
__device__ __forceinline__ float combine(int D, unsigned short dh, unsigned short mh, float s, float S) {
    if constexpr (BITS == 2) {
        (void)mh;
        return block_combine_q2(D, half_bits_to_float(dh), s, S);
    } else {
        return block_combine(D, half_bits_to_float(dh), half_bits_to_float(mh), s, S);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------- soft-cap + argmax ordering
// l = c * tanh(z / c) (c > 0; c <= 0: no cap), z / c taken as z times inv_c = the
// correctly rounded 1/c, computed once per kernel (within an ulp of the quotient)
__device__ __forceinline__ float softcap_inv(float c) { return c > 0.0f ? __frcp_rn(c) : 0.0f; }
__device__ __forceinline__ float softcap_apply(float z, float c, float inv_c) {
    return c > 0.0f ? c * tanhf(z * inv_c) : z;
}

// (value, index) order for the argmax: larger value first, then lower index; NaN never wins.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    if (v != v) return false;
    if (bv != bv) return true;
    return v > bv || (v == bv && i < bi);
}

struct ArgmaxPartial {
    float value;
    int index;
};

// Workspace of the vocabulary argmax: an arrival counter and the best (value, index)
// so far as one packed key (argmax_key); both zero between calls.
struct VocabWorkspace {
    unsigned int counter;
    unsigned int pad0;
    unsigned long long best;
    unsigned int pad[60];
};
static_assert(sizeof(VocabWorkspace) == 256, "vocabulary workspace layout");

// Workspace of the constrained selection: a counter, then one partial per CTA holding
// an online log-sum-exp (max m, sum of exp(l - m)) and a best (value, index).
constexpr int SELECT_MAX_CTAS = 1024;
struct SelectPartial {
    float m, s, bv;
    int bi;
};
struct SelectWorkspace {
    unsigned int counter;
    int scratch_index;  // the unconstrained argmax of the vocabulary kernel, unused afterwards
    unsigned int pad[62];
    SelectPartial part[SELECT_MAX_CTAS];
};

// (m, s) <- the log-sum-exp pair of the union of two sets, each held as its maximum m
// and sum of exp(value - m); an empty set is (-inf, 0), an infinite term makes the
// result (+inf, 1)
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == INFINITY || m2 == INFINITY) {
        m = INFINITY;
        s = 1.0f;
        return;
    }
    if (m == -INFINITY) {
        m = m2;
        s = s2;
        return;
    }
    const float M = fmaxf(m, m2);
    s = s * expf(m - M) + s2 * expf(m2 - M);
    m = M;
}

__device__ __forceinline__ void select_warp_reduce(float& m, float& s, float& bv, int& bi) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        lse_merge(m, s, m2, s2);
        if (better(v2, i2, bv, bi)) {
            bv = v2;
            bi = i2;
        }
    }
}

// block-wide merge of (m, s, bv, bi); the result is valid in thread 0
__device__ __forceinline__ void select_block_reduce(float& m, float& s, float& bv, int& bi, SelectPartial* sred) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    select_warp_reduce(m, s, bv, bi);
    __syncthreads();
    if (lane == 0) sred[wid] = SelectPartial{m, s, bv, bi};
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < nw; ++w) {
            lse_merge(m, s, sred[w].m, sred[w].s);
            if (better(sred[w].bv, sred[w].bi, bv, bi)) {
                bv = sred[w].bv;
                bi = sred[w].bi;
            }
        }
    }
}

// This CTA's partial (each thread's share in m, s, bv, bi) goes to ws; the last CTA to
// finish merges every CTA's partial, writes the selected id (-1 when nothing allowed
// is selectable) and bv - log-sum-exp, and re-arms the counter.  No CTA waits on
// another.  Called by all threads; gridDim.x <= SELECT_MAX_CTAS.
__device__ __forceinline__ void select_finish(float m, float s, float bv, int bi, SelectWorkspace* ws,
                                              int32_t* token, float* logprob, SelectPartial* sred /* [8] */,
                                              int* slast) {
    select_block_reduce(m, s, bv, bi, sred);
    if (threadIdx.x == 0) {
        ws->part[blockIdx.x] = SelectPartial{m, s, bv, bi};
        // acquire-release arrival: the partial above is visible to the last CTA
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(&ws->counter) : "memory");
        *slast = prev == gridDim.x - 1;
    }
    __syncthreads();
    if (!*slast) return;
    __threadfence();
    m = -INFINITY;
    s = 0.0f;
    bv = __int_as_float(0x7fc00000);
    bi = 0x7fffffff;
    for (int c = threadIdx.x; c < (int)gridDim.x; c += blockDim.x) {
        const float cm = __ldcg(&ws->part[c].m), cs = __ldcg(&ws->part[c].s);
        const float cv = __ldcg(&ws->part[c].bv);
        const int ci = __ldcg(&ws->part[c].bi);
        lse_merge(m, s, cm, cs);
        if (better(cv, ci, bv, bi)) {
            bv = cv;
            bi = ci;
        }
    }
    select_block_reduce(m, s, bv, bi, sred);
    if (threadIdx.x == 0) {
        const bool found = bi != 0x7fffffff;
        *token = found ? bi : -1;
        *logprob = found ? bv - (m + logf(s)) : __int_as_float(0x7fc00000);
        ws->counter = 0u;
    }
}

// (value, index) as one 64-bit key whose unsigned order is the argmax order of better():
// the high word maps the float's bits to an order-preserving unsigned (negative values
// complemented, positive ones with the sign bit set; -0 taken as +0, since the two
// compare equal), the low word is ~index, so that of equal values the lower index has
// the larger key.  NaN (never the best) is key 0, below every number's.
__device__ __forceinline__ unsigned long long argmax_key(float v, int i) {
    if (v != v) return 0ull;
    const unsigned u = __float_as_uint(v + 0.0f);
    const unsigned o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)o << 32) | (unsigned long long)(~(unsigned)i);
}

// Block-wide (value, index) reduction, then one atomic max of the block's key into the
// workspace and an arrival count; the last block to arrive reads the merged key, writes
// its index and re-arms the workspace.  The count is an acquire-release add: a block's
// max is visible to whichever block arrives after it, and the last one's read sees all.
// No block waits on another (measured on GB300, int2 262144 x 1536: 23.9 -> 22.3 us
// against a merge of per-block partials by the last block).  Called by all threads.
__device__ __forceinline__ void argmax_finish(float bv, int bi, VocabWorkspace* ws, int32_t* out,
                                              ArgmaxPartial* sred /* >= blockDim/32 entries */) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
        }
    }
    if (lane == 0) sred[wid] = ArgmaxPartial{bv, bi};
    __syncthreads();
    if (threadIdx.x != 0) return;
    for (int w = 1; w < nw; ++w)
        if (better(sred[w].value, sred[w].index, bv, bi)) {
            bv = sred[w].value;
            bi = sred[w].index;
        }
    const unsigned long long key = argmax_key(bv, bi);
    if (key) atomicMax(&ws->best, key);
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(&ws->counter) : "memory");
    if (prev != gridDim.x - 1) return;
    unsigned long long k;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(k) : "l"(&ws->best) : "memory");
    // every value NaN (or no rows): index 0, as the lowest index
    *out = k ? (int)~(unsigned)k : 0;
    ws->best = 0ull;
    ws->counter = 0u;
}

}  // namespace qg
