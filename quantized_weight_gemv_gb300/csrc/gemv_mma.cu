// Small-batch Q4 MMVQ on tensor cores (batch 8..16).
//
// With B activation columns the Q4 GEMV becomes a thin dense contraction (oxinfer
// README, "Speculative decoding": at Q4 the multi-token int8 kernels are
// instruction-bound).  Per block of 32 weights the integer dots D[r][c] =
// sum code * xq are computed with mma.sync m16n8k16 (f16 in, f32 accumulate), fresh
// for every block so that the per-block scales are applied exactly as in the
// single-column kernels:  y[c][r] += s[c] * (d[r] * D[r][c] + m[r] * S[c]).
// Exactness: codes 0..15 (and 16 * code for the high nibbles, <= 240) and int8
// activations are exact in f16, each product is an integer below 2^15 and each
// 16-term dot below 2^16, so every partial sum is exact in f32.
//
// Operand mapping (16 weight rows x 8 columns x 16 k per mma):
//  * the k order inside a block is permuted so that a thread's own 32-bit code word
//    is its A fragment: thread (g = lane/4, t = lane%4) reads bytes 4t..4t+3 of the
//    16-byte block of rows g and g+8; their low nibbles are elements 4t..4t+3 (first
//    mma, k-slots 2t, 2t+1, 8+2t, 9+2t), their high nibbles elements 16+4t..16+4t+3
//    (second mma).  Nibbles become f16 with the 0x6400 magic number: bits
//    0x6400 | c read as half are 1024 + c, minus 1024 exactly.
//  * the B fragments (activations) are written in the same permuted order straight
//    from the quantisation: each float4 of x quantises to exactly one 8-byte fragment.
//  * warps of a CTA split a group of 16-row blocks by k chunks of 512; partial sums
//    meet in shared memory.  Code words, scales and mins are loaded from global
//    memory straight into registers, eight blocks ahead.
#include <cuda_fp16.h>

#include "qg_internal.h"

namespace qg {
namespace mma {

constexpr int KC = 16;  // blocks per k chunk (512 elements)
constexpr int NW = 8;   // warps per CTA

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ uint32_t hsub1024(uint32_t v) {
    const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&v), __half2half2(__ushort_as_half(0x6400)));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// A fragments of one block from the code words of rows g (w0) and g+8 (w1)
__device__ __forceinline__ void a_frags(uint32_t w0, uint32_t w1, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
    const uint32_t p0 = __byte_perm(w0, 0u, 0x4140), q0 = __byte_perm(w0, 0u, 0x4342);
    const uint32_t p1 = __byte_perm(w1, 0u, 0x4140), q1 = __byte_perm(w1, 0u, 0x4342);
    lo[0] = hsub1024((p0 & 0x000F000Fu) | 0x64006400u);
    lo[1] = hsub1024((p1 & 0x000F000Fu) | 0x64006400u);
    lo[2] = hsub1024((q0 & 0x000F000Fu) | 0x64006400u);
    lo[3] = hsub1024((q1 & 0x000F000Fu) | 0x64006400u);
    hi[0] = hsub1024((p0 & 0x00F000F0u) | 0x64006400u);
    hi[1] = hsub1024((p1 & 0x00F000F0u) | 0x64006400u);
    hi[2] = hsub1024((q0 & 0x00F000F0u) | 0x64006400u);
    hi[3] = hsub1024((q1 & 0x00F000F0u) | 0x64006400u);
}

__device__ __forceinline__ uint32_t pack_h2(int a, int b) {
    const __half2 h = __halves2half2(__int2half_rn(a), __int2half_rn(b));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Shared layout: frag[nb][2][NT][32] uint2 | sv[nb][8*NT] f32 | Sv[nb][8*NT] f32 | part[NW][16][8*NT] f32
template <int NT>
struct Smem {
    __host__ __device__ static size_t frag_bytes(int nb) { return (size_t)nb * 2 * NT * 32 * 8; }
    __host__ __device__ static size_t sv_off(int nb) { return frag_bytes(nb); }
    __host__ __device__ static size_t Sv_off(int nb) { return sv_off(nb) + (size_t)nb * 8 * NT * 4; }
    __host__ __device__ static size_t part_off(int nb) { return Sv_off(nb) + (size_t)nb * 8 * NT * 4; }
    __host__ __device__ static size_t bytes(int nb) { return part_off(nb) + (size_t)NW * 16 * 8 * NT * 4; }
};

// Quantise the B activation columns straight into B fragments.  float4 number idx of
// column c (elements 4m..4m+3 of block b, m = idx & 7) becomes the fragment of lane
// 4*(c%8) + (m%4), k half m/4, tile c/8.
template <int NT>
__device__ __forceinline__ void quantize_to_frags(const float* __restrict__ X, int k, int batch, unsigned char* sm) {
    const int nb = k >> 5;
    uint2* frag = reinterpret_cast<uint2*>(sm);
    float* sv = reinterpret_cast<float*>(sm + Smem<NT>::sv_off(nb));
    float* Sv = reinterpret_cast<float*>(sm + Smem<NT>::Sv_off(nb));
    const int nf4 = k >> 2;
    const int total = 8 * NT * nf4;  // columns beyond the batch quantise zeros
    constexpr int CHUNK = 8;
    for (int r0 = 0; r0 < total; r0 += NW * 32 * CHUNK) {
        float4 rv[CHUNK];
#pragma unroll
        for (int i = 0; i < CHUNK; ++i) {
            const int idx_all = r0 + i * NW * 32 + threadIdx.x;
            const int c = idx_all / nf4;
            rv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx_all < total && c < batch)
                rv[i] = __ldg(reinterpret_cast<const float4*>(X + (size_t)c * k) + (idx_all - c * nf4));
        }
#pragma unroll
        for (int i = 0; i < CHUNK; ++i) {
            const int idx_all = r0 + i * NW * 32 + threadIdx.x;
            const int c = idx_all / nf4;
            const int idx = idx_all - c * nf4;
            const float4 r = rv[i];
            float a = fmaxf(fmaxf(fabsf(r.x), fabsf(r.y)), fmaxf(fabsf(r.z), fabsf(r.w)));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            const float s = __fdiv_rn(a, 127.0f);
            int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
            if (s != 0.0f) {
                q0 = max(-127, min(127, __float2int_rn(__fdiv_rn(r.x, s))));
                q1 = max(-127, min(127, __float2int_rn(__fdiv_rn(r.y, s))));
                q2 = max(-127, min(127, __float2int_rn(__fdiv_rn(r.z, s))));
                q3 = max(-127, min(127, __float2int_rn(__fdiv_rn(r.w, s))));
            }
            int S = q0 + q1 + q2 + q3;
            S += __shfl_xor_sync(0xffffffffu, S, 1);
            S += __shfl_xor_sync(0xffffffffu, S, 2);
            S += __shfl_xor_sync(0xffffffffu, S, 4);
            if (idx_all < total) {
                const int b = idx >> 3, m = idx & 7;
                const int lane = 4 * (c & 7) + (m & 3);
                frag[(((size_t)b * 2 + (m >> 2)) * NT + (c >> 3)) * 32 + lane] =
                    make_uint2(pack_h2(q0, q1), pack_h2(q2, q3));
                if (m == 0) {
                    sv[b * 8 * NT + c] = s;
                    Sv[b * 8 * NT + c] = (float)S;
                }
            }
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(NW * 32, 2) mma_batched_kernel(PlainParams p) {
    extern __shared__ __align__(16) unsigned char sm[];
    const int nb = p.k >> 5;
    const int QC = nb / KC;     // k chunks per row group (1, 2, 4 or 8)
    const int RG = NW / QC;     // row groups per CTA pass
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int my_rg = warp / QC, my_q = warp % QC;

    pdl_wait();
    if (threadIdx.x == 0) pdl_launch_dependents();
    quantize_to_frags<NT>(p.x, p.k, p.batch, sm);
    __syncthreads();

    const uint2* frag = reinterpret_cast<const uint2*>(sm);
    const float* sv = reinterpret_cast<const float*>(sm + Smem<NT>::sv_off(nb));
    const float* Sv = reinterpret_cast<const float*>(sm + Smem<NT>::Sv_off(nb));
    float* part = reinterpret_cast<float*>(sm + Smem<NT>::part_off(nb));

    const int n_groups = (p.n + 15) >> 4;
    const size_t row_bytes = (size_t)(p.k >> 1);
    for (int base = blockIdx.x * RG; base < n_groups; base += gridDim.x * RG) {
        const int grp = base + my_rg;
        float acc[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
        if (grp < n_groups) {
            const int ra = min(grp * 16 + g, p.n - 1), rb = min(grp * 16 + g + 8, p.n - 1);
            const uint8_t* ca = p.lo + (size_t)ra * row_bytes + 4 * t;
            const uint8_t* cb = p.lo + (size_t)rb * row_bytes + 4 * t;
            const uint16_t* da = p.scale + (size_t)ra * nb;
            const uint16_t* db = p.scale + (size_t)rb * nb;
            const uint16_t* ma = p.min + (size_t)ra * nb;
            const uint16_t* mb = p.min + (size_t)rb * nb;
#pragma unroll 1
            for (int half = 0; half < KC; half += 8) {
                const int b0 = my_q * KC + half;
                uint32_t w0[8], w1[8];
                unsigned short dA[8], dB[8], mA[8], mB[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    w0[j] = __ldg(reinterpret_cast<const unsigned int*>(ca + 16 * (b0 + j)));
                    w1[j] = __ldg(reinterpret_cast<const unsigned int*>(cb + 16 * (b0 + j)));
                    dA[j] = __ldg(da + b0 + j);
                    dB[j] = __ldg(db + b0 + j);
                    mA[j] = __ldg(ma + b0 + j);
                    mB[j] = __ldg(mb + b0 + j);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int b = b0 + j;
                    uint32_t alo[4], ahi[4];
                    a_frags(w0[j], w1[j], alo, ahi);
                    const float d0 = half_bits_to_float(dA[j]), d1 = half_bits_to_float(dB[j]);
                    const float m0 = half_bits_to_float(mA[j]), m1 = half_bits_to_float(mB[j]);
#pragma unroll
                    for (int tt = 0; tt < NT; ++tt) {
                        const uint2 bl = frag[(((size_t)b * 2 + 0) * NT + tt) * 32 + lane];
                        const uint2 bh = frag[(((size_t)b * 2 + 1) * NT + tt) * 32 + lane];
                        float dl[4], dh[4];
                        mma_16816(dl, alo, bl.x, bl.y);
                        mma_16816(dh, ahi, bh.x, bh.y);
                        const float2 s2 = *reinterpret_cast<const float2*>(sv + b * 8 * NT + tt * 8 + 2 * t);
                        const float2 S2 = *reinterpret_cast<const float2*>(Sv + b * 8 * NT + tt * 8 + 2 * t);
                        // (row g, col 2t), (row g, col 2t+1), (row g+8, col 2t), (row g+8, col 2t+1)
                        acc[tt][0] += s2.x * fmaf(d0, fmaf(dh[0], 0.0625f, dl[0]), m0 * S2.x);
                        acc[tt][1] += s2.y * fmaf(d0, fmaf(dh[1], 0.0625f, dl[1]), m0 * S2.y);
                        acc[tt][2] += s2.x * fmaf(d1, fmaf(dh[2], 0.0625f, dl[2]), m1 * S2.x);
                        acc[tt][3] += s2.y * fmaf(d1, fmaf(dh[3], 0.0625f, dl[3]), m1 * S2.y);
                    }
                }
            }
        }
        // partial sums of the QC k-chunk warps of each row group meet in shared memory
        float* mine = part + (size_t)warp * 16 * 8 * NT;
#pragma unroll
        for (int tt = 0; tt < NT; ++tt) {
            mine[g * 8 * NT + tt * 8 + 2 * t] = acc[tt][0];
            mine[g * 8 * NT + tt * 8 + 2 * t + 1] = acc[tt][1];
            mine[(g + 8) * 8 * NT + tt * 8 + 2 * t] = acc[tt][2];
            mine[(g + 8) * 8 * NT + tt * 8 + 2 * t + 1] = acc[tt][3];
        }
        __syncthreads();
        // RG row groups x 16 rows x batch columns, one output per thread per step
        for (int o = threadIdx.x; o < RG * 16 * 8 * NT; o += NW * 32) {
            const int rg = o / (16 * 8 * NT);
            const int rem = o - rg * 16 * 8 * NT;
            const int r = rem / (8 * NT), c = rem - r * 8 * NT;
            const int row = (base + rg) * 16 + r;
            if (c < p.batch && row < p.n) {
                float s = 0.0f;
                for (int q = 0; q < QC; ++q) s += part[((size_t)(rg * QC + q) * 16 + r) * 8 * NT + c];
                p.y[(size_t)c * p.n + row] = s;
            }
        }
        __syncthreads();
    }
}

}  // namespace mma

bool mma_supported(int bits, int k, int batch) {
    const int nb = k >> 5;
    return bits == 4 && batch >= 8 && batch <= 16 && (nb == 16 || nb == 32 || nb == 64 || nb == 128);
}

int launch_mma(const PlainParams& p, const LaunchCtx& lc) {
    const int nb = p.k >> 5;
    const int QC = nb / mma::KC, RG = mma::NW / QC;
    const int n_groups = (p.n + 15) >> 4;
    const int NT = p.batch <= 8 ? 1 : 2;
    const size_t smem = NT == 1 ? mma::Smem<1>::bytes(nb) : mma::Smem<2>::bytes(nb);
    const void* kern = NT == 1 ? (const void*)mma::mma_batched_kernel<1> : (const void*)mma::mma_batched_kernel<2>;
    if (int rc = ensure_smem_attr(kern, smem, lc)) return rc;
    int grid = (n_groups + RG - 1) / RG;
    if (grid > lc.sm_count * 2) grid = lc.sm_count * 2;
    if (grid < 1) grid = 1;
    if (NT == 1) return launch_kernel(mma::mma_batched_kernel<1>, dim3(grid), dim3(mma::NW * 32), smem, lc, p);
    return launch_kernel(mma::mma_batched_kernel<2>, dim3(grid), dim3(mma::NW * 32), smem, lc, p);
}

}  // namespace qg
