// Plain-load quantized-weight GEMV kernels: any k % 32 == 0, any n.
//
// One warp per output row (the warp-per-row GEMV of genie-ai-runtime, "The decode
// arc"; one 32-lane group per row in needle.js "Inference backends", "TypeGPU").
// Lane l takes blocks l, l+32, ... of the row: each block is one 16-byte load of
// codes (a whole Q4 block), decoded in registers and dotted with the int8
// activation by dp4a (genie-ai-runtime, "The decode arc": dp4a int8 MMVQ
// "instead of dequant-to-fp"; its 32-bit-word unpack of the Q4_K fast path).
// Every CTA quantises the activation columns into shared memory first.
#include "qg_internal.h"

namespace qg {

template <int BITS, int BC, int EPI>
__global__ void __launch_bounds__(256) gemv_plain_kernel(PlainParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int nb = p.k >> 5;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int xstride = xq_stride(nb);

    pdl_wait();  // x, y and the workspace may belong to the preceding kernel
    if (threadIdx.x == 0) pdl_launch_dependents();

    quantize_x_cols<256>(p.x, p.k, p.batch, smem, xstride, threadIdx.x);
    __syncthreads();

    float bv = __int_as_float(0x7fc00000);
    int bi = 0x7fffffff;
    const size_t code_row = (size_t)(BITS == 2 ? p.k >> 2 : p.k >> 1), hi_row = (size_t)(p.k >> 2);

    for (int r = blockIdx.x * 8 + wid; r < p.n; r += gridDim.x * 8) {
        float acc[BC];
#pragma unroll
        for (int c = 0; c < BC; ++c) acc[c] = 0.0f;
        const uint8_t* crow = p.lo + (size_t)r * code_row;
        const uint8_t* hrow = (BITS == 6) ? p.hi + (size_t)r * hi_row : nullptr;
        const uint16_t* srow = p.scale + (size_t)r * nb;
        const uint16_t* mrow = BITS == 2 ? nullptr : p.min + (size_t)r * nb;  // Q2: zero point 2, no min plane
#pragma unroll 2
        for (int b = lane; b < nb; b += 32) {
            uint4 cw = make_uint4(0u, 0u, 0u, 0u);
            uint2 hw = make_uint2(0u, 0u);
            if constexpr (BITS == 2) {
                hw = ldg_stream8(crow + 8 * (size_t)b);
            } else {
                cw = ldg_stream16(crow + 16 * (size_t)b);
                if constexpr (BITS == 6) hw = ldg_stream8(hrow + 8 * (size_t)b);
            }
            const unsigned short dh = ldg_stream2(srow + b);
            const unsigned short mh = BITS == 2 ? (unsigned short)0 : ldg_stream2(mrow + b);
#pragma unroll
            for (int c = 0; c < BC; ++c) {
                if (c < p.batch) {
                    const XqView v = xq_view(smem + c * xstride, nb);
                    const uint4 xl = *reinterpret_cast<const uint4*>(v.lo + 16 * b);
                    const uint4 xh = *reinterpret_cast<const uint4*>(v.hi + 16 * b);
                    acc[c] += combine<BITS>(qdot<BITS>(cw, hw, xl, xh), dh, mh, v.s[b], v.S[b]);
                }
            }
        }
#pragma unroll
        for (int c = 0; c < BC; ++c) acc[c] = warp_sum(acc[c]);
        if constexpr (EPI == EPI_STORE) {
            if (lane == 0) {
#pragma unroll
                for (int c = 0; c < BC; ++c)
                    if (c < p.batch) p.y[(size_t)c * p.n + r] = acc[c];
            }
        } else {
            const float l = softcap_apply(acc[0], p.softcap, softcap_inv(p.softcap));
            if (lane == 0 && p.y) p.y[r] = l;
            if (better(l, r, bv, bi)) {
                bv = l;
                bi = r;
            }
        }
    }
    if constexpr (EPI == EPI_ARGMAX) {
        __shared__ ArgmaxPartial sred[8];
        argmax_finish(bv, bi, p.ws, p.argmax, sred);
    }
}

// Exposed step: per-block activation quantisation of `batch` rows of x, one warp per block.
__global__ void __launch_bounds__(256) quantize_act_kernel(const float* __restrict__ x, int k, int batch,
                                                           int8_t* __restrict__ xq, float* __restrict__ xs,
                                                           int32_t* __restrict__ xsum) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long total = (long long)batch * (k >> 5);
    for (long long blk = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); blk < total;
         blk += (long long)gridDim.x * 8) {
        float s;
        int S;
        const int q = quantize_lane(x[blk * 32 + lane], s, S);
        xq[blk * 32 + lane] = (int8_t)q;
        if (lane == 0) {
            xs[blk] = s;
            xsum[blk] = S;
        }
    }
}

// Exposed step: integer block dots D[r][b], one thread per (row, block).
template <int BITS>
__global__ void __launch_bounds__(256) blockdots_kernel(const uint8_t* __restrict__ lo, const uint8_t* __restrict__ hi,
                                                        int n, int k, const int8_t* __restrict__ xq,
                                                        int32_t* __restrict__ dots) {
    pdl_wait();
    const int nb = k >> 5;
    const long long total = (long long)n * nb;
    for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const long long r = t / nb;
        const int b = (int)(t - r * nb);
        uint4 cw = make_uint4(0u, 0u, 0u, 0u);
        uint2 hw = make_uint2(0u, 0u);
        if constexpr (BITS == 2) {
            hw = ldg_stream8(lo + r * (k >> 2) + 8 * b);
        } else {
            cw = ldg_stream16(lo + r * (k >> 1) + 16 * b);
            if constexpr (BITS == 6) hw = ldg_stream8(hi + r * (k >> 2) + 8 * b);
        }
        const uint4 xl = *reinterpret_cast<const uint4*>(xq + 32 * b);
        const uint4 xh = *reinterpret_cast<const uint4*>(xq + 32 * b + 16);
        dots[t] = qdot<BITS>(cw, hw, xl, xh);
    }
}

// ---------------------------------------------------------------- host launchers
template <int BITS, int BC, int EPI>
static int launch_plain_t(const PlainParams& p, const LaunchCtx& lc) {
    auto kern = gemv_plain_kernel<BITS, BC, EPI>;
    const int nb = p.k >> 5;
    const size_t smem = (size_t)xq_stride(nb) * p.batch;
    if (smem > (size_t)lc.max_smem_optin) return QG_ERR_UNSUPPORTED;
    if (int rc = ensure_smem_attr((const void*)kern, smem, lc)) return rc;
    int rows_ctas = (p.n + 7) / 8;
    int grid = lc.sm_count * 8;
    if (EPI == EPI_ARGMAX) grid = lc.sm_count * 4;
    if (grid > rows_ctas) grid = rows_ctas;
    if (grid < 1) grid = 1;
    return launch_kernel(kern, dim3(grid), dim3(256), smem, lc, p);
}

int launch_plain(const PlainParams& p, int bits, int epi, const LaunchCtx& lc) {
    const int bc = p.batch <= 1 ? 1 : p.batch <= 2 ? 2 : p.batch <= 4 ? 4 : p.batch <= 8 ? 8 : 16;
    if (epi == EPI_ARGMAX)
        return bits == 2   ? launch_plain_t<2, 1, EPI_ARGMAX>(p, lc)
               : bits == 4 ? launch_plain_t<4, 1, EPI_ARGMAX>(p, lc)
                           : launch_plain_t<6, 1, EPI_ARGMAX>(p, lc);
#define QG_CASE(B)                                                     \
    case B:                                                            \
        return bits == 2   ? launch_plain_t<2, B, EPI_STORE>(p, lc)    \
               : bits == 4 ? launch_plain_t<4, B, EPI_STORE>(p, lc)    \
                           : launch_plain_t<6, B, EPI_STORE>(p, lc);
    switch (bc) {
        QG_CASE(1)
        QG_CASE(2)
        QG_CASE(4)
        QG_CASE(8)
        QG_CASE(16)
    }
#undef QG_CASE
    return QG_ERR_UNSUPPORTED;
}

// The plain-read floor: every 16-byte word of src read once with streaming loads (four
// per thread in flight), XOR-folded into *out.  The time of a kernel that only reads a
// buffer once is the floor of any kernel streaming the same bytes in the same launch
// setting (the decode bound of the oxinfer README, "Performance": every weight byte is
// read once per token).  The reads start before griddepcontrol.wait, as the GEMV
// kernels' weight streams do; *out is written after it.
__global__ void __launch_bounds__(512) read_floor_kernel(const uint4* __restrict__ src, size_t n16, uint32_t* out) {
    if (threadIdx.x == 0) pdl_launch_dependents();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = ldg_stream16(src + i), b = ldg_stream16(src + i + stride);
        const uint4 c = ldg_stream16(src + i + 2 * stride), d = ldg_stream16(src + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n16; i += stride) {
        const uint4 a = ldg_stream16(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    // one atomic per CTA: same-address atomics from every warp would serialise in L2
    __shared__ uint32_t sacc[16];
    if ((threadIdx.x & 31) == 0) sacc[threadIdx.x >> 5] = acc;
    __syncthreads();
    pdl_wait();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) acc ^= sacc[w];
        atomicXor(out, acc);
    }
}

int launch_read_floor(const void* src, size_t bytes, uint32_t* out, const LaunchCtx& lc) {
    const size_t n16 = bytes >> 4;
    long long grid = (long long)lc.sm_count * 4;  // 2048 threads per SM
    const long long need = (long long)((n16 + 511) / 512);
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    return launch_kernel(read_floor_kernel, dim3((unsigned)grid), dim3(512), 0, lc,
                         reinterpret_cast<const uint4*>(src), n16, out);
}

int launch_quantize_act(const float* x, int k, int batch, int8_t* xq, float* xs, int32_t* xsum, const LaunchCtx& lc) {
    const long long blocks = (long long)batch * (k >> 5);
    long long grid = (blocks + 7) / 8;
    if (grid > lc.sm_count * 16) grid = lc.sm_count * 16;
    return launch_kernel(quantize_act_kernel, dim3((unsigned)grid), dim3(256), 0, lc, x, k, batch, xq, xs, xsum);
}

int launch_blockdots(int bits, const uint8_t* lo, const uint8_t* hi, int n, int k, const int8_t* xq, int32_t* dots,
                     const LaunchCtx& lc) {
    const long long total = (long long)n * (k >> 5);
    long long grid = (total + 255) / 256;
    if (grid > lc.sm_count * 16) grid = lc.sm_count * 16;
    if (bits == 2)
        return launch_kernel(blockdots_kernel<2>, dim3((unsigned)grid), dim3(256), 0, lc, lo, hi, n, k, xq, dots);
    if (bits == 4)
        return launch_kernel(blockdots_kernel<4>, dim3((unsigned)grid), dim3(256), 0, lc, lo, hi, n, k, xq, dots);
    return launch_kernel(blockdots_kernel<6>, dim3((unsigned)grid), dim3(256), 0, lc, lo, hi, n, k, xq, dots);
}

}  // namespace qg
