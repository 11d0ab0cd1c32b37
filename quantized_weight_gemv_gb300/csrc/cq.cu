// Codebook-quantised (CQ) matvec in the Hadamard domain.
//
// needle.js "Inference backends", "Pure TypeScript": the activation is first put
// through a normalised fast Walsh-Hadamard transform per group, then the packed
// 4-bit codebook indices are decoded inside the dot product, so the inverse
// transform of the weights is never materialised.  "TypeGPU": one 32-lane group
// per output row.  "Custom backend": an optional contiguous row range.
//
// Each warp first pulls the packed indices of its first row into L1 and loads that
// row's scale (weights: under programmatic dependent launch they are read before the
// preceding kernel has finished), so that their latency overlaps the transform.  Each
// CTA transforms x itself: a warp owns a group of G = 32*J values, lane l holding
// elements J*l .. J*l+J-1.  The butterflies over the low log2(J) index
// bits run in registers, those over the lane bits through __shfl_xor_sync.  The
// result is kept in shared memory transposed (element J*l + j at j*32 + l), so
// that in the dot loop lane l reads its J values without bank conflicts.
#include <type_traits>

#include "gemv_stream.cuh"  // stream::halving_reduce
#include "qg_internal.h"

namespace qg {

template <int J>
__device__ __forceinline__ void load_lane_group(const float* __restrict__ src, float (&v)[J]) {
    if constexpr (J % 4 == 0) {
#pragma unroll
        for (int q = 0; q < J / 4; ++q) {
            const float4 t = reinterpret_cast<const float4*>(src)[q];
            v[4 * q] = t.x;
            v[4 * q + 1] = t.y;
            v[4 * q + 2] = t.z;
            v[4 * q + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < J; ++j) v[j] = src[j];
    }
}

// J/2 index bytes of one lane as 32-bit words (J/8 words; J = 4 uses the low half of one)
template <int J>
__device__ __forceinline__ void load_lane_indices(const uint8_t* __restrict__ src, uint32_t (&w)[(J + 7) / 8]) {
    if constexpr (J == 32) {
        const uint4 t = ldg_stream16(src);
        w[0] = t.x;
        w[1] = t.y;
        w[2] = t.z;
        w[3] = t.w;
    } else if constexpr (J == 16) {
        const uint2 t = ldg_stream8(src);
        w[0] = t.x;
        w[1] = t.y;
    } else if constexpr (J == 8) {
        w[0] = __ldg(reinterpret_cast<const unsigned int*>(src));
    } else {
        w[0] = ldg_stream2(src);
    }
}

template <int J>
__global__ void __launch_bounds__(256) cq_kernel(CqParams p) {
    constexpr int G = 32 * J;
    extern __shared__ __align__(16) float su[];  // [k], transposed per group
    __shared__ float scb[16];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int ngroups = p.k / G;
    const size_t row_bytes = (size_t)(p.k >> 1);

    // the warp's first row: index lines prefetched into L1, row scale loaded, before the wait
    const int j0 = blockIdx.x * 8 + wid;
    unsigned short scale0 = 0;
    if (j0 < p.row_count) {
        const uint8_t* rp = p.idx + (size_t)(p.row_start + j0) * row_bytes;
        for (size_t off = (size_t)lane * 128; off < row_bytes; off += 32 * 128)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(rp + off));
        scale0 = p.row_scale[p.row_start + j0];
    }
    if (threadIdx.x < 16) scb[threadIdx.x] = half_bits_to_float(p.codebook[threadIdx.x]);

    pdl_wait();
    if (threadIdx.x == 0) pdl_launch_dependents();

    for (int g = wid; g < ngroups; g += 8) {
        float v[J];
        load_lane_group<J>(p.x + (size_t)g * G + J * lane, v);
#pragma unroll
        for (int h = 1; h < J; h <<= 1) {
#pragma unroll
            for (int j = 0; j < J; ++j) {
                if ((j & h) == 0) {
                    const float a = v[j], b = v[j + h];
                    v[j] = a + b;
                    v[j + h] = a - b;
                }
            }
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const float o = __shfl_xor_sync(0xffffffffu, v[j], m);
                v[j] = upper ? (o - v[j]) : (v[j] + o);
            }
        }
#pragma unroll
        for (int j = 0; j < J; ++j) su[g * G + j * 32 + lane] = v[j] * p.inv_sqrt_group;
    }
    __syncthreads();

    for (int j = j0; j < p.row_count; j += gridDim.x * 8) {
        const int r = p.row_start + j;
        const uint8_t* rp = p.idx + (size_t)r * row_bytes;
        float acc = 0.0f;
        for (int g = 0; g < ngroups; ++g) {
            uint32_t w[(J + 7) / 8];
            load_lane_indices<J>(rp + (size_t)g * (G / 2) + (J / 2) * lane, w);
            const float* ug = su + g * G + lane;
#pragma unroll
            for (int e = 0; e < J; ++e) {
                const uint32_t c = (w[e >> 3] >> (4 * (e & 7))) & 15u;
                acc = fmaf(scb[c], ug[e * 32], acc);
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) p.y[j] = half_bits_to_float(j == j0 ? scale0 : p.row_scale[r]) * acc;
    }
}

// One group per row (k == group, G = 32*J, J >= 8): the transform is split over all
// eight warps and each warp keeps several rows in flight.
//  * Before griddepcontrol.wait each warp loads the packed indices of up to RPW of its
//    rows into registers (lane l: the J/2 bytes of elements J*l .. J*l+J-1) and their
//    scales: under programmatic dependent launch the weight reads overlap the preceding
//    kernel's tail.
//  * Transform: thread t holds elements E*t .. E*t+E-1 (E = J/8).  The butterflies over
//    the low log2(E) index bits run in registers, the next five (the lane bits) through
//    __shfl_xor_sync, and the top three (the warp bits) after one pass through shared
//    memory, where each of 4J threads takes the eight elements c + 4J*m (m < 8) of one
//    column c.  Its results, times 1/sqrt(G), go to the dot layout (element J*l + e at
//    e*33 + l: the padded row stride keeps the scatter free of bank conflicts).
//  * Each lane then holds its J transformed values in registers for all its rows: per
//    row only the codebook look-ups (16 entries in 16 distinct banks: conflict-free for
//    any index pattern) and the fused multiply-adds remain.
template <int J>
__global__ void __launch_bounds__(256) cq_onegroup_kernel(CqParams p) {
    constexpr int E = J / 8;
    constexpr int RPW = 4;                 // rows per warp loaded before the wait
    constexpr int NWI = (J + 7) / 8;       // index words per lane and row
    static_assert(J >= 8, "at least one element per thread");
    extern __shared__ __align__(16) float sm[];
    constexpr int SU = 33;  // row stride of the dot layout (32 + 1: conflict-free scatter)
    float* su = sm;           // [J][SU], dot layout
    float* sc = sm + J * SU;  // [32 J], natural order (transform scratch)
    __shared__ float scb[16];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int tw = gridDim.x * 8;
    const int gw = blockIdx.x * 8 + wid;
    const int my_rows = p.row_count > gw ? (p.row_count - gw + tw - 1) / tw : 0;
    const size_t row_bytes = (size_t)(p.k >> 1);

    uint32_t wi[RPW][NWI];
    unsigned short sh[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        sh[i] = 0;
#pragma unroll
        for (int q = 0; q < NWI; ++q) wi[i][q] = 0u;
        if (i < my_rows) {
            const int r = p.row_start + gw + i * tw;
            load_lane_indices<J>(p.idx + (size_t)r * row_bytes + (J / 2) * lane, wi[i]);
            sh[i] = p.row_scale[r];
        }
    }
    if (threadIdx.x < 16) scb[threadIdx.x] = half_bits_to_float(p.codebook[threadIdx.x]);

    pdl_wait();
    if (threadIdx.x == 0) pdl_launch_dependents();

    // ---- transform: registers, lanes, then warps through shared memory
    const int t = threadIdx.x;
    float v[E];
    if constexpr (E == 1) {
        v[0] = p.x[t];
    } else if constexpr (E == 2) {
        const float2 a = reinterpret_cast<const float2*>(p.x)[t];
        v[0] = a.x;
        v[1] = a.y;
    } else {
        const float4 a = reinterpret_cast<const float4*>(p.x)[t];
        v[0] = a.x;
        v[1] = a.y;
        v[2] = a.z;
        v[3] = a.w;
    }
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if ((e & h) == 0) {
                const float a = v[e], b = v[e + h];
                v[e] = a + b;
                v[e + h] = a - b;
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, v[e], m);
            v[e] = upper ? (o - v[e]) : (v[e] + o);
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) sc[E * t + e] = v[e];
    __syncthreads();
    if (t < 4 * J) {
        float u[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) u[m] = sc[t + 4 * J * m];
#pragma unroll
        for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                if ((m & h) == 0) {
                    const float a = u[m], b = u[m + h];
                    u[m] = a + b;
                    u[m + h] = a - b;
                }
            }
        }
        // element i = t + 4J*m goes to (i % J) * SU + i / J
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int i = t + 4 * J * m;
            su[(i % J) * SU + i / J] = u[m] * p.inv_sqrt_group;
        }
    }
    __syncthreads();

    float ul[J];
#pragma unroll
    for (int e = 0; e < J; ++e) ul[e] = su[e * SU + lane];

    // ---- the rows: codebook look-ups against the lane's transformed values
    auto lane_dot = [&](const uint32_t(&w)[NWI]) {
        float acc = 0.0f;
#pragma unroll
        for (int e = 0; e < J; ++e) {
            const uint32_t c = (w[e >> 3] >> (4 * (e & 7))) & 15u;
            acc = fmaf(scb[c], ul[e], acc);
        }
        return acc;
    };
    auto dot_row = [&](const uint32_t(&w)[NWI], unsigned short scale_h, int j) {
        const float acc = warp_sum(lane_dot(w));
        if (lane == 0) p.y[j] = half_bits_to_float(scale_h) * acc;
    };
    // the preloaded rows: the lane sums of RR of them reduced together (RR - 1 halving
    // shuffles and log2(32 / RR) more instead of 5 per row); lane (32 / RR) i then holds
    // row i's total
    auto joint = [&](auto rr) {
        constexpr int RR = decltype(rr)::value;
        float acc[RR];
#pragma unroll
        for (int i = 0; i < RR; ++i) acc[i] = lane_dot(wi[i]);
        stream::halving_reduce<RR, 5>(acc);
        constexpr int LPR = 32 / RR;
        const int i = lane / LPR;
        uint32_t s_me = sh[0];
#pragma unroll
        for (int r = 1; r < RR; ++r) s_me = i == r ? sh[r] : s_me;
        if (lane % LPR == 0 && i < my_rows) p.y[gw + i * tw] = half_bits_to_float((unsigned short)s_me) * acc[0];
    };
    static_assert(RPW == 4, "rows preloaded per warp");
    if (my_rows >= 3)
        joint(std::integral_constant<int, 4>{});
    else if (my_rows == 2)
        joint(std::integral_constant<int, 2>{});
    else if (my_rows == 1)
        dot_row(wi[0], sh[0], gw);
    for (int i = RPW; i < my_rows; ++i) {
        const int j = gw + i * tw;
        const int r = p.row_start + j;
        uint32_t w[NWI];
        load_lane_indices<J>(p.idx + (size_t)r * row_bytes + (J / 2) * lane, w);
        dot_row(w, p.row_scale[r], j);
    }
}

template <int J>
static int launch_cq_onegroup_t(const CqParams& p, const LaunchCtx& lc) {
    auto kern = cq_onegroup_kernel<J>;
    const size_t smem = (size_t)(33 + 32) * J * sizeof(float);
    if (int rc = ensure_smem_attr((const void*)kern, smem, lc)) return rc;
    int grid = (p.row_count + 7) / 8;  // at least one row per warp
    if (grid > lc.sm_count * 2) grid = lc.sm_count * 2;
    if (grid < 1) grid = 1;
    return launch_kernel(kern, dim3(grid), dim3(256), smem, lc, p);
}

template <int J>
static int launch_cq_t(const CqParams& p, const LaunchCtx& lc) {
    auto kern = cq_kernel<J>;
    const size_t smem = (size_t)p.k * sizeof(float);
    if (smem > (size_t)lc.max_smem_optin) return QG_ERR_UNSUPPORTED;
    if (int rc = ensure_smem_attr((const void*)kern, smem, lc)) return rc;
    int grid = (p.row_count + 7) / 8;
    if (grid > lc.sm_count * 8) grid = lc.sm_count * 8;
    if (grid < 1) grid = 1;
    return launch_kernel(kern, dim3(grid), dim3(256), smem, lc, p);
}

int launch_cq(const CqParams& p, const LaunchCtx& lc) {
    if (p.k == p.group) {
        switch (p.group) {
            case 256:
                return launch_cq_onegroup_t<8>(p, lc);
            case 512:
                return launch_cq_onegroup_t<16>(p, lc);
            case 1024:
                return launch_cq_onegroup_t<32>(p, lc);
        }
    }
    switch (p.group) {
        case 128:
            return launch_cq_t<4>(p, lc);
        case 256:
            return launch_cq_t<8>(p, lc);
        case 512:
            return launch_cq_t<16>(p, lc);
        case 1024:
            return launch_cq_t<32>(p, lc);
    }
    return QG_ERR_UNSUPPORTED;
}

}  // namespace qg
