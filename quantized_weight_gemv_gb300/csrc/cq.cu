// Codebook-quantised (CQ) matvec in the Hadamard domain.
//
// needle.js "Inference backends", "Pure TypeScript": the activation is first put
// through a normalised fast Walsh-Hadamard transform per group, then the packed
// 4-bit codebook indices are decoded inside the dot product, so the inverse
// transform of the weights is never materialised.  "TypeGPU": one 32-lane group
// per output row.  "Custom backend": an optional contiguous row range.
//
// Two kernels.  cq_regs_kernel (rows of up to 64 values per lane: k <= 2048, groups of
// 256 to 1024) keeps each lane's transformed values in registers for all its rows; it
// is described above its definition.  cq_kernel takes every other shape: each warp
// first pulls the packed indices of its first row into L1 and loads that row's scale
// (weights: under programmatic dependent launch they are read before the preceding
// kernel has finished), so that their latency overlaps the transform.  Each CTA
// transforms x itself: a warp owns a group of G = 32*J values, lane l holding elements
// J*l .. J*l+J-1.  The butterflies over the low log2(J) index bits run in registers,
// those over the lane bits through __shfl_xor_sync.  The result is kept in shared
// memory transposed (element J*l + j at j*32 + l), so that in the dot loop lane l
// reads its J values without bank conflicts.
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

// Up to GM groups per row (k = ng * G, ng <= GM, G = 32*J, J >= 8, GM * J <= 64): the
// transform is split over all eight warps and each warp keeps several rows in flight.
//  * Before griddepcontrol.wait each warp loads the packed indices of up to RPW of its
//    rows into registers (lane l, group g: the J/2 bytes of the group's elements
//    J*l .. J*l+J-1) and their scales: under programmatic dependent launch the weight
//    reads overlap the preceding kernel's tail.
//  * Transform, every group at once: thread t holds elements E*t .. E*t+E-1 of each group
//    (E = J/8).  The butterflies over the low log2(E) index bits run in registers, the
//    next five (the lane bits) through __shfl_xor_sync, and the top three (the warp bits)
//    after one pass through shared memory, where each of 4J threads takes the eight
//    elements c + 4J*m (m < 8) of column c of every group.  Its results, times 1/sqrt(G),
//    go to the dot layout (element J*l + e of group g at (g*J + e)*33 + l: the padded row
//    stride keeps the scatter free of bank conflicts).
//  * Each lane then holds its ng*J transformed values in registers for all its rows: per
//    row only the codebook look-ups (16 entries in 16 distinct banks: conflict-free for
//    any index pattern) and the fused multiply-adds remain.
template <int J, int GM>
__global__ void __launch_bounds__(256) cq_regs_kernel(CqParams p) {
    constexpr int E = J / 8;
    constexpr int RPW = GM * J <= 32 ? 4 : 2;  // rows per warp loaded before the wait
    constexpr int NWI = (J + 7) / 8;           // index words per lane, row and group
    constexpr int NW = GM * NWI;               // index words per lane and row
    constexpr int G = 32 * J;
    static_assert(J >= 8, "at least one element per thread");
    static_assert(GM * J <= 64, "transformed values per lane held in registers");
    extern __shared__ __align__(16) float sm[];
    constexpr int SU = 33;  // row stride of the dot layout (32 + 1: conflict-free scatter)
    float* su = sm;                // [GM J][SU], dot layout
    float* sc = sm + GM * J * SU;  // [GM][32 J], natural order (transform scratch)
    __shared__ float scb[16];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int tw = gridDim.x * 8;
    const int gw = blockIdx.x * 8 + wid;
    const int my_rows = p.row_count > gw ? (p.row_count - gw + tw - 1) / tw : 0;
    const int ng = GM == 1 ? 1 : p.k / G;  // groups per row
    const size_t row_bytes = (size_t)(p.k >> 1);
    auto has = [&](int g) { return GM == 1 || g < ng; };

    auto load_row = [&](int r, uint32_t(&w)[NW]) {
        const uint8_t* rp = p.idx + (size_t)r * row_bytes + (J / 2) * lane;
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            uint32_t t[NWI];
#pragma unroll
            for (int q = 0; q < NWI; ++q) t[q] = 0u;
            if (has(g)) load_lane_indices<J>(rp + (size_t)g * (G / 2), t);
#pragma unroll
            for (int q = 0; q < NWI; ++q) w[g * NWI + q] = t[q];
        }
    };
    uint32_t wi[RPW][NW];
    unsigned short sh[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        sh[i] = 0;
#pragma unroll
        for (int q = 0; q < NW; ++q) wi[i][q] = 0u;
        if (i < my_rows) {
            const int r = p.row_start + gw + i * tw;
            load_row(r, wi[i]);
            sh[i] = p.row_scale[r];
        }
    }
    if (threadIdx.x < 16) scb[threadIdx.x] = half_bits_to_float(p.codebook[threadIdx.x]);

    pdl_wait();
    if (threadIdx.x == 0) pdl_launch_dependents();

    // ---- transform: registers, lanes, then warps through shared memory
    const int t = threadIdx.x;
    float v[GM][E];
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        const float* xg = p.x + (size_t)(has(g) ? g : 0) * G;
        if constexpr (E == 1) {
            v[g][0] = xg[t];
        } else if constexpr (E == 2) {
            const float2 a = reinterpret_cast<const float2*>(xg)[t];
            v[g][0] = a.x;
            v[g][1] = a.y;
        } else {
            const float4 a = reinterpret_cast<const float4*>(xg)[t];
            v[g][0] = a.x;
            v[g][1] = a.y;
            v[g][2] = a.z;
            v[g][3] = a.w;
        }
    }
#pragma unroll
    for (int g = 0; g < GM; ++g) {
#pragma unroll
        for (int h = 1; h < E; h <<= 1) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if ((e & h) == 0) {
                    const float a = v[g][e], b = v[g][e + h];
                    v[g][e] = a + b;
                    v[g][e + h] = a - b;
                }
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int g = 0; g < GM; ++g) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float o = __shfl_xor_sync(0xffffffffu, v[g][e], m);
                v[g][e] = upper ? (o - v[g][e]) : (v[g][e] + o);
            }
        }
    }
#pragma unroll
    for (int g = 0; g < GM; ++g)
#pragma unroll
        for (int e = 0; e < E; ++e) sc[g * G + E * t + e] = v[g][e];
    __syncthreads();
    if (t < 4 * J) {
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            float u[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) u[m] = sc[g * G + t + 4 * J * m];
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
            // element i = t + 4J*m of group g goes to (g*J + i % J) * SU + i / J
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int i = t + 4 * J * m;
                su[(g * J + i % J) * SU + i / J] = u[m] * p.inv_sqrt_group;
            }
        }
    }
    __syncthreads();

    float ul[GM * J];
#pragma unroll
    for (int e = 0; e < GM * J; ++e) ul[e] = su[e * SU + lane];

    // ---- the rows: codebook look-ups against the lane's transformed values
    auto lane_dot = [&](const uint32_t(&w)[NW]) {
        float acc = 0.0f;
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            if (!has(g)) continue;
#pragma unroll
            for (int e = 0; e < J; ++e) {
                const uint32_t c = (w[g * NWI + (e >> 3)] >> (4 * (e & 7))) & 15u;
                acc = fmaf(scb[c], ul[g * J + e], acc);
            }
        }
        return acc;
    };
    auto dot_row = [&](const uint32_t(&w)[NW], unsigned short scale_h, int j) {
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
    static_assert(RPW == 4 || RPW == 2, "rows preloaded per warp");
    if constexpr (RPW == 4) {
        if (my_rows >= 3)
            joint(std::integral_constant<int, 4>{});
        else if (my_rows == 2)
            joint(std::integral_constant<int, 2>{});
        else if (my_rows == 1)
            dot_row(wi[0], sh[0], gw);
    } else {
        if (my_rows >= 2)
            joint(std::integral_constant<int, 2>{});
        else if (my_rows == 1)
            dot_row(wi[0], sh[0], gw);
    }
    for (int i = RPW; i < my_rows; ++i) {
        const int j = gw + i * tw;
        const int r = p.row_start + j;
        uint32_t w[NW];
        load_row(r, w);
        dot_row(w, p.row_scale[r], j);
    }
}

template <int J, int GM>
static int launch_cq_regs_t(const CqParams& p, const LaunchCtx& lc) {
    auto kern = cq_regs_kernel<J, GM>;
    const size_t smem = (size_t)(33 + 32) * GM * J * sizeof(float);
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
    // the register form while a lane's transformed values fit (ng * J <= 64: k <= 2048),
    // with the smallest group bound that holds the row's groups
    const int ng = p.group > 0 ? p.k / p.group : 0;
    switch (p.group) {
        case 256:
            if (ng == 1) return launch_cq_regs_t<8, 1>(p, lc);
            if (ng == 2) return launch_cq_regs_t<8, 2>(p, lc);
            if (ng <= 4) return launch_cq_regs_t<8, 4>(p, lc);
            if (ng <= 8) return launch_cq_regs_t<8, 8>(p, lc);
            break;
        case 512:
            if (ng == 1) return launch_cq_regs_t<16, 1>(p, lc);
            if (ng == 2) return launch_cq_regs_t<16, 2>(p, lc);
            if (ng <= 4) return launch_cq_regs_t<16, 4>(p, lc);
            break;
        case 1024:
            if (ng == 1) return launch_cq_regs_t<32, 1>(p, lc);
            if (ng == 2) return launch_cq_regs_t<32, 2>(p, lc);
            break;
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
