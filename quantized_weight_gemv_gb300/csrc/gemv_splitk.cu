// Split-K streaming GEMV for short-N / long-K matrices (k = 4096, 8192 or 16384 and
// few rows per CTA), e.g. a decoder's down projection 2048 x 16384 called on its own.
//
// genie-ai-runtime, "v1.3.0 - split-K decode attention": when the output is short
// and the reduction long, a row-per-warp grid leaves the GPU idle; the reduction
// dimension is split over more workers and the partial results are combined exactly
// afterwards.  Here the single-matrix streaming kernel would make every CTA quantise
// the whole k-long activation (for 2048 x 16384, 304 CTAs x 64 KB of x against 21 MB
// of weights) and give each warp whole 16384-wide rows.  Instead:
//  * the k range is cut into S slices of 2048 values (64 blocks of 32); a thread-block
//    cluster of S CTAs owns a contiguous row range, CTA s of the cluster slice s;
//  * each CTA quantises only its 2048 activations and streams its slice of the rows
//    exactly as the streaming kernel streams a k = 2048 matrix: per-warp bulk-copy
//    rings (one copy per row and plane, rows of the slice are 1 KB apart from the next
//    row's), stages of R slice rows, dp4a block dots, fp32 combine, halving tree;
//  * each slice row's partial sum stays in the CTA's shared memory; after a cluster
//    barrier CTA s adds, for rows s, s+S, ..., the S partials in slice order through
//    distributed shared memory and stores y.  The sum order is fixed: the result does
//    not depend on timing.
// Every mbarrier wait is bounded; on expiry the kernel records the error word, drains
// its copies in flight (bounded) and still meets both cluster barriers.
#include <cooperative_groups.h>

#include "gemv_stream_launch.cuh"

namespace cg = cooperative_groups;

namespace qg {
namespace splitk {

using namespace stream;

constexpr int NBS = 64;  // blocks of 32 per k slice (2048 values)
constexpr int W = 8;     // warps per CTA

template <int BITS>
__host__ __device__ constexpr int sb_of() {
    return stage_blocks<BITS, 1, NBS>();  // 256 blocks (Q2: 512) per stage
}

template <int BITS, int S>
__global__ void __launch_bounds__(256, 2) gemv_splitk_kernel(StreamParams p) {
    constexpr int SB = sb_of<BITS>();
    constexpr int JL = SB / 32;    // blocks per lane per stage
    constexpr int R = SB / NBS;    // slice rows per stage
    constexpr int JR = JL / R;     // blocks per lane and row (2)
    constexpr int NXB = NBS / 32;  // activation blocks a lane meets (2)
    using SL = Slot<BITS, SB>;

    extern __shared__ __align__(128) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int s = (int)cluster.block_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.stages;

    unsigned char* slots = smem + (size_t)warp * D * SL::BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)W * D * SL::BYTES) + warp * D;
    unsigned char* xqbase = smem + xq_offset(W * D, SL::BYTES);
    float* spart = reinterpret_cast<float*>(xqbase + xq_stride(NBS));

    const int nbt = p.k >> 5;  // blocks per full row
    const int ncl = gridDim.x / S;
    const int cl = blockIdx.x / S;
    const long long r0 = (long long)cl * p.n / ncl;
    const long long r1 = (long long)(cl + 1) * p.n / ncl;
    const int nrows = (int)(r1 - r0);
    const int nunits = (nrows + R - 1) / R;
    const int my_units = nunits > warp ? (nunits - warp + W - 1) / W : 0;

    const uint64_t pol = policy_evict_first();
    // unit t of this warp (stage rows r0 + R*(warp + W*t) ...) into slot `slot`: one copy
    // per slice row and plane
    auto issue = [&](int t, int slot) {
        const int u = warp + W * t;
        const long long row = r0 + (long long)u * R;
        const int rows_u = min(R, nrows - u * R);
        unsigned char* st = slots + (size_t)slot * SL::BYTES;
        uint64_t* bar = &full[slot];
        mbar_arrive_expect_tx(bar, (uint32_t)(rows_u * NBS * SL::BPB));
        for (int r = 0; r < rows_u; ++r) {
            const size_t blk0 = (size_t)(row + r) * nbt + (size_t)s * NBS;
            const int off = r * NBS;
            bulk_g2s(st + off * SL::CODE, p.lo + blk0 * SL::CODE, NBS * SL::CODE, bar, pol);
            if constexpr (BITS == 6) bulk_g2s(st + SL::HI + off * 8, p.hi + blk0 * 8, NBS * 8, bar, pol);
            bulk_g2s(st + SL::SC + off * 2, p.scale + blk0, NBS * 2, bar, pol);
            if constexpr (BITS != 2) bulk_g2s(st + SL::MN + off * 2, p.min + blk0, NBS * 2, bar, pol);
        }
    };

    if (lane == 0) {
        pdl_launch_dependents();
        for (int i = 0; i < D; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
        for (int t = 0; t < D && t < my_units; ++t) issue(t, t);
    }
    __syncwarp();

    // ---- this slice's activations (after the preceding kernel, which may have written x)
    pdl_wait();
    quantize_x_cols<256>(p.x + (size_t)s * NBS * 32, NBS * 32, 1, xqbase, xq_stride(NBS), threadIdx.x);
    __syncthreads();

    // block f = lane + 32 j of a stage is block (lane + 32 (j % 2)) of slice row j / 2
    uint4 xl[NXB], xh[NXB];
    float xs[NXB], xS[NXB];
    {
        const XqView v = xq_view(xqbase, NBS);
#pragma unroll
        for (int j = 0; j < NXB; ++j) {
            const int blk = lane + 32 * j;
            xl[j] = *reinterpret_cast<const uint4*>(v.lo + 16 * blk);
            xh[j] = *reinterpret_cast<const uint4*>(v.hi + 16 * blk);
            xs[j] = v.s[blk];
            xS[j] = v.S[blk];
        }
    }

    int slot = 0;
    uint32_t phase = 0;
    int failed_at = -1;
    for (int t = 0; t < my_units; ++t, slot = slot + 1 == D ? 0 : slot + 1, phase ^= slot == 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], phase))) {  // warp-uniform
            if (lane == 0) atomicOr(p.err, ERR_WAIT_FULL);
            failed_at = t;
            break;
        }
        const int u = warp + W * t;
        const int rows_u = min(R, nrows - u * R);
        const unsigned char* st = slots + (size_t)slot * SL::BYTES;

        uint4 cw[JL];
        uint2 hw[JL];
        unsigned short dh[JL], mh[JL];
#pragma unroll
        for (int j = 0; j < JL; ++j) {
            const int fb = lane + 32 * j;
            if constexpr (BITS == 2) {
                cw[j] = make_uint4(0u, 0u, 0u, 0u);
                hw[j] = *reinterpret_cast<const uint2*>(st + 8 * fb);
                mh[j] = 0;
            } else {
                cw[j] = *reinterpret_cast<const uint4*>(st + 16 * fb);
                if constexpr (BITS == 6)
                    hw[j] = *reinterpret_cast<const uint2*>(st + SL::HI + 8 * fb);
                else
                    hw[j] = make_uint2(0u, 0u);
                mh[j] = *reinterpret_cast<const unsigned short*>(st + SL::MN + 2 * fb);
            }
            dh[j] = *reinterpret_cast<const unsigned short*>(st + SL::SC + 2 * fb);
        }
        __syncwarp();
        if (lane == 0 && t + D < my_units) {
            fence_proxy_async();  // the slot's generic reads are done before the async refill
            issue(t + D, slot);
        }

        // slice row r of the stage: its JR blocks per lane are j = JR r .. JR r + JR - 1.
        // Rows past the stage's last row are computed on stale slot bytes and never kept.
        float rs[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float a = 0.0f;
#pragma unroll
            for (int q = 0; q < JR; ++q) {
                const int j = r * JR + q;
                const int xj = j % NXB;
                a += combine<BITS>(qdot<BITS>(cw[j], hw[j], xl[xj], xh[xj]), dh[j], mh[j], xs[xj], xS[xj]);
            }
            rs[r] = a;
        }
        halving_reduce<R, 5>(rs);  // lane l: the total of row l / (32 / R)
        constexpr int LPR = 32 / R;
        if ((lane & (LPR - 1)) == 0) {
            const int r = lane / LPR;
            if (r < rows_u) spart[u * R + r] = rs[0];
        }
    }
    if (failed_at >= 0 && lane == 0) {
        // copies still in flight land in this CTA's shared memory: wait for them (bounded)
        for (int t = failed_at; t < my_units && t < failed_at + D; ++t)
            if (!mbar_wait(&full[t % D], (uint32_t)((t / D) & 1))) atomicOr(p.err, ERR_WAIT_DRAIN);
    }

    // every slice's partial sums are in its CTA's shared memory
    cluster.sync();
    for (int i = s + S * (int)threadIdx.x; i < nrows; i += S * (int)blockDim.x) {
        float v = 0.0f;
#pragma unroll
        for (int q = 0; q < S; ++q) v += cluster.map_shared_rank(spart, q)[i];
        p.y[r0 + i] = v;
    }
    cluster.sync();  // no CTA leaves while another still reads its shared memory
}

template <int BITS, int S>
int launch_t(StreamParams p, const LaunchCtx& lc) {
    using SL = Slot<BITS, sb_of<BITS>()>;
    constexpr int R = sb_of<BITS>() / NBS;
    auto kern = gemv_splitk_kernel<BITS, S>;
    // The grid is the clusters that are resident at once (clusters of S CTAs are placed
    // within one GPC, so fewer than SMs / S may fit), sized with the shared memory of the
    // largest row range a cluster can get; one CTA per SM at most (a second CTA per SM
    // adds no stream at these sizes, and the next call's CTAs then find room: 2048 x
    // 16384 8.25 -> 7.77 us, 1024 x 4096 3.68 -> 3.00 us back to back on GB300).
    const size_t cap = (size_t)lc.max_smem_optin - 1024;
    int ncl = lc.sm_count / S;
    int D = 1;
    size_t smem = 0;
    for (int pass = 0; pass < 2; ++pass) {
        if (ncl > p.n) ncl = p.n;
        if (ncl < 1) ncl = 1;
        const int rows_max = (p.n + ncl - 1) / ncl;
        const int units_max = (rows_max + R - 1) / R;
        const int per_warp = (units_max + W - 1) / W;
        // every stage of a warp in flight at once when two fit, else double buffering
        D = stream::env_int("QG_SPLITK_SLOTS", per_warp < 2 ? 1 : 2);
        if (D < 1) D = 1;
        if (D > 4) D = 4;
        const size_t fixed = (size_t)xq_stride(NBS) + (size_t)rows_max * 4;
        smem = xq_offset(W * D, SL::BYTES) + fixed;
        while (smem > cap && D > 1) {
            --D;
            smem = xq_offset(W * D, SL::BYTES) + fixed;
        }
        if (smem > cap) return QG_ERR_UNSUPPORTED;
        if (int rc = ensure_smem_attr((const void*)kern, smem, lc)) return rc;
        if (pass == 0) {
            const int fit = max_active_clusters((const void*)kern, S, W * 32, smem, lc);
            if (fit < 1) return QG_ERR_UNSUPPORTED;
            if (fit >= ncl) break;
            ncl = fit;  // fewer clusters: more rows each, size the shared memory again
        }
    }
    p.stages = D;
    p.err = lc.err;
    LaunchCtx lc2 = lc;
    lc2.cluster = S;
    return launch_kernel(kern, dim3(ncl * S), dim3(W * 32), smem, lc2, p);
}

template <int BITS>
int launch_bits(const StreamParams& p, const LaunchCtx& lc) {
    switch (p.k >> 11) {
        case 2: return launch_t<BITS, 2>(p, lc);
        case 4: return launch_t<BITS, 4>(p, lc);
        case 8: return launch_t<BITS, 8>(p, lc);
    }
    return QG_ERR_UNSUPPORTED;
}

}  // namespace splitk

// Split k when the activation is long (k = 4096, 8192, 16384) and the matrix short:
// below 8192 rows every CTA of the row-split kernel would quantise the whole
// activation for a few rows' weights.
bool splitk_wanted(int n, int k, int batch, int epi) {
    if (stream::env_int("QG_SPLITK", 1) == 0) return false;  // diagnostics: the row-split kernel
    return epi == EPI_STORE && batch == 1 && (k == 4096 || k == 8192 || k == 16384) && n <= 8192;
}

int launch_splitk(const StreamParams& p, int bits, const LaunchCtx& lc) {
    if (bits == 2) return splitk::launch_bits<2>(p, lc);
    return bits == 4 ? splitk::launch_bits<4>(p, lc) : splitk::launch_bits<6>(p, lc);
}

}  // namespace qg
