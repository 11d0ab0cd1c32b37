// Dependent GEMV chain: phases of quantized-weight GEMVs, each phase reading what
// earlier phases wrote, in one persistent cooperative launch.
//
// A decode token is a chain: every projection quantises and reads a vector that an
// earlier projection has just written (Gemma WebGPU Engine, "Decode pipeline";
// genie-ai-runtime, "The decode arc": activation quantised per matmul).  One launch
// per link pays a kernel boundary per link.  Here one CTA per SM walks all phases:
//  * A phase is a list of GEMV descriptors whose inputs all exist before it.  Its work
//    is cut as in the grouped GEMV: units of 256 blocks of 32 (whole rows), or single
//    rows of k/8192 such units; CTA b takes the units whose first bulk-copy tile lies
//    in its equal share of the phase's tiles, warp w every 16th of them from w on.
//  * Each warp pulls weight tiles through a private ring of cp.async.bulk copies
//    completed on mbarriers.  Weights do not depend on the chain, so the ring runs
//    ahead across phase boundaries: while a CTA waits for the others at the end of a
//    phase, its ring is already filling with the next phase's tiles.
//  * Between phases: a grid-wide barrier on an arrival counter in the caller's
//    workspace (fence + atomic add, acquire loads, bounded by %globaltimer, with an
//    abort word that stops every CTA once one gives up), then every CTA quantises the
//    next phase's distinct inputs into shared memory, reading them through L2
//    (ld.global.cg): other SMs wrote them during this launch.
//  * The last CTA to finish re-arms the counters, so the workspace needs no memset
//    between calls.
#include <cstring>

#include "gemv_stream.cuh"

namespace qg {
namespace chain {

using stream::JPL;
using stream::SBW;
constexpr int NW = 16;  // warps per CTA
constexpr int NT = NW * 32;

struct CDesc {
    const uint8_t* lo;
    const uint8_t* hi;
    const uint16_t* scale;
    const uint16_t* min;
    float* y;
    int n;
    int log2nb;       // log2(k / 32), 5..9
    int parts;        // tiles per unit
    int unit_prefix;  // units of the phase's earlier descriptors
    int tile_prefix;  // tiles of the phase's earlier descriptors
    int img;          // byte offset of its input's activation image in shared memory
};

struct CPhase {
    int d0, d1;  // descriptors [d0, d1)
    int units, tiles;
    int in0, in1;  // distinct inputs [in0, in1)
};

struct CInput {
    const float* x;
    int k;
    int img;
};

struct CParams {
    int nphase;
    int slots;  // ring slots per warp
    unsigned int* err;
    unsigned int* ctl;  // [0] barrier arrivals, [1] abort, [2] CTAs finished
    CDesc d[QG_MAX_GROUP];
    CPhase ph[QG_MAX_GROUP];
    CInput in[QG_MAX_GROUP];
};

// descriptor of phase f holding index v of a prefix field (largest d with prefix <= v)
template <typename F>
__device__ __forceinline__ int find_in_phase(const CParams& p, const CPhase& f, int v, F prefix) {
    int lo = f.d0, hi = f.d1 - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix(p.d[mid]) <= v)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// first unit of phase f whose first tile is at or after tile x of the phase
__device__ __forceinline__ int unit_at_tile(const CParams& p, const CPhase& f, long long x) {
    if (x >= f.tiles) return f.units;
    const int di = find_in_phase(p, f, (int)x, [](const CDesc& d) { return d.tile_prefix; });
    const CDesc& d = p.d[di];
    return d.unit_prefix + (int)((x - d.tile_prefix + d.parts - 1) / d.parts);
}

// A warp's walk over its tiles: phase, unit within the phase, tile within the unit.
struct Cursor {
    int f;
    int g;
    int part;
    int d;
    int ue;  // end of this CTA's units in phase f
};

// Place c on the warp's first tile of phase f (c.g >= c.ue: the warp has none there).
// Called about twice per phase and warp, so kept out of line.
__device__ __noinline__ void cursor_begin(const CParams& p, Cursor& c, int f) {
    const CPhase& ph = p.ph[f];
    const long long T = ph.tiles;
    const int ub = unit_at_tile(p, ph, T * blockIdx.x / gridDim.x);
    c.f = f;
    c.ue = unit_at_tile(p, ph, T * (blockIdx.x + 1) / gridDim.x);
    c.g = ub + (int)(threadIdx.x >> 5);
    c.part = 0;
    c.d = c.g < c.ue ? find_in_phase(p, ph, c.g, [](const CDesc& d) { return d.unit_prefix; }) : ph.d0;
}

// next tile of the warp within the phase (c.g >= c.ue once its share is done)
__device__ __forceinline__ void cursor_next(const CParams& p, Cursor& c) {
    if (++c.part == p.d[c.d].parts) {
        c.part = 0;
        c.g += NW;
        const int d1 = p.ph[c.f].d1;
        while (c.d + 1 < d1 && c.g >= p.d[c.d + 1].unit_prefix) ++c.d;
    }
}

// Move on to the next phase that holds a tile for this warp (c.f == nphase: none
// left).  The phase index is carried in a local and the end marker written once,
// after the loop.
__device__ __forceinline__ void cursor_settle(const CParams& p, Cursor& c) {
    int f = c.f;
    while (f < p.nphase && c.g >= c.ue) {
        ++f;
        if (f < p.nphase) cursor_begin(p, c, f);
    }
    c.f = f;
}

template <int BITS>
__device__ __forceinline__ void issue_tile(const CParams& p, const Cursor& c, unsigned char* slot, uint64_t* bar,
                                           uint64_t pol) {
    using SL = stream::Slot<BITS>;
    const CDesc& d = p.d[c.d];
    const int nb = 1 << d.log2nb;
    const int R = nb >= SBW ? 1 : SBW / nb;
    const int ul = c.g - d.unit_prefix;
    const int rows_u = R == 1 ? 1 : min(R, d.n - ul * R);
    const uint32_t blocks = (uint32_t)(nb >= SBW ? SBW : rows_u * nb);
    const size_t blk0 = (size_t)ul * R * nb + (size_t)c.part * SBW;
    stream::mbar_arrive_expect_tx(bar, blocks * SL::BPB);
    stream::bulk_g2s(slot, d.lo + blk0 * SL::CODE, blocks * SL::CODE, bar, pol);
    if constexpr (BITS == 6) stream::bulk_g2s(slot + SL::HI, d.hi + blk0 * 8, blocks * 8, bar, pol);
    stream::bulk_g2s(slot + SL::SC, d.scale + blk0, blocks * 2, bar, pol);
    stream::bulk_g2s(slot + SL::MN, d.min + blk0, blocks * 2, bar, pol);
}

// One tile of unit `ul` of descriptor d: JPL blocks per lane, dotted with the
// activation image in shared memory, rows reduced across the warp and stored.
template <int BITS, int L>
__device__ __forceinline__ void tile_compute(const CDesc& d, const unsigned char* img, int ul, int part,
                                             const uint4 (&cw)[JPL], const uint2 (&hw)[JPL],
                                             const unsigned short (&dh)[JPL], const unsigned short (&mh)[JPL],
                                             float& rowacc) {
    constexpr int NB = 1 << L;
    constexpr int R = NB >= SBW ? 1 : SBW / NB;
    constexpr int PARTS = NB > SBW ? NB / SBW : 1;
    constexpr int JM = NB < SBW ? NB / 32 : JPL;  // distinct activation blocks of a lane
    const int lane = threadIdx.x & 31;
    const int rows_u = R == 1 ? 1 : min(R, d.n - ul * R);
    const XqView v = xq_view(const_cast<unsigned char*>(img), NB);

    float pj[JPL];
#pragma unroll
    for (int j = 0; j < JPL; ++j) {
        const int rloc = NB >= SBW ? 0 : ((lane + 32 * j) >> L);
        const int blk = NB < SBW ? lane + 32 * (j % JM) : part * SBW + lane + 32 * j;
        const uint4 a = *reinterpret_cast<const uint4*>(v.lo + 16 * blk);
        const uint4 b = *reinterpret_cast<const uint4*>(v.hi + 16 * blk);
        const float r = block_combine(qdot<BITS>(cw[j], hw[j], a, b), half_bits_to_float(dh[j]),
                                      half_bits_to_float(mh[j]), v.s[blk], v.S[blk]);
        pj[j] = rloc < rows_u ? r : 0.0f;
    }
    constexpr int JR = JPL / R;
    float rs[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float s = 0.0f;
#pragma unroll
        for (int q = 0; q < JR; ++q) s += pj[r * JR + q];
        rs[r] = s;
    }
    if constexpr (PARTS > 1) {
        rowacc += rs[0];
        if (part != PARTS - 1) return;
        rs[0] = rowacc;
        rowacc = 0.0f;
    }
    stream::halving_reduce<R, 5>(rs);
    constexpr int LPR = 32 / R;
    if ((lane & (LPR - 1)) == 0) {
        const int r = lane / LPR;
        if (r < rows_u) d.y[(long long)ul * R + r] = rs[0];
    }
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned int* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Thread 0 of each CTA: arrive, then wait until `target` arrivals (all CTAs of this
// and every earlier boundary).  False when the wait ran out or another CTA gave up.
__device__ bool grid_barrier(const CParams& p, unsigned target) {
    __threadfence();  // the CTA's outputs (ordered before by __syncthreads) before the arrival
    atomicAdd(p.ctl, 1u);
    if (ld_acquire_gpu(p.ctl) >= target) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (ld_acquire_gpu(p.ctl) >= target) return true;
        if (ld_acquire_gpu(p.ctl + 1) != 0u) return false;
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(p.err, ERR_WAIT_GRID);
            atomicExch(p.ctl + 1, 1u);
            return false;
        }
    }
}

template <int BITS>
__global__ void __launch_bounds__(NT, 1) chain_kernel(const __grid_constant__ CParams p) {
    using SL = stream::Slot<BITS>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.slots;
    unsigned char* slots = smem + (size_t)warp * D * SL::BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NW * D * SL::BYTES) + warp * D;
    unsigned char* img = smem + stream::xq_offset(NW * D, SL::BYTES);
    const uint64_t pol = stream::policy_evict_first();

    if (threadIdx.x == 0) s_abort = 0;
    Cursor ic;  // issue cursor, lane 0 only
    int issued = 0;
    if (lane == 0) {
        for (int s = 0; s < D; ++s) stream::mbar_init(&full[s], 1);
        stream::fence_mbar_init();
        cursor_begin(p, ic, 0);
        cursor_settle(p, ic);
        while (issued < D && ic.f < p.nphase) {
            issue_tile<BITS>(p, ic, slots + (size_t)(issued % D) * SL::BYTES, &full[issued % D], pol);
            ++issued;
            cursor_next(p, ic);
            cursor_settle(p, ic);
        }
    }
    __syncwarp();

    int t = 0;  // tiles consumed by this warp
    for (int f = 0; f < p.nphase; ++f) {
        // ---- phase boundary.  Every thread takes each __syncthreads below the same
        // number of times: s_abort only changes between the first two (thread 0) or
        // after the third (a warp whose tile never landed), and is read between the
        // second and the third.
        __syncthreads();
        if (threadIdx.x == 0) {
            if (s_abort)
                atomicExch(p.ctl + 1, 1u);
            else if (f > 0 && !grid_barrier(p, gridDim.x * (unsigned)f))
                s_abort = 1;
        }
        __syncthreads();
        if (s_abort) break;
        const CPhase& ph = p.ph[f];
        for (int i = ph.in0; i < ph.in1; ++i)
            quantize_x_cols<NT, true>(p.in[i].x, p.in[i].k, 1, img + p.in[i].img, 0, threadIdx.x);
        __syncthreads();

        Cursor cc;
        cursor_begin(p, cc, f);
        float rowacc = 0.0f;
        while (cc.g < cc.ue) {
            const int slot = t % D;
            // all lanes poll; the decision is taken together so that the warp stays converged
            if (!__all_sync(0xffffffffu, stream::mbar_wait(&full[slot], (uint32_t)((t / D) & 1)))) {
                if (lane == 0) atomicOr(p.err, ERR_WAIT_FULL);
                s_abort = 1;
                break;
            }
            const unsigned char* st = slots + (size_t)slot * SL::BYTES;
            uint4 cw[JPL];
            uint2 hw[JPL];
            unsigned short dh[JPL], mh[JPL];
#pragma unroll
            for (int j = 0; j < JPL; ++j) {
                const int fb = lane + 32 * j;
                cw[j] = *reinterpret_cast<const uint4*>(st + 16 * fb);
                if constexpr (BITS == 6)
                    hw[j] = *reinterpret_cast<const uint2*>(st + SL::HI + 8 * fb);
                else
                    hw[j] = make_uint2(0u, 0u);
                dh[j] = *reinterpret_cast<const unsigned short*>(st + SL::SC + 2 * fb);
                mh[j] = *reinterpret_cast<const unsigned short*>(st + SL::MN + 2 * fb);
            }
            __syncwarp();
            if (lane == 0 && ic.f < p.nphase) {
                stream::fence_proxy_async();  // the slot's generic reads are done before the refill
                issue_tile<BITS>(p, ic, slots + (size_t)(issued % D) * SL::BYTES, &full[issued % D], pol);
                ++issued;
                cursor_next(p, ic);
                cursor_settle(p, ic);
            }
            ++t;

            const CDesc& d = p.d[cc.d];
            const unsigned char* xim = img + d.img;
            const int ul = cc.g - d.unit_prefix;
            switch (d.log2nb) {
                case 5:
                    tile_compute<BITS, 5>(d, xim, ul, cc.part, cw, hw, dh, mh, rowacc);
                    break;
                case 6:
                    tile_compute<BITS, 6>(d, xim, ul, cc.part, cw, hw, dh, mh, rowacc);
                    break;
                case 7:
                    tile_compute<BITS, 7>(d, xim, ul, cc.part, cw, hw, dh, mh, rowacc);
                    break;
                case 8:
                    tile_compute<BITS, 8>(d, xim, ul, cc.part, cw, hw, dh, mh, rowacc);
                    break;
                default:
                    tile_compute<BITS, 9>(d, xim, ul, cc.part, cw, hw, dh, mh, rowacc);
                    break;
            }
            cursor_next(p, cc);
        }
    }

    // ---- stopping early: let this warp's copies in flight land before the CTA exits
    if (lane == 0) {
        for (int u = t; u < issued; ++u) {
            if (!stream::mbar_wait(&full[u % D], (uint32_t)((u / D) & 1))) {
                atomicOr(p.err, ERR_WAIT_DRAIN);
                break;
            }
        }
    }
    // ---- the last CTA out re-arms the counters for the next call
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.ctl + 2, 1u) == gridDim.x - 1) {
            atomicExch(p.ctl, 0u);
            atomicExch(p.ctl + 1, 0u);
            atomicExch(p.ctl + 2, 0u);
            __threadfence();
        }
    }
}

}  // namespace chain

size_t chain_workspace_bytes(const qg_gemv_desc* descs, int count, const int* phase_sizes, int nphase) {
    (void)count;
    size_t mx = 0;
    int off = 0;
    for (int f = 0; f < nphase; ++f) {
        const size_t b = grouped_workspace_bytes(descs + off, phase_sizes[f]);
        if (b > mx) mx = b;
        off += phase_sizes[f];
    }
    return (size_t)QG_CHAIN_CTL_BYTES + mx;
}

int launch_chain(int bits, const qg_gemv_desc* descs, int count, const int* phase_sizes, int nphase,
                 unsigned char* ws, const LaunchCtx& lc) {
    using namespace chain;
    (void)count;
    if (lc.flags & QG_FLAG_CHAIN_LAUNCHES) {
        int off = 0;
        bool launched = false;
        for (int f = 0; f < nphase; ++f) {
            LaunchCtx l2 = lc;
            if (launched) l2.flags |= QG_FLAG_PDL;
            bool any = false;
            for (int i = off; i < off + phase_sizes[f]; ++i) any = any || descs[i].n > 0;
            if (any) {
                const int rc = launch_grouped(bits, descs + off, phase_sizes[f], ws + QG_CHAIN_CTL_BYTES, l2);
                if (rc != QG_OK) return rc;
                launched = true;
            }
            off += phase_sizes[f];
        }
        return QG_OK;
    }

    static_assert(sizeof(CParams) < 32000, "chain parameters must fit the kernel parameter space");
    CParams p;
    memset(&p, 0, sizeof(p));
    int m = 0, nf = 0, ni = 0, img_max = 0, off = 0;
    for (int f = 0; f < nphase; ++f) {
        CPhase& P = p.ph[nf];
        P.d0 = m;
        P.in0 = ni;
        long long units = 0, tiles = 0;
        int img = 0;
        for (int i = off; i < off + phase_sizes[f]; ++i) {
            const qg_gemv_desc& s = descs[i];
            if (s.n == 0) continue;
            const int nb = s.k >> 5;
            int l = 0;
            while ((1 << l) < nb) ++l;
            int in = P.in0;
            while (in < ni && !(p.in[in].x == s.x && p.in[in].k == s.k)) ++in;
            if (in == ni) {
                p.in[ni].x = s.x;
                p.in[ni].k = s.k;
                p.in[ni].img = img;
                img += xq_stride(nb);
                ++ni;
            }
            CDesc& d = p.d[m++];
            d.lo = s.lo;
            d.hi = s.hi;
            d.scale = s.scale;
            d.min = s.min;
            d.y = s.y;
            d.n = s.n;
            d.log2nb = l;
            d.img = p.in[in].img;
            const int R = nb >= 256 ? 1 : 256 / nb;
            d.parts = nb > 256 ? nb / 256 : 1;
            const long long du = nb >= 256 ? s.n : (s.n + R - 1) / R;
            d.unit_prefix = (int)units;
            d.tile_prefix = (int)tiles;
            units += du;
            tiles += du * d.parts;
        }
        off += phase_sizes[f];
        if (m == P.d0) continue;  // nothing to compute: no boundary needed
        if (tiles > 0x7fffffffLL) return QG_ERR_UNSUPPORTED;
        P.d1 = m;
        P.in1 = ni;
        P.units = (int)units;
        P.tiles = (int)tiles;
        if (img > img_max) img_max = img;
        ++nf;
    }
    if (nf == 0) return QG_OK;
    p.nphase = nf;
    p.err = lc.err;
    p.ctl = reinterpret_cast<unsigned int*>(ws);

    const int slot = bits == 4 ? stream::Slot<4>::BYTES : stream::Slot<6>::BYTES;
    const size_t cap = (size_t)lc.max_smem_optin - 1024;
    int D = 4;
    while (D > 1 && stream::xq_offset(NW * D, slot) + (size_t)img_max > cap) --D;
    const size_t smem = stream::xq_offset(NW * D, slot) + (size_t)img_max;
    if (smem > cap) return QG_ERR_UNSUPPORTED;
    p.slots = D;
    const void* kern = bits == 4 ? (const void*)chain_kernel<4> : (const void*)chain_kernel<6>;
    if (int e = ensure_smem_attr(kern, smem, lc)) return e;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return QG_ERR_CUDA;
    }
    if (per_sm < 1) return QG_ERR_UNSUPPORTED;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)lc.sm_count);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = bits == 4 ? cudaLaunchKernelEx(&cfg, chain_kernel<4>, p)
                                    : cudaLaunchKernelEx(&cfg, chain_kernel<6>, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return QG_ERR_CUDA;
    }
    return QG_OK;
}

}  // namespace qg
