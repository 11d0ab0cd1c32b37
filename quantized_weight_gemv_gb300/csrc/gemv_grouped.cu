// Grouped GEMV: many independent quantized-weight GEMVs in two launches.
//
// needle.js "Inference backends", "Hybrid GPU execution": independent projections
// go through matvecBatch, their packed weights combined so that one dispatch covers
// the whole group; genie-ai-runtime "v1.2.0": a triple QKV GEMV sharing one q8_1
// activation.  Here the group is a list of up to QG_MAX_GROUP descriptors (weights,
// x, y, n, k), passed by value as the kernel parameter, so nothing is allocated:
//  1. grouped_quantize_kernel: every activation of the group, quantised per block
//     of 32 (one warp per block) into the caller's workspace;
//     (A group whose distinct activations are short may skip this launch: the GEMV
//     kernel then quantises them itself into shared memory, see SMX below.  So may a
//     group whose images the preceding launch produced: see the images-out tail.)
//  2. grouped_gemv_kernel (programmatic dependent launch on 1): persistent CTAs
//     split the concatenated work of all descriptors - units of 256 blocks (whole
//     rows), or single rows of k/8192 such units for k > 8192 - into contiguous,
//     equal shares of bulk-copy stages.  Each warp streams its units through a
//     private ring exactly as the single-matrix streaming kernel does; the ring
//     starts filling before griddepcontrol.wait, i.e. while kernel 1 still runs.
//     Optionally (the dependent chain) it also writes the activation images of some
//     of its outputs for the next launch: the CTA ranges inside those descriptors are
//     aligned to whole blocks of 32 rows, and each CTA quantises its own rows once
//     they are stored.
#include <cstring>

#include "gemv_stream.cuh"

namespace qg {
namespace grouped {

using stream::SBW;
using stream::JPL;

struct GDesc {
    const uint8_t* lo;
    const uint8_t* hi;
    const uint16_t* scale;
    const uint16_t* min;
    const float* x;
    float* y;
    int n;
    int log2nb;        // log2(k / 32), 5..9
    int units;         // work units of this descriptor
    int parts;         // stages per unit (1, or nb / 256)
    int unit_prefix;   // units of the descriptors before
    int stage_prefix;  // stages of the descriptors before
    int qb_prefix;     // activation blocks of the descriptors before
    int ws_off;        // byte offset of this descriptor's activation image in the workspace
                       // (SMX: in the kernel's shared-memory image area)
    int qalign;        // units per 32 rows when its output image is produced here, else 1
};

struct GInput {  // a distinct activation of an SMX group and its shared-memory image
    const float* x;
    int k;
    int off;
};

// An activation image that the kernel produces from one descriptor's output for the
// next launch (the chain's long-input phases).  The CTAs' unit ranges are aligned to
// whole blocks of 32 rows inside a producing descriptor, so each CTA quantises the
// blocks of its own rows once they are stored.
struct GOut {
    int desc;            // producing descriptor
    int nq;              // blocks of 32 outputs (its n / 32)
    unsigned char* img;  // the image (xq_view layout for nq blocks)
};

struct GParams {
    int count;
    int total_units;
    int total_stages;
    int total_qblocks;
    int stages_per_warp;
    unsigned int* err;
    unsigned char* ws;
    int nin;        // SMX: distinct activations, quantised by every CTA after griddepcontrol.wait
    int img_bytes;  // SMX: bytes of their shared-memory images
    int nout;  // images produced for the next launch
    GOut out[GROUPED_MAX_OUT];
    GDesc d[QG_MAX_GROUP];
    GInput in[QG_MAX_GROUP];
};

// activation image reads: the workspace through the read-only path, or shared memory
template <bool SMX, typename T>
__device__ __forceinline__ T ldx(const T* ptr) {
    if constexpr (SMX)
        return *ptr;
    else
        return __ldg(ptr);
}

// descriptor holding global index v of a prefix array (largest d with prefix <= v)
template <typename F>
__device__ __forceinline__ int find_desc(const GParams& p, int v, F prefix) {
    int lo = 0, hi = p.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix(p.d[mid]) <= v)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(256) grouped_quantize_kernel(const __grid_constant__ GParams p) {
    pdl_wait();
    if (threadIdx.x == 0) pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    for (int g = blockIdx.x * 8 + (threadIdx.x >> 5); g < p.total_qblocks; g += gridDim.x * 8) {
        const int di = find_desc(p, g, [](const GDesc& d) { return d.qb_prefix; });
        const GDesc& d = p.d[di];
        const int b = g - d.qb_prefix;
        const int nb = 1 << d.log2nb;
        float s;
        int S;
        const int q = quantize_lane(d.x[32 * b + lane], s, S);
        const XqView v = xq_view(p.ws + d.ws_off, nb);
        if (lane < 16)
            v.lo[16 * b + lane] = (int8_t)q;
        else
            v.hi[16 * b + lane - 16] = (int8_t)q;
        if (lane == 0) {
            v.s[b] = s;
            v.S[b] = (float)S;
        }
    }
}

// Walks one warp's units: w, w+8, ... of the CTA's unit range, part by part.
struct Cursor {
    int g;     // global unit
    int part;  // stage within the unit
    int d;     // descriptor of g
    __device__ __forceinline__ void advance(const GParams& p) {
        if (++part == p.d[d].parts) {
            part = 0;
            g += 8;
            while (d + 1 < p.count && g >= p.d[d + 1].unit_prefix) ++d;
        }
    }
};

// first global unit whose first stage is at or after global stage x; inside a
// descriptor whose output image is produced, rounded up to a whole block of 32 rows
// (monotone in x, so consecutive CTAs' ranges still tile the units)
__device__ __forceinline__ int unit_at_stage(const GParams& p, int x) {
    if (x >= p.total_stages) return p.total_units;
    const int di = find_desc(p, x, [](const GDesc& d) { return d.stage_prefix; });
    const GDesc& d = p.d[di];
    int local = (x - d.stage_prefix + d.parts - 1) / d.parts;
    if (d.qalign > 1) local = min((local + d.qalign - 1) / d.qalign * d.qalign, d.units);
    return d.unit_prefix + local;
}

template <int BITS, int L, bool SMX>
__device__ __forceinline__ void stage_compute(const GDesc& d, const unsigned char* xqws, int unit_local, int part,
                                              const uint4 (&cw)[JPL], const uint2 (&hw)[JPL],
                                              const unsigned short (&dh)[JPL], const unsigned short (&mh)[JPL],
                                              const uint4 (&xl)[2], const uint4 (&xh)[2], const float (&xs)[2],
                                              const float (&xS)[2], float& rowacc) {
    constexpr int NB = 1 << L;
    constexpr int R = NB >= SBW ? 1 : SBW / NB;
    constexpr int PARTS = NB > SBW ? NB / SBW : 1;
    constexpr bool XREG = NB <= 64;
    const int lane = threadIdx.x & 31;
    const long long row0 = (long long)unit_local * R;
    const int rows_u = R == 1 ? 1 : min(R, d.n - unit_local * R);
    const XqView v = xq_view(const_cast<unsigned char*>(xqws), NB);

    float pj[JPL];
#pragma unroll
    for (int j = 0; j < JPL; ++j) {
        const int rloc = (NB >= SBW) ? 0 : ((lane + 32 * j) >> L);

        const float dd = half_bits_to_float(dh[j]);
        const float mm = half_bits_to_float(mh[j]);
        float r;
        if constexpr (XREG) {
            const int xj = j % (NB / 32);
            r = block_combine(qdot<BITS>(cw[j], hw[j], xl[xj], xh[xj]), dd, mm, xs[xj], xS[xj]);
        } else {
            const int blk = (part * SBW + lane + 32 * j) & (NB - 1);
            const uint4 a = ldx<SMX>(reinterpret_cast<const uint4*>(v.lo + 16 * blk));
            const uint4 b = ldx<SMX>(reinterpret_cast<const uint4*>(v.hi + 16 * blk));
            r = block_combine(qdot<BITS>(cw[j], hw[j], a, b), dd, mm, ldx<SMX>(v.s + blk), ldx<SMX>(v.S + blk));
        }
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
        if (r < rows_u) d.y[row0 + r] = rs[0];
    }
}

// SMX: the group's activations are quantised by each CTA into shared memory (after
// the ring slots) instead of being read from the workspace kernel 1 filled.
template <int BITS, int MINB, bool SMX>
__global__ void __launch_bounds__(256, MINB) grouped_gemv_kernel(const __grid_constant__ GParams p) {
    using SL = stream::Slot<BITS>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.stages_per_warp;
    unsigned char* slots = smem + (size_t)warp * D * SL::BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)8 * D * SL::BYTES) + warp * D;

    // this CTA's units: those whose first stage lies in its equal share of all stages
    const long long T = p.total_stages;
    const int u_begin = unit_at_stage(p, (int)(T * blockIdx.x / gridDim.x));
    const int u_end = unit_at_stage(p, (int)(T * (blockIdx.x + 1) / gridDim.x));

    Cursor ic, cc;  // issue and consume cursors
    ic.g = u_begin + warp;
    ic.part = 0;
    ic.d = ic.g < p.total_units ? find_desc(p, ic.g, [](const GDesc& d) { return d.unit_prefix; }) : 0;
    cc = ic;

    const uint64_t pol = stream::policy_evict_first();
    auto issue = [&](int slot) {  // stage at cursor ic into the given slot
        const GDesc& d = p.d[ic.d];
        const int nb = 1 << d.log2nb;
        const int R = nb >= SBW ? 1 : SBW / nb;
        const int ul = ic.g - d.unit_prefix;
        const int rows_u = R == 1 ? 1 : min(R, d.n - ul * R);
        const uint32_t blocks = (uint32_t)(nb >= SBW ? SBW : rows_u * nb);
        const size_t blk0 = (size_t)ul * R * nb + (size_t)ic.part * SBW;
        unsigned char* st = slots + (size_t)slot * SL::BYTES;
        uint64_t* bar = &full[slot];
        stream::mbar_arrive_expect_tx(bar, blocks * SL::BPB);
        stream::bulk_g2s(st, d.lo + blk0 * 16, blocks * 16, bar, pol);
        if constexpr (BITS == 6) stream::bulk_g2s(st + SL::HI, d.hi + blk0 * 8, blocks * 8, bar, pol);
        stream::bulk_g2s(st + SL::SC, d.scale + blk0, blocks * 2, bar, pol);
        stream::bulk_g2s(st + SL::MN, d.min + blk0, blocks * 2, bar, pol);
    };

    int issued = 0;
    if (lane == 0) {
        pdl_launch_dependents();
        for (int s = 0; s < D; ++s) stream::mbar_init(&full[s], 1);
        stream::fence_mbar_init();
        while (issued < D && ic.g < u_end) {
            issue(issued);
            ++issued;
            ic.advance(p);
        }
    }
    __syncwarp();
    pdl_wait();  // the activation images and the outputs depend on the preceding kernel
    unsigned char* const xbase = SMX ? smem + stream::xq_offset(8 * D, SL::BYTES) : p.ws;
    if constexpr (SMX) {
        for (int i = 0; i < p.nin; ++i)
            quantize_x_cols<256>(p.in[i].x, p.in[i].k, 1, xbase + p.in[i].off, 0, threadIdx.x);
        __syncthreads();
    }

    uint4 xl[2], xh[2];
    float xs[2], xS[2];
    int xd = -1;  // descriptor whose activation words are in registers
    float rowacc = 0.0f;

    // slot = t % D and its phase parity (t / D) & 1 of stage t, as running counters
    int slot = 0;
    uint32_t phase = 0;
    for (; cc.g < u_end; slot = slot + 1 == D ? 0 : slot + 1, phase ^= slot == 0) {
        if (!__all_sync(0xffffffffu, stream::mbar_wait(&full[slot], phase))) {  // warp-uniform
            atomicOr(p.err, ERR_WAIT_FULL);
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
        if (lane == 0 && ic.g < u_end) {
            stream::fence_proxy_async();
            issue(slot);
            ic.advance(p);
        }

        const GDesc& d = p.d[cc.d];
        const unsigned char* xqws = xbase + d.ws_off;
        if (d.log2nb <= 6 && xd != cc.d) {  // activation words of a new descriptor
            const int nb = 1 << d.log2nb;
            const XqView v = xq_view(const_cast<unsigned char*>(xqws), nb);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int blk = min(lane + 32 * j, nb - 1);
                xl[j] = ldx<SMX>(reinterpret_cast<const uint4*>(v.lo + 16 * blk));
                xh[j] = ldx<SMX>(reinterpret_cast<const uint4*>(v.hi + 16 * blk));
                xs[j] = ldx<SMX>(v.s + blk);
                xS[j] = ldx<SMX>(v.S + blk);
            }
            xd = cc.d;
        }
        const int ul = cc.g - d.unit_prefix;
        switch (d.log2nb) {
            case 5:
                stage_compute<BITS, 5, SMX>(d, xqws, ul, cc.part, cw, hw, dh, mh, xl, xh, xs, xS, rowacc);
                break;
            case 6:
                stage_compute<BITS, 6, SMX>(d, xqws, ul, cc.part, cw, hw, dh, mh, xl, xh, xs, xS, rowacc);
                break;
            case 7:
                stage_compute<BITS, 7, SMX>(d, xqws, ul, cc.part, cw, hw, dh, mh, xl, xh, xs, xS, rowacc);
                break;
            case 8:
                stage_compute<BITS, 8, SMX>(d, xqws, ul, cc.part, cw, hw, dh, mh, xl, xh, xs, xS, rowacc);
                break;
            default:
                stage_compute<BITS, 9, SMX>(d, xqws, ul, cc.part, cw, hw, dh, mh, xl, xh, xs, xS, rowacc);
                break;
        }
        cc.advance(p);
    }

    if (p.nout > 0) {
        // Images for the next launch: this CTA's rows of a producing descriptor are whole
        // blocks of 32 (aligned ranges), visible to the whole CTA after the barrier; a
        // warp per block quantises them exactly as the activation quantisation kernel does.
        __syncthreads();
        for (int o = 0; o < p.nout; ++o) {
            const GOut& out = p.out[o];
            const GDesc& d = p.d[out.desc];
            const int R = d.log2nb >= 8 ? 1 : 256 >> d.log2nb;
            const int ua = max(u_begin, d.unit_prefix) - d.unit_prefix;
            const int ub = min(u_end, d.unit_prefix + d.units) - d.unit_prefix;
            if (ua >= ub) continue;
            const int qb = min(ub * R, d.n) >> 5;
            for (int q = ((ua * R) >> 5) + warp; q < qb; q += 8) {
                float s;
                int S;
                const int code = quantize_lane(__ldcg(d.y + 32 * q + lane), s, S);
                const XqView v = xq_view(out.img, out.nq);
                if (lane < 16)
                    v.lo[16 * q + lane] = (int8_t)code;
                else
                    v.hi[16 * q + lane - 16] = (int8_t)code;
                if (lane == 0) {
                    v.s[q] = s;
                    v.S[q] = (float)S;
                }
            }
        }
    }
}

// fused form: distinct activations of at most this many image bytes (k <= 6144 in total)
constexpr int SMX_MAX_IMAGE = 7680;

static int env_int(const char* name, int dflt) {
    const char* v = getenv(name);
    if (!v || !*v) return dflt;
    return atoi(v);
}

}  // namespace grouped

size_t grouped_workspace_bytes(const qg_gemv_desc* descs, int count) {
    size_t off = 0;
    for (int i = 0; i < count; ++i) off += (size_t)xq_stride(descs[i].k >> 5);
    return off;
}

// distinct activations (by x and k) of the active descriptors and their image bytes
static int distinct_image_bytes(const qg_gemv_desc* descs, int count) {
    int bytes = 0;
    for (int i = 0; i < count && bytes <= grouped::SMX_MAX_IMAGE; ++i) {
        if (descs[i].n == 0) continue;
        bool seen = false;
        for (int j = 0; j < i && !seen; ++j)
            seen = descs[j].n > 0 && descs[j].x == descs[i].x && descs[j].k == descs[i].k;
        if (!seen) bytes += xq_stride(descs[i].k >> 5);
    }
    return bytes;
}

bool grouped_fuses(const qg_gemv_desc* descs, int count) {
    return distinct_image_bytes(descs, count) <= grouped::SMX_MAX_IMAGE;
}

int launch_grouped(int bits, const qg_gemv_desc* descs, int count, unsigned char* ws, const LaunchCtx& lc,
                   bool fuse, const GroupedOut* outs, int nout, bool images_ready) {
    using namespace grouped;
    static_assert(sizeof(GParams) < 32000, "grouped parameters must fit the kernel parameter space");
    GParams p;
    memset(&p, 0, sizeof(p));
    long long units = 0, stages = 0, qblocks = 0, off = 0;
    int m = 0;
    int internal[QG_MAX_GROUP];  // caller's descriptor index -> p.d index (-1: empty)
    for (int i = 0; i < count; ++i) {
        const qg_gemv_desc& s = descs[i];
        internal[i] = s.n == 0 ? -1 : m;
        if (s.n == 0) continue;
        const int nb = s.k >> 5;
        int l = 0;
        while ((1 << l) < nb) ++l;
        GDesc& d = p.d[m++];
        d.lo = s.lo;
        d.hi = s.hi;
        d.scale = s.scale;
        d.min = s.min;
        d.x = s.x;
        d.y = s.y;
        d.n = s.n;
        d.log2nb = l;
        d.qalign = 1;
        const int R = nb >= 256 ? 1 : 256 / nb;
        d.parts = nb > 256 ? nb / 256 : 1;
        d.units = nb >= 256 ? s.n : (s.n + R - 1) / R;
        d.unit_prefix = (int)units;
        d.stage_prefix = (int)stages;
        d.qb_prefix = (int)qblocks;
        d.ws_off = (int)off;
        units += d.units;
        stages += (long long)d.units * d.parts;
        qblocks += nb;
        off += xq_stride(nb);
    }
    if (m == 0) return QG_OK;
    if (stages > 0x7fffffffLL || off > 0x7fffffffLL) return QG_ERR_UNSUPPORTED;
    p.count = m;
    p.total_units = (int)units;
    p.total_stages = (int)stages;
    p.total_qblocks = (int)qblocks;
    p.err = lc.err;
    p.ws = ws;
    if (nout < 0 || nout > GROUPED_MAX_OUT || (nout > 0 && !outs)) return QG_ERR_INVALID_ARG;
    for (int o = 0; o < nout; ++o) {
        const int di = outs[o].desc;
        if (di < 0 || di >= count || internal[di] < 0 || descs[di].n % 32 != 0) return QG_ERR_INVALID_ARG;
        GDesc& d = p.d[internal[di]];
        d.qalign = 32 / (d.log2nb >= 8 ? 1 : 256 >> d.log2nb);  // units per 32 rows
        p.out[p.nout++] = GOut{internal[di], descs[di].n / 32, outs[o].img};
    }

    // Fused form: when the group's distinct activations (by x and k) are short, every
    // CTA quantises them itself into shared memory after griddepcontrol.wait and the
    // quantisation launch is skipped - one dependent launch instead of two.
    bool smx = false;
    if (fuse && !images_ready) {
        int ni = 0, ioff = 0, woff[QG_MAX_GROUP];
        for (int i = 0; i < m && ioff <= SMX_MAX_IMAGE; ++i) {
            const int k = 32 << p.d[i].log2nb;
            int j = 0;
            while (j < ni && !(p.in[j].x == p.d[i].x && p.in[j].k == k)) ++j;
            if (j == ni) {
                p.in[ni].x = p.d[i].x;
                p.in[ni].k = k;
                p.in[ni].off = ioff;
                ioff += xq_stride(k >> 5);
                ++ni;
            }
            woff[i] = p.in[j].off;
        }
        if (ioff <= SMX_MAX_IMAGE) {
            smx = true;
            p.nin = ni;
            p.img_bytes = ioff;
            for (int i = 0; i < m; ++i) p.d[i].ws_off = woff[i];
        }
    }

    // 1. activations (unless the preceding launch produced them)
    if (!smx && !images_ready) {
        long long qgrid = (qblocks + 7) / 8;
        if (qgrid > lc.sm_count * 16) qgrid = lc.sm_count * 16;
        int rc = launch_kernel(grouped_quantize_kernel, dim3((unsigned)qgrid), dim3(256), 0, lc, p);
        if (rc != QG_OK) return rc;
    }

    // 2. the GEMVs, chained to 1 by programmatic dependent launch (fused form: the
    // caller's flags).  Default: two CTAs per SM (16 warps, at most 128 registers each)
    // and one ring slot per warp - measured on GB300 as the fastest shape: the slot is
    // refilled as soon as it has been copied to registers, so 16 x 5 KB stay in flight
    // per SM.  The diagnostic switches QG_GROUPED_CTAS_PER_SM (1 or 2: the kernel's
    // register bound), QG_GROUPED_GRID_PER_SM (1 or 2: the grid, by default the same
    // except for short groups, below) and QG_GROUPED_SLOTS (slots per warp) override it.
    int per_sm = env_int("QG_GROUPED_CTAS_PER_SM", 2);
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 2) per_sm = 2;
    const int slot = bits == 4 ? stream::Slot<4>::BYTES : stream::Slot<6>::BYTES;
    int D = env_int("QG_GROUPED_SLOTS", 1);
    if (D < 1) D = 1;
    if (D > 16) D = 16;
    const size_t cap = (size_t)lc.max_smem_optin - 1024;
    while (stream::xq_offset(8 * D, slot) + (size_t)p.img_bytes > cap && D > 1) --D;
    const size_t smem = stream::xq_offset(8 * D, slot) + (size_t)p.img_bytes;
    p.stages_per_warp = D;
    using K = void (*)(GParams);
    static const K kerns[2][2][2] = {
        {{grouped_gemv_kernel<4, 1, false>, grouped_gemv_kernel<4, 1, true>},
         {grouped_gemv_kernel<4, 2, false>, grouped_gemv_kernel<4, 2, true>}},
        {{grouped_gemv_kernel<6, 1, false>, grouped_gemv_kernel<6, 1, true>},
         {grouped_gemv_kernel<6, 2, false>, grouped_gemv_kernel<6, 2, true>}}};
    const K kern = kerns[bits == 4 ? 0 : 1][per_sm - 1][smx ? 1 : 0];
    if (int e = ensure_smem_attr((const void*)kern, smem, lc)) return e;
    // A short group (fewer stages than 8 per SM: the chain's q/k/v and o phases) takes one
    // CTA per SM: a second adds no stream there, and the next launch's CTAs find room
    // beside it while it runs (decode chain 798 -> 753 us per token on GB300).
    int grid_per_sm = env_int("QG_GROUPED_GRID_PER_SM", stages < 8LL * lc.sm_count ? 1 : per_sm);
    if (grid_per_sm < 1) grid_per_sm = 1;
    if (grid_per_sm > 2) grid_per_sm = 2;
    long long grid = (long long)lc.sm_count * grid_per_sm;
    if (grid > units) grid = units;
    LaunchCtx lc2 = lc;
    if (!smx && !images_ready) lc2.flags |= QG_FLAG_PDL;
    return launch_kernel(kern, dim3((unsigned)grid), dim3(256), smem, lc2, p);
}

}  // namespace qg
