// Dependent GEMV chain: phases of quantized-weight GEMVs, each phase reading what
// earlier phases wrote - one grouped launch per phase (default), or one persistent
// cooperative launch for all of them.
//
// A decode token is a chain: every projection quantises and reads a vector that an
// earlier projection has just written (Gemma WebGPU Engine, "Roadmap": the layer's
// ordered dispatches, the attention output bound straight into the O projection and
// its output into the MLP; genie-ai-runtime, "The decode arc": activation quantised
// per matmul, and "v1.2.0": ~448 dependent kernel launches per token).
// Per-phase mode: each phase is one grouped launch chained to the one before by
// programmatic dependent launch; short inputs are quantised by every CTA, and long
// inputs that are whole outputs of the phase before arrive as activation images that
// the phase before wrote (its CTA ranges aligned to 32-row blocks), so no phase needs
// a separate quantisation launch in the decode chain.
// Persistent mode: one CTA per SM walks all phases:
//  * A phase is a list of GEMV descriptors whose inputs all exist before it.  Its work
//    is cut as in the grouped GEMV: units of 256 blocks of 32 (whole rows), or single
//    rows of k/8192 such units; CTA b takes the units whose first bulk-copy tile lies
//    in its equal share of the phase's tiles.
//  * One producer warp streams the CTA's weight tiles, phase after phase, into a
//    CTA-wide ring of cp.async.bulk slots (full / empty mbarrier pair per slot).
//    Weights do not depend on the chain, so the producer never waits for a phase
//    boundary: while the CTA waits for the others at the end of a phase, the ring
//    fills with the next phase's tiles, up to ~200 KB ahead.
//  * Fifteen consumer warps take the phase's units round-robin, read each tile's slot
//    into registers, release it, and compute as the streaming kernels do.  A consumer
//    waits for a tile's slot only once the producer has published the tile as issued,
//    which keeps every parity wait within one lap of the ring.
//  * Between phases (consumers only, named barrier 1): a grid-wide barrier on an
//    arrival counter in the caller's workspace (fence + atomic add, acquire loads,
//    bounded by %globaltimer, with an abort word that stops every CTA once one gives
//    up), then the consumers quantise the next phase's distinct inputs into shared
//    memory, reading them through L2 (ld.global.cg): other SMs wrote them during this
//    launch.
//  * The last CTA to finish re-arms the counters, so the workspace needs no memset
//    between calls.
#include <cstring>

#include "gemv_stream.cuh"

namespace qg {
namespace chain {

using stream::JPL;
using stream::SBW;
constexpr int NC = 15;             // consumer warps
constexpr int NTC = NC * 32;       // consumer threads
constexpr int NT = NTC + 32;       // + the producer warp

struct CDesc {
    const uint8_t* lo;
    const uint8_t* hi;
    const uint16_t* scale;
    const uint16_t* min;
    float* y;
    int n;
    int log2nb;       // log2(k / 32), 5..9; a unit has 2^(log2nb-8) tiles when log2nb > 8
    int unit_prefix;  // units of the phase's earlier descriptors
    int tile_prefix;  // tiles of the phase's earlier descriptors
    int img;          // byte offset of its input's activation image in shared memory
};

__host__ __device__ __forceinline__ int parts_of(int log2nb) { return log2nb > 8 ? 1 << (log2nb - 8) : 1; }

struct CPhase {
    int d0, d1;  // descriptors [d0, d1)
    int units, tiles;
    int in0, in1;  // distinct inputs [in0, in1)
};

struct CInput {
    const float* x;
    int k;
    int img;  // byte offset of its image in shared memory
};

struct CParams {
    int nphase;
    int log2slots;  // log2 of the CTA's ring slots
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
    const int parts = parts_of(d.log2nb);
    return d.unit_prefix + (int)((x - d.tile_prefix + parts - 1) / parts);
}

__device__ __forceinline__ int tile_index(const CDesc& d, int u, int part) {
    return d.tile_prefix + (u - d.unit_prefix) * parts_of(d.log2nb) + part;
}

// This CTA's units [ub, ue) of phase f, the phase's index of the first of their tiles
// and their number.  Called twice per phase, so kept out of line.
struct Range {
    int ub, ue, t0, tiles;
};

__device__ __noinline__ Range cta_range(const CParams& p, int f) {
    const CPhase& ph = p.ph[f];
    const long long T = ph.tiles;
    Range r;
    r.ub = unit_at_tile(p, ph, T * blockIdx.x / gridDim.x);
    r.ue = unit_at_tile(p, ph, T * (blockIdx.x + 1) / gridDim.x);
    auto first_tile = [&](int u) {
        if (u >= ph.units) return ph.tiles;
        const int di = find_in_phase(p, ph, u, [](const CDesc& d) { return d.unit_prefix; });
        return tile_index(p.d[di], u, 0);
    };
    r.t0 = first_tile(r.ub);
    r.tiles = first_tile(r.ue) - r.t0;
    return r;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(stream::smem_u32(bar)) : "memory");
}

// named barrier of the consumer warps (the producer warp never joins it)
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"r"(NTC) : "memory"); }

// Producer: wait until the slot's previous tile has been read.  False when the CTA
// is stopping (abort flag) or after WAIT_LIMIT_NS.
__device__ bool wait_empty(uint64_t* bar, uint32_t parity, const volatile int* abort_flag, unsigned int* err) {
    if (stream::mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (stream::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(err, ERR_WAIT_EMPTY);
            return false;
        }
    }
}

// Consumer: wait until the producer has issued at least n + 1 tiles (bounded; false when
// the CTA is stopping or after WAIT_LIMIT_NS).  A tile is waited for on its slot's full
// barrier only once issued: the producer issues tile n after tile n - NS was read, so the
// barrier has then completed tile n - NS's phase and a parity wait cannot take that
// earlier phase for tile n's.  Without this a warp whose next tile lies two ring laps
// ahead of the oldest pending one (15 warps, two tiles a unit, 16 slots) would pass on
// the parity of the phase two laps back.
__device__ bool wait_issued(const volatile int* issued, int n, const volatile int* abort_flag) {
    if (*issued > n) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (*issued > n) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
}

template <int BITS>
__device__ __forceinline__ void issue_tile(const CDesc& d, int ul, int part, unsigned char* slot, uint64_t* bar,
                                           uint64_t pol) {
    using SL = stream::Slot<BITS>;
    const int l = d.log2nb;
    const int lr = l >= 8 ? 0 : 8 - l;  // log2 of the rows per unit (256 blocks per tile)
    const int rows_u = min(1 << lr, d.n - (ul << lr));
    const uint32_t blocks = l >= 8 ? (uint32_t)SBW : (uint32_t)rows_u << l;
    const size_t blk0 = ((size_t)ul << (lr + l)) + (size_t)part * SBW;
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
// and every earlier boundary).  False when the wait ran out (ERR_WAIT_GRID, and the abort
// word set for the others) or the abort word is set (ERR_ABORTED): the abort word is read
// before every look at the count, so once it is set no CTA passes another boundary.
__device__ bool grid_barrier(const CParams& p, unsigned target) {
    // release: the CTA's outputs (ordered before by the consumers' barrier) before the arrival
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.ctl) : "memory");
    const unsigned long long t0 = globaltimer_ns();
    for (int spin = 0;; ++spin) {
        if (ld_acquire_gpu(p.ctl + 1) != 0u) {
            atomicOr(p.err, ERR_ABORTED);
            return false;
        }
        if (ld_acquire_gpu(p.ctl) >= target) return true;
        if ((spin & 15) == 15 && globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(p.err, ERR_WAIT_GRID);
            atomicExch(p.ctl + 1, 1u);
            return false;
        }
    }
}

// byte offsets of the shared-memory regions: ring | full[NS] | empty[NS] | image
__host__ __device__ constexpr size_t chain_full_off(int ns, int slot_bytes) { return (size_t)ns * slot_bytes; }
__host__ __device__ constexpr size_t chain_img_off(int ns, int slot_bytes) {
    return ((size_t)ns * (slot_bytes + 16) + 15) & ~(size_t)15;
}

template <int BITS>
__global__ void __launch_bounds__(NT, 1) chain_kernel(const __grid_constant__ CParams p) {
    using SL = stream::Slot<BITS>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ volatile int s_abort;
    __shared__ volatile int s_issued;  // tiles the producer has issued
    __shared__ Range s_range[QG_MAX_GROUP];  // this CTA's share of every phase
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NS = 1 << p.log2slots;
    const int LS = p.log2slots;
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + chain_full_off(NS, SL::BYTES));
    uint64_t* empty = full + NS;
    unsigned char* img = smem + chain_img_off(NS, SL::BYTES);

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_issued = 0;
        for (int i = 0; i < NS; ++i) {
            stream::mbar_init(&full[i], 1);
            stream::mbar_init(&empty[i], 1);
        }
        stream::fence_mbar_init();
    }
    // the ranges need dependent reads of the parameter block: all phases at once, here
    for (int f = threadIdx.x; f < p.nphase; f += NT) s_range[f] = cta_range(p, f);
    __syncthreads();

    if (warp == NC) {
        // ---------------- producer: every tile of the CTA, phase after phase.  The warp
        // walks the tile sequence together; each batch of up to 8 tiles is issued by
        // lanes 0-7 at once, lane i taking the batch's i-th tile.
        const uint64_t pol = stream::policy_evict_first();
        int f = 0, u = 0, ue = 0, di = 0, part = 0;  // walk cursor (the same in every lane)
        auto enter = [&](int from) {                  // first phase >= from with a tile here
            for (f = from; f < p.nphase; ++f) {
                const Range r = s_range[f];
                if (r.ub < r.ue) {
                    u = r.ub;
                    ue = r.ue;
                    di = find_in_phase(p, p.ph[f], u, [](const CDesc& d) { return d.unit_prefix; });
                    part = 0;
                    return;
                }
            }
        };
        enter(0);
        int n = 0;  // tiles issued
        bool stop = false;
        while (!stop && f < p.nphase) {
            int my_di = 0, my_ul = 0, my_part = 0, cnt = 0;
            for (; cnt < 8 && f < p.nphase; ++cnt) {
                if (lane == cnt) {
                    my_di = di;
                    my_ul = u - p.d[di].unit_prefix;
                    my_part = part;
                }
                if (++part == parts_of(p.d[di].log2nb)) {
                    part = 0;
                    if (++u == ue) {
                        enter(f + 1);
                    } else {
                        while (di + 1 < p.ph[f].d1 && u >= p.d[di + 1].unit_prefix) ++di;
                    }
                }
            }
            const int m = n + lane;
            const int slot = m & (NS - 1);
            bool ok = true;
            // The first pass over the ring finds every slot free (parity 1 of a fresh
            // barrier).  The consumer's arrive on `empty` releases its reads of the slot;
            // this wait acquires them before the copy overwrites it.
            if (lane < cnt) ok = wait_empty(&empty[slot], (uint32_t)(((m >> LS) & 1) ^ 1), &s_abort, p.err);
            stop = __any_sync(0xffffffffu, !ok);
            if (!stop && lane < cnt)
                issue_tile<BITS>(p.d[my_di], my_ul, my_part, ring + (size_t)slot * SL::BYTES, &full[slot], pol);
            if (!stop) n += cnt;
            __syncwarp();
            if (lane == 0 && !stop) {  // publish the batch to the consumers
                __threadfence_block();
                s_issued = n;
            }
        }
        // copies in flight land before the CTA exits (the last NS issued)
        if (lane == 0) {
            for (int m = n > NS ? n - NS : 0; m < n; ++m) {
                if (!stream::mbar_wait(&full[m & (NS - 1)], (uint32_t)((m >> LS) & 1))) {
                    atomicOr(p.err, ERR_WAIT_DRAIN);
                    break;
                }
            }
        }
    } else {
        // ---------------- consumers
        int base = 0;     // tiles of this CTA in earlier phases
        int issued = 0;   // tiles this lane has seen published as issued
        for (int f = 0; f < p.nphase; ++f) {
            // Phase boundary.  The consumers take each consumer_sync the same number of
            // times: s_abort changes only between the first two (thread 0) or after the
            // third (a warp whose tile never landed) and is read between the second and
            // the third.
            const CPhase& ph = p.ph[f];
            consumer_sync();
            if (threadIdx.x == 0) {
                if (s_abort)
                    atomicExch(p.ctl + 1, 1u);
                else if (f > 0 && !grid_barrier(p, gridDim.x * (unsigned)f))
                    s_abort = 1;
            }
            consumer_sync();
            if (s_abort) break;
            for (int i = ph.in0; i < ph.in1; ++i)
                quantize_x_cols<NTC, true>(p.in[i].x, p.in[i].k, 1, img + p.in[i].img, 0, threadIdx.x);
            consumer_sync();

            const Range r = s_range[f];
            float rowacc = 0.0f;
            bool bad = false;
            int di = ph.d0;
            for (int u = r.ub + warp; u < r.ue && !bad; u += NC) {
                while (di + 1 < ph.d1 && u >= p.d[di + 1].unit_prefix) ++di;
                const CDesc& d = p.d[di];
                const int ul = u - d.unit_prefix;
                const int parts = parts_of(d.log2nb);
                for (int part = 0; part < parts; ++part) {
                    const int n = base + tile_index(d, u, part) - r.t0;
                    const int slot = n & (NS - 1);
                    // all lanes poll; the decision is taken together so that the warp stays converged.
                    // The published count is re-read only once this tile lies beyond the last
                    // one seen (the producer normally runs ahead).
                    bool ready = true;
                    if (n >= issued) {
                        ready = wait_issued(&s_issued, n, &s_abort);
                        issued = s_issued;
                        __threadfence_block();
                    }
                    if (!__all_sync(0xffffffffu, ready && stream::mbar_wait(&full[slot], (uint32_t)((n >> LS) & 1)))) {
                        if (lane == 0) atomicOr(p.err, ERR_WAIT_FULL);
                        s_abort = 1;
                        bad = true;
                        break;
                    }
                    const unsigned char* st = ring + (size_t)slot * SL::BYTES;
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
                    if (lane == 0) mbar_arrive(&empty[slot]);  // the slot may be refilled

                    const unsigned char* xim = img + d.img;
                    switch (d.log2nb) {
                        case 5:
                            tile_compute<BITS, 5>(d, xim, ul, part, cw, hw, dh, mh, rowacc);
                            break;
                        case 6:
                            tile_compute<BITS, 6>(d, xim, ul, part, cw, hw, dh, mh, rowacc);
                            break;
                        case 7:
                            tile_compute<BITS, 7>(d, xim, ul, part, cw, hw, dh, mh, rowacc);
                            break;
                        case 8:
                            tile_compute<BITS, 8>(d, xim, ul, part, cw, hw, dh, mh, rowacc);
                            break;
                        default:
                            tile_compute<BITS, 9>(d, xim, ul, part, cw, hw, dh, mh, rowacc);
                            break;
                    }
                }
            }
            base += r.tiles;
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

// Workspace of the per-phase mode after the control words: three regions of A bytes,
// the images of a phase that quantises its own inputs and two (by phase parity) for
// images that a phase produces for the next one.
static size_t chain_image_region(const qg_gemv_desc* descs, const int* phase_sizes, int nphase) {
    size_t A = 0;
    int off = 0;
    for (int f = 0; f < nphase; ++f) {
        const size_t b = grouped_workspace_bytes(descs + off, phase_sizes[f]);
        if (b > A) A = b;
        off += phase_sizes[f];
    }
    return (A + 15) & ~(size_t)15;
}

size_t chain_workspace_bytes(const qg_gemv_desc* descs, int count, const int* phase_sizes, int nphase) {
    (void)count;
    return (size_t)QG_CHAIN_CTL_BYTES + 3 * chain_image_region(descs, phase_sizes, nphase);
}

// Whether the images of phase C (nc descriptors) can come from phase P: C takes the
// two-launch form (its inputs are long), and every active descriptor of C reads the
// whole output of an active descriptor of P (x == y, k == n, n a multiple of 32).  On
// success outs[0..*nout) name the producers with C's image offsets (in C's workspace
// layout, based at img).
static bool plan_produced(const qg_gemv_desc* P, int np, const qg_gemv_desc* C, int nc, unsigned char* img,
                          GroupedOut* outs, int* nout) {
    *nout = 0;
    if (grouped_fuses(C, nc)) return false;
    size_t off = 0;
    for (int j = 0; j < nc; ++j) {
        if (C[j].n == 0) continue;
        int i = 0;
        while (i < np && !(P[i].n > 0 && P[i].n % 32 == 0 && P[i].y == C[j].x && P[i].n == C[j].k)) ++i;
        if (i == np || *nout == GROUPED_MAX_OUT) return false;
        outs[*nout] = GroupedOut{i, img + off};
        ++*nout;
        off += (size_t)xq_stride(C[j].k >> 5);
    }
    return *nout > 0;
}

int launch_chain(int bits, const qg_gemv_desc* descs, int count, const int* phase_sizes, int nphase,
                 unsigned char* ws, const LaunchCtx& lc) {
    using namespace chain;
    (void)count;
    if (!(lc.flags & QG_FLAG_CHAIN_PERSISTENT)) {
        // One grouped launch (pair) per phase.  A phase with long inputs that are whole
        // outputs of the phase before takes its images from that phase, which quantises
        // its outputs block by block as they complete: one launch instead of two.
        const size_t A = chain_image_region(descs, phase_sizes, nphase);
        unsigned char* own = ws + QG_CHAIN_CTL_BYTES;
        unsigned char* produced[2] = {own + A, own + 2 * A};
        int off = 0;
        bool launched = false, ready = false;
        for (int f = 0; f < nphase; ++f) {
            LaunchCtx l2 = lc;
            if (launched) l2.flags |= QG_FLAG_PDL;
            bool any = false;
            for (int i = off; i < off + phase_sizes[f]; ++i) any = any || descs[i].n > 0;
            GroupedOut outs[GROUPED_MAX_OUT];
            int nout = 0;
            const bool next_ready =
                any && f + 1 < nphase &&
                plan_produced(descs + off, phase_sizes[f], descs + off + phase_sizes[f], phase_sizes[f + 1],
                              produced[(f + 1) & 1], outs, &nout);
            if (any) {
                const int rc = launch_grouped(bits, descs + off, phase_sizes[f], ready ? produced[f & 1] : own, l2,
                                              true, outs, next_ready ? nout : 0, ready);
                if (rc != QG_OK) return rc;
                launched = true;
            }
            ready = next_ready;
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
            const int parts = parts_of(l);
            const long long du = nb >= 256 ? s.n : (s.n + R - 1) / R;
            d.unit_prefix = (int)units;
            d.tile_prefix = (int)tiles;
            units += du;
            tiles += du * parts;
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

    // the ring takes what the activation images leave of the opt-in shared memory
    const int slot = bits == 4 ? stream::Slot<4>::BYTES : stream::Slot<6>::BYTES;
    const size_t cap = (size_t)lc.max_smem_optin - 1024 - sizeof(Range) * QG_MAX_GROUP - 128;
    int ls = 6;  // a power of two number of slots, at most 64
    while (ls > 1 && chain_img_off(1 << ls, slot) + (size_t)img_max > cap) --ls;
    const size_t smem = chain_img_off(1 << ls, slot) + (size_t)img_max;
    if (smem > cap) return QG_ERR_UNSUPPORTED;
    p.log2slots = ls;
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
