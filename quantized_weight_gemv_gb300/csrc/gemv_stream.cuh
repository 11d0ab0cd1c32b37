// Streaming quantized-weight GEMV: persistent CTAs whose warps each pull their own
// weight stages through a private shared-memory ring with the bulk-copy engine (TMA).
//
// Decode is bandwidth-bound: every weight byte is read once per token (oxinfer
// README, "Performance"; genie-ai-runtime, "The decode arc").  The kernel is shaped
// for that:
//  * CTA b owns the contiguous rows [b*n/G, (b+1)*n/G) of the matrix (G = grid).
//  * A stage is SB consecutive blocks of 32 weights in row-major order (SB = 256, or
//    512 for Q2 at one column: the same 5 KB): R = SB/nb whole rows when nb = k/32 <=
//    SB, else one SB-block part of a row.  Each stage is one contiguous span per plane
//    (codes, [hi,] scale, min), fetched by one cp.async.bulk per plane, completion
//    tracked by an mbarrier.
//  * Warp w of the CTA owns units w, w+W, w+2W, ... (a unit is a stage's rows, or
//    one whole row of nb/SB stages when nb > SB) and keeps D stages of its own in
//    flight in D private slots.  Its lane 0 issues the copies.  The first D are
//    issued before griddepcontrol.wait, so under programmatic dependent launch the
//    weight stream overlaps the tail of the preceding kernel.
//  * A warp moves a landed stage from shared memory into registers, refills the
//    slot with its next stage at once, and only then computes: lane l takes blocks
//    l + 32j (j < SB/32) of the stage, dots each with the int8 activation by dp4a over
//    nibbles unpacked from 32-bit words (genie-ai-runtime, "The decode arc": dp4a
//    int8 MMVQ "instead of dequant-to-fp"; its uint32 fast path for the dequant
//    loop), applies the fp32 block combine s_b * (scale * D + min * S_b), and
//    reduces the stage's rows together with a halving shuffle tree (warp-per-row
//    reduction: genie-ai-runtime, "The decode arc"; one 32-lane group per row in
//    needle.js "Inference backends", "TypeGPU").  No barrier couples the warps.
//  * A lane's block positions are the same in every stage, so for short rows its
//    activation words live in registers; for long rows they are read from shared
//    memory, stored as split halves so that the 128-bit reads are conflict-free.
//  * Epilogues: plain store; soft-cap + argmax; soft-cap + constrained selection (each
//    lane folds the rows it emits into a log-sum-exp; the allowed best is taken from
//    the CTA's written rows).  Both reductions end with the last CTA to arrive at a
//    counter finishing the result (the argmax from one packed atomic key, the selection
//    from every CTA's partial); no CTA waits on another.
//  * Every wait is bounded (mbarrier try_wait against %globaltimer); on expiry the
//    kernel ORs a code into the library's device error word and stops.
#pragma once

#include "qg_internal.h"

namespace qg {
namespace stream {

constexpr int SBW = 256;  // blocks per stage (the grouped and chain kernels; the base size here)
constexpr int JPL = 8;    // blocks per lane per stage of SBW blocks

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase of the given parity to complete; false after WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// Slot layout for SB blocks: codes[SB][CODE] | [hi[SB][8]] | scale[SB] | [min[SB]]
// (Q4/Q6: 16-byte code blocks; Q2: 8-byte code blocks and no min plane)
template <int BITS, int SB = SBW>
struct Slot {
    static constexpr int CODE = BITS == 2 ? 8 : 16;
    static constexpr int BPB = CODE + (BITS == 6 ? 8 : 0) + (BITS == 2 ? 2 : 4);
    static constexpr int BYTES = SB * BPB;
    static constexpr int HI = SB * 16;
    static constexpr int SC = SB * (CODE + (BITS == 6 ? 8 : 0));
    static constexpr int MN = SC + SB * 2;
};

// Blocks per stage of the single-matrix kernel.  A Q2 block is 10 bytes against 20 for
// Q4, so for one column and rows of at least 32 blocks a Q2 stage holds 512 blocks
// (the same 5 KB), which halves the per-stage work (ring wait, copy issue, the row
// reduction and the epilogue) per block.
template <int BITS, int BC, int NB>
__host__ __device__ constexpr int stage_blocks() {
    return BITS == 2 && BC == 1 && NB >= 32 ? 2 * SBW : SBW;
}

// Halving reduction over the lane bits [0, LOG2SEG): V values per lane, each to be
// summed over the 2^LOG2SEG lanes of a segment.  Step s pairs lanes across bit
// LOG2SEG-1-s; the lower lane keeps (and sums) the lower half of the values still
// held, the upper lane the upper half, so V values cost V-1 shuffles instead of
// V*LOG2SEG.  The bits left after log2(V) steps are summed with plain xor steps.
// On return v[0] of lane l is the segment total of value index
// (l & (2^LOG2SEG - 1)) >> (LOG2SEG - log2(V)).
template <int V, int LOG2SEG>
__device__ __forceinline__ void halving_reduce(float (&v)[V]) {
    static_assert((V & (V - 1)) == 0 && V >= 1, "V power of two");
    const int lane = threadIdx.x & 31;
    int cur = V;
    int off = 1 << (LOG2SEG - 1);
#pragma unroll
    for (int step = 0; (1 << step) < V; ++step) {
        const int half = cur >> 1;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < V / 2; ++i) {
            if (i < half) {
                const float send = upper ? v[i] : v[i + half];
                const float keep = upper ? v[i + half] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
        cur = half;
        off >>= 1;
    }
#pragma unroll
    for (; off > 0; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
}

// byte offset of the activation columns after `nslots` slots and their mbarriers
__host__ __device__ constexpr size_t xq_offset(int nslots, int slot_bytes) {
    return (((size_t)nslots * (size_t)(slot_bytes + 8)) + 15) & ~(size_t)15;
}

// One finished row: stored (EPI_STORE), or soft-capped, stored when logits are wanted and
// folded into the lane's running (value, index) best; under EPI_SELECT also into its
// online log-sum-exp (lm, ls; NaN skipped), the best only when no allowed list restricts it.
template <int EPI, int BC>
__device__ __forceinline__ void emit_row(const StreamParams& p, long long row, const float (&v)[BC], float& bv,
                                         int& bi, float& lm, float& ls, float inv_c) {
    if constexpr (EPI == EPI_STORE) {
        (void)lm;
        (void)ls;
#pragma unroll
        for (int c = 0; c < BC; ++c)
            if (c < p.batch) p.y[(size_t)c * p.n + row] = v[c];
    } else if constexpr (EPI == EPI_SELECT) {
        const float l = softcap_apply(v[0], p.softcap, inv_c);
        p.y[row] = l;
        if (l == l) lse_merge(lm, ls, l, 1.0f);
        if (!p.allowed && better(l, (int)row, bv, bi)) {
            bv = l;
            bi = (int)row;
        }
    } else {
        (void)lm;
        (void)ls;
        const float l = softcap_apply(v[0], p.softcap, inv_c);
        if (p.y) p.y[row] = l;
        if (better(l, (int)row, bv, bi)) {
            bv = l;
            bi = (int)row;
        }
    }
}

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v >> 1); }

// NB = k / 32 blocks per row: a power of two from 8 to 512, or 48 (k = 1536).  For 48 a
// stage holds whole rows (5 in 240 blocks, or 10 in 480 for the 512-block Q2 stage) and
// the rows, which straddle the lanes' block groups, are summed per lane and then
// through one halving tree (GEN below).
template <int BITS, int BC, int EPI, int NB, int W>
__global__ void __launch_bounds__(W * 32, (W == 8 && BC <= 2) ? 2 : 1) gemv_stream_kernel(StreamParams p) {
    constexpr int SB = stage_blocks<BITS, BC, NB>();  // blocks per stage (capacity)
    constexpr int JL = SB / 32;                        // blocks per lane per stage
    using SL = Slot<BITS, SB>;
    constexpr bool GEN = (NB & (NB - 1)) != 0;       // not a power of two
    constexpr int LOG2NB = GEN ? 0 : ilog2(NB);
    constexpr int R = NB >= SB ? 1 : SB / NB;         // rows per stage
    constexpr int PARTS = NB > SB ? NB / SB : 1;      // stages per row
    constexpr int JU = GEN ? (R * NB + 31) / 32 : JL;  // blocks per lane that can be in a stage
    // HALF (48-block rows, 10 per 512-block stage): rows 2i and 2i+1 go to the two half
    // warps, lane l taking blocks l % 16 + 16q (q = 0, 1, 2) of row 2i + l / 16 (j = 3i + q),
    // so each lane sums its own three blocks per row and a row is reduced over 16 lanes.
    // A half warp's loads of one j are then 16 consecutive blocks: their 2-byte scales
    // fill 8 banks, the other half's (96 bytes on) 8 others.
    // Otherwise lane l takes blocks l + 32j of the stage.
    constexpr bool HALF = GEN && R == 10;
    // distinct activation blocks per lane.  GEN (48 blocks per row): three, l % 16 + 16q
    // under HALF, else (l + 32j) mod 48, where 96 = 0 mod 48 leaves only j mod 3
    constexpr int NXB = GEN ? 3 : NB >= 32 ? (NB < SB ? NB / 32 : JL) : 1;
    // activation words in registers, except for four columns of rows of 64+ blocks, whose
    // 80 registers of words would leave room for only one 8-warp CTA per SM
    constexpr bool XREG = NB <= 128 && BC * NXB <= (BC == 4 ? 4 : 8);
    constexpr int NXR = XREG ? NXB : 1;
    // Q2 in the HALF mapping with the activation words in registers: a lane's three blocks
    // of a row meet its three activation blocks, so their scales multiply in the row sum
    constexpr bool SFOLD = BITS == 2 && HALF && XREG;
    static_assert(!GEN || NB == 48, "blocks per row: a power of two, or 48");

    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.stages;  // slots per warp

    // shared layout: slots[W][D] | full[W][D] | xq columns (16-byte aligned)
    unsigned char* slots = smem + (size_t)warp * D * SL::BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)W * D * SL::BYTES) + warp * D;
    unsigned char* xqbase = smem + xq_offset(W * D, SL::BYTES);
    const int xstride = xq_stride(NB);

    const long long r0 = (long long)blockIdx.x * p.n / gridDim.x;
    const long long r1 = (long long)(blockIdx.x + 1) * p.n / gridDim.x;
    const int nrows = (int)(r1 - r0);
    const int nunits = NB >= SB ? nrows : (nrows + R - 1) / R;       // unit: R rows, or one row
    const int my_units = nunits > warp ? (nunits - warp + W - 1) / W : 0;
    const int my_stages = my_units * PARTS;

    const uint64_t pol = policy_evict_first();
    // issue stage t of this warp (unit warp + W*(t/PARTS), part t%PARTS) into slot t%D
    auto issue = [&](int t, int slot) {
        const int u = warp + W * (t / PARTS);
        const int part = t % PARTS;
        const long long row = r0 + (long long)u * R;
        const int rows_u = R == 1 ? 1 : min(R, nrows - u * R);
        const uint32_t blocks = (uint32_t)(NB >= SB ? SB : rows_u * NB);
        const size_t blk0 = (size_t)row * NB + (size_t)part * SB;  // first block in the matrix
        unsigned char* st = slots + (size_t)slot * SL::BYTES;
        uint64_t* bar = &full[slot];
        mbar_arrive_expect_tx(bar, blocks * SL::BPB);
        bulk_g2s(st, p.lo + blk0 * SL::CODE, blocks * SL::CODE, bar, pol);
        if constexpr (BITS == 6) bulk_g2s(st + SL::HI, p.hi + blk0 * 8, blocks * 8, bar, pol);
        bulk_g2s(st + SL::SC, p.scale + blk0, blocks * 2, bar, pol);
        if constexpr (BITS != 2) bulk_g2s(st + SL::MN, p.min + blk0, blocks * 2, bar, pol);
    };

    if (lane == 0) {
        pdl_launch_dependents();
        for (int s = 0; s < D; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        for (int t = 0; t < D && t < my_stages; ++t) issue(t, t);
    }
    __syncwarp();

    // stage t (in slot `slot_`, phase parity `phase_`) -> registers, then the slot refilled
    // with stage t + D; false when the bounded wait ran out (warp-uniform)
    uint4 cw[JU];
    uint2 hw[JU];
    unsigned short dh[JU], mh[JU];
    auto fetch = [&](int t, int slot_, uint32_t phase_) -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[slot_], phase_))) return false;
        const unsigned char* st = slots + (size_t)slot_ * SL::BYTES;
#pragma unroll
        for (int j = 0; j < JU; ++j) {
            const int fb = HALF ? (2 * (j / 3) + (lane >> 4)) * NB + (lane & 15) + 16 * (j % 3) : lane + 32 * j;
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
        if (lane == 0 && t + D < my_stages) {
            fence_proxy_async();  // the slot's generic reads are done before the async refill
            issue(t + D, slot_);
        }
        return true;
    };
    // 16-warp CTAs (a small share per SM): the first stage goes to registers and its slot
    // is refilled before the wait below, one more stage per warp requested while the
    // preceding kernel finishes.
    const bool first_held = W == 16 && my_stages > 0 && fetch(0, 0, 0u);

    // ---- activation prologue (after the preceding kernel, which may have written x)
    pdl_wait();
    quantize_x_cols<W * 32>(p.x, p.k, p.batch, xqbase, xstride, threadIdx.x);
    __syncthreads();

    uint4 xl[BC][NXR], xh[BC][NXR];
    float xs[BC][NXR], xS[BC][NXR];
    int xT[BC][NXR];  // Q2: 64 x the zero-point term -2 S_b, the seed of the block dot
    if constexpr (XREG) {
#pragma unroll
        for (int j = 0; j < NXR; ++j) {
            const int blk = HALF  ? (lane & 15) + 16 * j
                            : GEN ? (lane + 32 * j) % NB
                            : NB >= 32 ? lane + 32 * j
                                       : (lane & (NB - 1));
#pragma unroll
            for (int c = 0; c < BC; ++c) {
                const XqView v = xq_view(xqbase + c * xstride, NB);
                const bool ok = c < p.batch;
                xl[c][j] = ok ? *reinterpret_cast<const uint4*>(v.lo + 16 * blk) : make_uint4(0, 0, 0, 0);
                xh[c][j] = ok ? *reinterpret_cast<const uint4*>(v.hi + 16 * blk) : make_uint4(0, 0, 0, 0);
                xs[c][j] = ok ? v.s[blk] : 0.0f;
                xS[c][j] = ok ? v.S[blk] : 0.0f;
                xT[c][j] = -128 * __float2int_rn(xS[c][j]);
            }
        }
    }

    float bv = __int_as_float(0x7fc00000);
    int bi = 0x7fffffff;
    float lm = -INFINITY, ls = 0.0f;  // selection: online log-sum-exp of the emitted logits
    const float inv_c = softcap_inv(p.softcap);
    float rowacc[BC];  // running sum of a row that spans several stages
#pragma unroll
    for (int c = 0; c < BC; ++c) rowacc[c] = 0.0f;

    // slot = t % D and its phase parity (t / D) & 1, kept as running counters
    int slot = 0;
    uint32_t phase = 0;
    for (int t = 0; t < my_stages; ++t, slot = slot + 1 == D ? 0 : slot + 1, phase ^= slot == 0) {
        if (!(t == 0 && first_held) && !fetch(t, slot, phase)) {
            atomicOr(p.err, ERR_WAIT_FULL);
            break;
        }
        const int u = warp + W * (t / PARTS);
        const int part = t % PARTS;
        const long long row0 = r0 + (long long)u * R;
        const int rows_u = R == 1 ? 1 : min(R, nrows - u * R);

        // block partials: part j of the lane belongs to row (lane + 32j) / NB of the stage.
        // In a stage of fewer than R rows the blocks past its last row are computed on
        // stale slot bytes; every reduction below keeps rows apart and only the stage's
        // rows are emitted, so they are never masked here.
        float pj[BC][JU];
#pragma unroll
        for (int j = 0; j < JU; ++j) {
#pragma unroll
            for (int c = 0; c < BC; ++c) {
                if constexpr (XREG && BITS == 2) {
                    // scale * (D - 2 S_b) straight from the seeded dot; the activation scale
                    // s_b is applied in the row sums under SFOLD, else here
                    const int xj = NB >= 32 ? (j % NXR) : 0;
                    const float t = half_bits_to_float(dh[j]) *
                                    (float)block_dot_q2(hw[j], xl[c][xj], xh[c][xj], xT[c][xj]);
                    pj[c][j] = SFOLD ? t : xs[c][xj] * t;
                } else if constexpr (XREG) {
                    const int xj = NB >= 32 ? (j % NXR) : 0;
                    pj[c][j] = combine<BITS>(qdot<BITS>(cw[j], hw[j], xl[c][xj], xh[c][xj]), dh[j], mh[j], xs[c][xj],
                                             xS[c][xj]);
                } else {
                    const int blk = HALF  ? (lane & 15) + 16 * (j % 3)
                                    : GEN ? (lane + 32 * j) % NB
                                          : (part * SB + lane + 32 * j) & (NB - 1);
                    const XqView v = xq_view(xqbase + c * xstride, NB);
                    const uint4 a = *reinterpret_cast<const uint4*>(v.lo + 16 * blk);
                    const uint4 b = *reinterpret_cast<const uint4*>(v.hi + 16 * blk);
                    pj[c][j] = combine<BITS>(qdot<BITS>(cw[j], hw[j], a, b), dh[j], mh[j], v.s[blk], v.S[blk]);
                }
            }
        }

        if constexpr (HALF) {
            // row 2i + l / 16 of lane l: its three blocks j = 3i .. 3i+2; the 5 row pairs
            // padded to 8 go through one halving tree over each half warp, after which
            // lane l holds row pair (l % 16) / 2 of its half
#pragma unroll
            for (int c = 0; c < BC; ++c) {
                float rs[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = i < 5 ? 3 * i : 0;  // JU = 15: j + 2 < JU for every row pair
                    if constexpr (SFOLD)  // block j + q meets activation block q of the lane
                        rs[i] = i < 5 ? fmaf(xs[c][2], pj[c][j + 2], fmaf(xs[c][1], pj[c][j + 1], xs[c][0] * pj[c][j]))
                                      : 0.0f;
                    else
                        rs[i] = i < 5 ? pj[c][j] + pj[c][j + 1] + pj[c][j + 2] : 0.0f;
                }
                halving_reduce<8, 4>(rs);
                pj[c][0] = rs[0];
            }
            const int i = (lane & 15) >> 1, r = 2 * i + (lane >> 4);
            if ((lane & 1) == 0 && i < 5 && r < rows_u) {
                float out[BC];
#pragma unroll
                for (int c = 0; c < BC; ++c) out[c] = pj[c][0];
                emit_row<EPI, BC>(p, row0 + r, out, bv, bi, lm, ls, inv_c);
            }
        } else if constexpr (GEN) {
            // rows straddle the lanes' block groups: block l + 32j of lane l lies in row
            // (l + 32j) / 48, and every three j cover 96 blocks, two rows - j = 3i is in
            // row 2i, j = 3i+1 in row 2i (lanes 0-15) or 2i+1 (lanes 16-31), j = 3i+2 in
            // row 2i+1.  Each lane sums its blocks per row; the R rows padded to RV go
            // through one halving tree, after which lane l holds row l / (32 / RV)
            constexpr int RV = R <= 8 ? 8 : 16;
            const bool lo = lane < 16;
#pragma unroll
            for (int c = 0; c < BC; ++c) {
                float rs[RV];
#pragma unroll
                for (int i = 0; i < RV / 2; ++i) {
                    const float a = 3 * i < JU ? pj[c][3 * i < JU ? 3 * i : 0] : 0.0f;
                    const float b = 3 * i + 1 < JU ? pj[c][3 * i + 1 < JU ? 3 * i + 1 : 0] : 0.0f;
                    const float e = 3 * i + 2 < JU ? pj[c][3 * i + 2 < JU ? 3 * i + 2 : 0] : 0.0f;
                    rs[2 * i] = a + (lo ? b : 0.0f);
                    rs[2 * i + 1] = (lo ? 0.0f : b) + e;
                }
                halving_reduce<RV, 5>(rs);
                pj[c][0] = rs[0];
            }
            constexpr int LPR = 32 / RV;  // lanes holding one row's total
            if ((lane & (LPR - 1)) == 0) {
                const int r = lane / LPR;
                if (r < rows_u) {
                    float out[BC];
#pragma unroll
                    for (int c = 0; c < BC; ++c) out[c] = pj[c][0];
                    emit_row<EPI, BC>(p, row0 + r, out, bv, bi, lm, ls, inv_c);
                }
            }
        } else if constexpr (NB >= 32) {
            // R rows per stage, JL/R consecutive j per row
            constexpr int JR = JL / R;
#pragma unroll
            for (int c = 0; c < BC; ++c) {
                float rs[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float s = 0.0f;
#pragma unroll
                    for (int q = 0; q < JR; ++q) s += pj[c][r * JR + q];
                    rs[r] = s;
                }
                if constexpr (PARTS > 1) {
                    rowacc[c] += rs[0];
                    if (part == PARTS - 1) {
                        float one[1] = {rowacc[c]};
                        halving_reduce<1, 5>(one);
                        pj[c][0] = one[0];
                        rowacc[c] = 0.0f;
                    }
                } else {
                    halving_reduce<R, 5>(rs);
                    pj[c][0] = rs[0];
                }
            }
            if (PARTS == 1 || part == PARTS - 1) {
                constexpr int LANES_PER_ROW = 32 / R;
                if ((lane & (LANES_PER_ROW - 1)) == 0) {
                    const int r = lane / LANES_PER_ROW;
                    if (r < rows_u) {
                        float out[BC];
#pragma unroll
                        for (int c = 0; c < BC; ++c) out[c] = pj[c][0];
                        emit_row<EPI, BC>(p, row0 + r, out, bv, bi, lm, ls, inv_c);
                    }
                }
            }
        } else {
            // NB < 32: value j of lane l is row j*(32/NB) + l/NB, summed over NB-lane segments
#pragma unroll
            for (int c = 0; c < BC; ++c) halving_reduce<JL, LOG2NB>(pj[c]);
            constexpr int KEEP = NB / JL;  // lanes holding the same value after the halving steps
            if ((lane & (KEEP - 1)) == 0) {
                const int v = (lane & (NB - 1)) / KEEP;
                const int r = v * (32 / NB) + lane / NB;
                if (r < rows_u) {
                    float out[BC];
#pragma unroll
                    for (int c = 0; c < BC; ++c) out[c] = pj[c][0];
                    emit_row<EPI, BC>(p, row0 + r, out, bv, bi, lm, ls, inv_c);
                }
            }
        }
    }

    if constexpr (EPI == EPI_ARGMAX) {
        __shared__ ArgmaxPartial sred[W];
        argmax_finish(bv, bi, p.ws, p.argmax, sred);
    } else if constexpr (EPI == EPI_SELECT) {
        // Constrained selection over this CTA's rows [r0, r1): each lane's online
        // log-sum-exp of the rows it emitted (NaN skipped) and, without a list, its best
        // (value, lowest id); with a list, the best among the allowed ids that fall in the
        // range, from one pass over the list after the barrier (the CTA's logits in y are
        // then visible to all its threads).  The last CTA to finish merges every CTA's
        // partial.
        __shared__ SelectPartial sred[W];
        __shared__ int slast;
        float m = lm, s = ls;
        float sv = bv;
        int si = bi;
        if (p.allowed) {
            __syncthreads();
            for (int j = threadIdx.x; j < p.n_allowed; j += blockDim.x) {
                const long long id = p.allowed[j];
                if (id < r0 || id >= r1) continue;
                const float l = p.y[id];
                if (better(l, (int)id, sv, si)) {
                    sv = l;
                    si = (int)id;
                }
            }
        }
        select_finish(m, s, sv, si, p.sws, p.token, p.logprob, sred, &slast);
    }
}

}  // namespace stream

// host launcher for one format (defined in gemv_stream_q4.cu / gemv_stream_q6.cu)
template <int BITS>
int launch_stream_bits(const StreamParams& p, int epi, const LaunchCtx& lc);

}  // namespace qg
