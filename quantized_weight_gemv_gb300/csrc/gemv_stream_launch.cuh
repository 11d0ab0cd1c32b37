// Host-side choice of ring depth and grid for the streaming GEMV, per format.
#pragma once

#include <cstdlib>

#include "gemv_stream.cuh"

namespace qg {
namespace stream {

inline int env_int(const char* name, int dflt) {
    const char* v = getenv(name);
    if (!v || !*v) return dflt;
    return atoi(v);
}

template <int BITS, int BC, int EPI, int NB, int W>
int launch_w(StreamParams p, const LaunchCtx& lc, int D, int per_sm) {
    using SL = Slot<BITS, stage_blocks<BITS, BC, NB>()>;
    auto kern = gemv_stream_kernel<BITS, BC, EPI, NB, W>;
    const size_t fixed = (size_t)BC * xq_stride(NB);
    if (D < 1) D = 1;
    if (D > 8) D = 8;
    const size_t cap = (size_t)lc.max_smem_optin - 1024;  // room for static shared memory
    size_t smem = xq_offset(W * D, SL::BYTES) + fixed;
    while (smem > cap && D > 1) {
        --D;
        smem = xq_offset(W * D, SL::BYTES) + fixed;
    }
    if (smem > cap) return QG_ERR_UNSUPPORTED;
    if (int rc = ensure_smem_attr((const void*)kern, smem, lc)) return rc;
    p.stages = D;
    p.err = lc.err;
    if (per_sm < 1) per_sm = 1;
    int grid = lc.sm_count * per_sm;
    if (EPI == EPI_SELECT && grid > SELECT_MAX_CTAS) grid = SELECT_MAX_CTAS;
    if (grid > p.n) grid = p.n;
    if (grid < 1) grid = 1;
    return launch_kernel(kern, dim3(grid), dim3(W * 32), smem, lc, p);
}

template <int BITS, int BC, int EPI, int NB>
int launch_t(StreamParams p, const LaunchCtx& lc) {
    constexpr int SB = stage_blocks<BITS, BC, NB>();
    constexpr int R = NB >= SB ? 1 : SB / NB;
    constexpr int PARTS = NB > SB ? NB / SB : 1;
    // Default: 8 warps per CTA, two CTAs per SM (one from four columns), one ring slot
    // per warp: a slot is refilled as soon as it has been copied to registers, and the
    // stream of a large matrix keeps every warp busy (measured on GB300 as the fastest
    // shape for the vocabulary heads and the large projections).
    // A GEMV of up to four columns whose share per SM is one to four stages per warp of
    // one 16-warp CTA (for 16384 x 2048: 27 stages of 5 KB per SM) takes that CTA, with enough
    // slots that every stage of every warp is requested before the kernel waits for the
    // preceding work (one stage in registers, the rest in slots): the weight stream then
    // overlaps the preceding kernel's tail and the activation prologue.
    // Q6 at three or four columns keeps the 8-warp form: its 16-warp kernel exceeds the
    // 128 registers a thread has there and spills (16384 x 2048, four columns: 15.5 us
    // against 11.7 us measured on GB300).
    // A smaller GEMV (fewer than 16 stages per SM: 1024 x 1024, 2048 x 2048) takes one
    // 8-warp CTA per SM: a second CTA per SM adds no stream there, only launch and
    // completion work (1024 x 1024 2.06 -> 1.77 us, 2048 x 2048 2.38 -> 2.09 us back to back
    // on GB300).
    // Q2 streams take two slots per warp: its 10-byte blocks are few instructions each, so a
    // warp finishes a stage in about one DRAM round trip and a single refilled slot leaves
    // it waiting (262144 x 1536 with soft-cap and argmax: 25.5 -> 24.4 us on GB300).
    // QG_STREAM_WARPS (8 or 16), QG_STREAM_SLOTS and QG_STREAM_CTAS_PER_SM override it.
    constexpr bool W16 = BC <= 4 && EPI == EPI_STORE && !(BITS == 6 && BC == 4);
    int W = 8, D = 1, per_sm = BC <= 2 ? 2 : 1;
    const long long rows = ((long long)p.n + lc.sm_count - 1) / lc.sm_count;
    const long long stages = (NB >= SB ? rows : (rows + R - 1) / R) * PARTS;  // per SM
    if (stages < 16) per_sm = 1;
    if (BITS == 2 && stages >= 16) D = 2;
    if constexpr (W16) {
        const long long per_warp = (stages + 15) / 16;
        if (stages >= 16 && per_warp <= 4) {
            W = 16;
            per_sm = 1;
            D = per_warp > 1 ? (int)per_warp - 1 : 1;
        }
        W = env_int("QG_STREAM_WARPS", W) == 16 ? 16 : 8;
    }
    D = env_int("QG_STREAM_SLOTS", D);
    per_sm = env_int("QG_STREAM_CTAS_PER_SM", per_sm);
    if constexpr (W16) {
        if (W == 16) return launch_w<BITS, BC, EPI, NB, 16>(p, lc, D, per_sm);
    }
    return launch_w<BITS, BC, EPI, NB, 8>(p, lc, D, per_sm);
}

template <int BITS, int BC, int EPI>
int launch_l(const StreamParams& p, const LaunchCtx& lc) {
    switch (p.k >> 5) {
        case 8: return launch_t<BITS, BC, EPI, 8>(p, lc);
        case 16: return launch_t<BITS, BC, EPI, 16>(p, lc);
        case 32: return launch_t<BITS, BC, EPI, 32>(p, lc);
        case 48: return launch_t<BITS, BC, EPI, 48>(p, lc);
        case 64: return launch_t<BITS, BC, EPI, 64>(p, lc);
        case 128: return launch_t<BITS, BC, EPI, 128>(p, lc);
        case 256: return launch_t<BITS, BC, EPI, 256>(p, lc);
        case 512: return launch_t<BITS, BC, EPI, 512>(p, lc);
    }
    return QG_ERR_UNSUPPORTED;
}

template <int BITS>
int launch_bits(const StreamParams& p, int epi, const LaunchCtx& lc) {
    if (epi == EPI_ARGMAX) return launch_l<BITS, 1, EPI_ARGMAX>(p, lc);
    if (epi == EPI_SELECT) return launch_l<BITS, 1, EPI_SELECT>(p, lc);
    switch (p.batch) {
        case 1: return launch_l<BITS, 1, EPI_STORE>(p, lc);
        case 2: return launch_l<BITS, 2, EPI_STORE>(p, lc);
        default: return launch_l<BITS, 4, EPI_STORE>(p, lc);
    }
}

}  // namespace stream
}  // namespace qg
