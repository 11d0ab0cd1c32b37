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

template <int BITS, int BC, int EPI, int NB>
int launch_t(StreamParams p, const LaunchCtx& lc) {
    using SL = Slot<BITS, stage_blocks<BITS, BC, NB>()>;
    auto kern = gemv_stream_kernel<BITS, BC, EPI, NB>;
    constexpr int W = 8;  // warps per CTA
    const size_t fixed = (size_t)BC * xq_stride(NB);
    // Default: one ring slot per warp and two CTAs per SM (measured on GB300 as the
    // fastest shape: a slot is refilled as soon as it has been copied to registers).
    // QG_STREAM_SLOTS (slots per warp) and QG_STREAM_CTAS_PER_SM override it.
    int D = env_int("QG_STREAM_SLOTS", 1);
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
    int per_sm = env_int("QG_STREAM_CTAS_PER_SM", BC <= 2 ? 2 : 1);
    if (per_sm < 1) per_sm = 1;
    int grid = lc.sm_count * per_sm;
    if (EPI == EPI_ARGMAX && grid > VOCAB_MAX_CTAS) grid = VOCAB_MAX_CTAS;
    if (EPI == EPI_SELECT && grid > SELECT_MAX_CTAS) grid = SELECT_MAX_CTAS;
    if (grid > p.n) grid = p.n;
    if (grid < 1) grid = 1;
    return launch_kernel(kern, dim3(grid), dim3(W * 32), smem, lc, p);
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
