// Entry of the streaming GEMV: shape support and dispatch by format.
#include "gemv_stream.cuh"

namespace qg {

bool stream_supported(int bits, int n, int k, int batch, int epi) {
    if (bits != 2 && bits != 4 && bits != 6) return false;
    // nb = k/32 a power of two in [8, 512], or 48 (k = 1536, the hidden width of the
    // int2 LM head of the Gemma WebGPU Engine, "Roadmap")
    if (k != 1536 && (k < 256 || k > 16384 || (k & (k - 1)) != 0)) return false;
    if (batch < 1 || batch > 4) return false;
    if ((epi == EPI_ARGMAX || epi == EPI_SELECT) && batch != 1) return false;
    (void)n;
    return true;
}

int launch_stream(const StreamParams& p0, int bits, int epi, const LaunchCtx& lc) {
    if (!stream_supported(bits, p0.n, p0.k, p0.batch, epi)) return QG_ERR_UNSUPPORTED;
    StreamParams p = p0;
    if (splitk_wanted(p.n, p.k, p.batch, epi)) {
        const int rc = launch_splitk(p, bits, lc);
        if (rc != QG_ERR_UNSUPPORTED) return rc;
    }
    if (bits == 2) return launch_stream_bits<2>(p, epi, lc);
    return bits == 4 ? launch_stream_bits<4>(p, epi, lc) : launch_stream_bits<6>(p, epi, lc);
}

}  // namespace qg
