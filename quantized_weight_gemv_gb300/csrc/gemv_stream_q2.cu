// Streaming GEMV instantiations for 2-bit weights.
#include "gemv_stream_launch.cuh"

namespace qg {
template <>
int launch_stream_bits<2>(const StreamParams& p, int epi, const LaunchCtx& lc) {
    return stream::launch_bits<2>(p, epi, lc);
}
}  // namespace qg
