// Streaming quantized-weight GEMV: a persistent CTA per SM that pulls its weight
// rows through a shared-memory ring with the bulk-copy engine (TMA).
//
// Decode is bandwidth-bound: every weight byte is read once per token (oxinfer
// README, "Performance"; genie-ai-runtime, "The decode arc").  The kernel is shaped
// for that:
//  * CTA b owns the contiguous rows [b*n/G, (b+1)*n/G) of the matrix (G = grid).
//  * A stage is 512 consecutive blocks of 32 weights in row-major order, i.e. whole
//    rows (512/nb of them when nb = k/32 <= 512): one contiguous span in each
//    plane (codes, [hi,] scale, min), fetched by one cp.async.bulk per plane into
//    a ring of `stages` slots, completion tracked by mbarriers.
//  * Warp 8 is the producer: one lane issues the copies, keeping the ring full.
//    It starts before griddepcontrol.wait, so under programmatic dependent launch
//    the weight stream overlaps the tail of the preceding kernel.
//  * Warps 0..7 consume: thread t owns flattened blocks t and t+256 of every
//    stage.  Because 512/nb rows fit a stage exactly, the block-in-row of a thread
//    is the same in every stage, so its int8 activation words stay in registers
//    for the whole kernel.  The dot is dp4a over nibbles unpacked from 32-bit
//    words; the per-block fp32 combine follows; rows are reduced with shuffles
//    (nb < 32) or shuffles then a 16-entry shared table (nb >= 32).
//  * Every wait is bounded (mbarrier try_wait against %globaltimer); on expiry the
//    kernel records an error code in the library's device error word and stops instead of hanging.
#include "qg_internal.h"

namespace qg {

constexpr int SB = 512;         // blocks per stage
constexpr int NCONS = 256;      // consumer threads
constexpr int NTHREADS = NCONS + 32;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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
// Wait for the phase of the given parity; false after WAIT_LIMIT_NS.
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
__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int BITS>
struct StageLayout {
    static constexpr int HI_OFF = SB * 16;
    static constexpr int SC_OFF = HI_OFF + (BITS == 6 ? SB * 8 : 0);
    static constexpr int MN_OFF = SC_OFF + SB * 2;
    static constexpr int BYTES = MN_OFF + SB * 2;
    static constexpr int BPB = 16 + (BITS == 6 ? 8 : 0) + 4;  // bytes per block
};

template <int BITS, int BC, int EPI, bool TWO>
__global__ void __launch_bounds__(NTHREADS, 1) gemv_stream_kernel(StreamParams p) {
    using L = StageLayout<BITS>;
    constexpr int NJ = TWO ? 2 : 1;  // distinct activation blocks per thread
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int log2nb = p.log2nb, nb = 1 << log2nb;
    const int stages = p.stages;

    // shared layout: ring | xq columns | wsum[2][BC][16] | full[stages] | empty[stages] | flags
    unsigned char* ring = smem;
    unsigned char* xqbase = ring + (size_t)stages * L::BYTES;
    const int xstride = xq_stride(nb);
    float* wsum = reinterpret_cast<float*>(xqbase + (size_t)BC * xstride);
    uint64_t* full = reinterpret_cast<uint64_t*>(wsum + 2 * BC * 16);
    uint64_t* empty = full + stages;
    int* abort_flag = reinterpret_cast<int*>(empty + stages);

    const long long r0 = (long long)blockIdx.x * p.n / gridDim.x;
    const long long r1 = (long long)(blockIdx.x + 1) * p.n / gridDim.x;
    const int nrows = (int)(r1 - r0);
    const int rps = TWO ? 1 : (SB >> log2nb);  // rows per stage
    const int nst = (nrows + rps - 1) / rps;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCONS / 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    float bv = __int_as_float(0x7fc00000);
    int bi = 0x7fffffff;

    if (warp == NCONS / 32) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            pdl_launch_dependents();
            const uint64_t pol = policy_evict_first();
            const size_t kb = (size_t)nb;  // blocks per row
            int slot = 0;
            uint32_t round = 0;
            for (int i = 0; i < nst; ++i) {
                if (i >= stages && !mbar_wait(&empty[slot], (round - 1) & 1u)) {
                    atomicOr(p.err, ERR_WAIT_EMPTY);
                    break;
                }
                if (*(volatile int*)abort_flag) break;
                const long long row = r0 + (long long)i * rps;
                const int rows_i = min(rps, nrows - i * rps);
                const uint32_t blocks = (uint32_t)rows_i * (uint32_t)nb;
                unsigned char* st = ring + (size_t)slot * L::BYTES;
                mbar_arrive_expect_tx(&full[slot], blocks * L::BPB);
                bulk_g2s(st, p.lo + (size_t)row * kb * 16, blocks * 16, &full[slot], pol);
                if constexpr (BITS == 6) bulk_g2s(st + L::HI_OFF, p.hi + (size_t)row * kb * 8, blocks * 8, &full[slot], pol);
                bulk_g2s(st + L::SC_OFF, p.scale + (size_t)row * kb, blocks * 2, &full[slot], pol);
                bulk_g2s(st + L::MN_OFF, p.min + (size_t)row * kb, blocks * 2, &full[slot], pol);
                if (++slot == stages) {
                    slot = 0;
                    ++round;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        pdl_wait();  // x and the outputs may belong to the preceding kernel
        for (int c = 0; c < p.batch; ++c)
            quantize_to_smem(p.x + (size_t)c * p.k, nb, xq_view(xqbase + c * xstride, nb), warp, NCONS / 32);
        consumer_bar();

        uint4 xl[BC][NJ], xh[BC][NJ];
        float xs[BC][NJ], xS[BC][NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int blk = (tid + NCONS * j) & (nb - 1);
#pragma unroll
            for (int c = 0; c < BC; ++c) {
                const XqView v = xq_view(xqbase + c * xstride, nb);
                if (c < p.batch) {
                    xl[c][j] = *reinterpret_cast<const uint4*>(v.lo + 16 * blk);
                    xh[c][j] = *reinterpret_cast<const uint4*>(v.hi + 16 * blk);
                    xs[c][j] = v.s[blk];
                    xS[c][j] = v.S[blk];
                } else {
                    xl[c][j] = make_uint4(0, 0, 0, 0);
                    xh[c][j] = make_uint4(0, 0, 0, 0);
                    xs[c][j] = 0.0f;
                    xS[c][j] = 0.0f;
                }
            }
        }

        int slot = 0, par = 0;
        uint32_t round = 0;
        for (int i = 0; i < nst; ++i) {
            if (!mbar_wait(&full[slot], round & 1u)) {
                atomicOr(p.err, ERR_WAIT_FULL);
                *(volatile int*)abort_flag = 1;
                break;
            }
            const unsigned char* st = ring + (size_t)slot * L::BYTES;
            const long long row0 = r0 + (long long)i * rps;
            const int rows_i = min(rps, nrows - i * rps);

            float part[BC][2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int fb = tid + NCONS * j;
                const bool valid = (fb >> log2nb) < rows_i;
#pragma unroll
                for (int c = 0; c < BC; ++c) part[c][j] = 0.0f;
                if (valid) {
                    const uint4 cw = *reinterpret_cast<const uint4*>(st + 16 * fb);
                    Codes32 cc;
                    if constexpr (BITS == 4)
                        cc = unpack_q4(cw);
                    else
                        cc = unpack_q6(cw, *reinterpret_cast<const uint2*>(st + L::HI_OFF + 8 * fb));
                    const float d = half_bits_to_float(*reinterpret_cast<const unsigned short*>(st + L::SC_OFF + 2 * fb));
                    const float m = half_bits_to_float(*reinterpret_cast<const unsigned short*>(st + L::MN_OFF + 2 * fb));
                    const int jj = TWO ? j : 0;
#pragma unroll
                    for (int c = 0; c < BC; ++c)
                        part[c][j] = block_combine(block_dot(cc, xl[c][jj], xh[c][jj]), d, m, xs[c][jj], xS[c][jj]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);

            if (nb < 32) {
                // rows of nb lanes inside a warp
                for (int off = nb >> 1; off > 0; off >>= 1) {
#pragma unroll
                    for (int c = 0; c < BC; ++c) {
                        part[c][0] += __shfl_xor_sync(0xffffffffu, part[c][0], off);
                        part[c][1] += __shfl_xor_sync(0xffffffffu, part[c][1], off);
                    }
                }
                if ((lane & (nb - 1)) == 0) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int rloc = (tid + NCONS * j) >> log2nb;
                        if (rloc < rows_i) {
                            const long long row = row0 + rloc;
                            if constexpr (EPI == EPI_STORE) {
#pragma unroll
                                for (int c = 0; c < BC; ++c)
                                    if (c < p.batch) p.y[(size_t)c * p.n + row] = part[c][j];
                            } else {
                                const float l = softcap_apply(part[0][j], p.softcap);
                                if (p.y) p.y[row] = l;
                                if (better(l, (int)row, bv, bi)) {
                                    bv = l;
                                    bi = (int)row;
                                }
                            }
                        }
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < BC; ++c) {
                    part[c][0] = warp_sum(part[c][0]);
                    part[c][1] = warp_sum(part[c][1]);
                }
                float* ws = wsum + par * (BC * 16);
                if (lane == 0) {
#pragma unroll
                    for (int c = 0; c < BC; ++c) {
                        ws[c * 16 + warp] = part[c][0];
                        ws[c * 16 + 8 + warp] = part[c][1];
                    }
                }
                consumer_bar();
                if (tid < rows_i) {
                    const int epw = nb >> 5;  // 32-block entries per row
                    const long long row = row0 + tid;
                    float tot[BC];
#pragma unroll
                    for (int c = 0; c < BC; ++c) {
                        float t = 0.0f;
                        for (int e = 0; e < epw; ++e) t += ws[c * 16 + tid * epw + e];
                        tot[c] = t;
                    }
                    if constexpr (EPI == EPI_STORE) {
#pragma unroll
                        for (int c = 0; c < BC; ++c)
                            if (c < p.batch) p.y[(size_t)c * p.n + row] = tot[c];
                    } else {
                        const float l = softcap_apply(tot[0], p.softcap);
                        if (p.y) p.y[row] = l;
                        if (better(l, (int)row, bv, bi)) {
                            bv = l;
                            bi = (int)row;
                        }
                    }
                }
                par ^= 1;
            }
            if (++slot == stages) {
                slot = 0;
                ++round;
            }
        }
    }

    if constexpr (EPI == EPI_ARGMAX) {
        __shared__ ArgmaxPartial sred[NTHREADS / 32];
        __shared__ int sflag;
        argmax_finish(bv, bi, p.ws, p.argmax, sred, &sflag);
    }
}

// ---------------------------------------------------------------- host side
static int env_int(const char* name, int dflt) {
    const char* v = getenv(name);
    if (!v || !*v) return dflt;
    return atoi(v);
}

bool stream_supported(int bits, int n, int k, int batch, int epi) {
    if (bits != 4 && bits != 6) return false;
    if (k < 256 || k > 16384 || (k & (k - 1)) != 0) return false;  // nb a power of two in [8, 512]
    const int nb = k >> 5;
    const int bc_max = nb == 512 ? 2 : 4;
    if (batch < 1 || batch > bc_max) return false;
    if (epi == EPI_ARGMAX && batch != 1) return false;
    (void)n;
    return true;
}

template <int BITS, int BC, int EPI, bool TWO>
static int launch_stream_t(StreamParams p, const LaunchCtx& lc) {
    using L = StageLayout<BITS>;
    auto kern = gemv_stream_kernel<BITS, BC, EPI, TWO>;
    const int nb = p.k >> 5;
    const size_t fixed = (size_t)BC * xq_stride(nb) + 2 * BC * 16 * sizeof(float) + 16;
    // ring depth: ~72 KB of shared memory per CTA by default, so that up to three
    // CTAs of consecutive launches can be resident on an SM under PDL
    const int budget = env_int("QG_STREAM_SMEM_KB", 72) * 1024;
    int stages = env_int("QG_STREAM_STAGES", 0);
    if (stages <= 0) stages = (int)((budget - (long long)fixed) / (L::BYTES + 16));
    if (stages < 2) stages = 2;
    if (stages > 32) stages = 32;
    size_t smem = (size_t)stages * (L::BYTES + 16) + fixed;
    const size_t cap = (size_t)lc.max_smem_optin - 1024;  // room for the kernel's static shared memory
    while (smem > cap && stages > 2) {
        --stages;
        smem = (size_t)stages * (L::BYTES + 16) + fixed;
    }
    if (smem > cap) return QG_ERR_UNSUPPORTED;
    if (int rc = ensure_smem_attr((const void*)kern, smem, lc)) return rc;
    p.stages = stages;
    p.err = lc.err;
    int per_sm = env_int("QG_STREAM_CTAS_PER_SM", 1);
    if (per_sm < 1) per_sm = 1;
    int grid = lc.sm_count * per_sm;
    if (EPI == EPI_ARGMAX && grid > VOCAB_MAX_CTAS) grid = VOCAB_MAX_CTAS;
    if (grid > p.n) grid = p.n;
    if (grid < 1) grid = 1;
    return launch_kernel(kern, dim3(grid), dim3(NTHREADS), smem, lc, p);
}

int launch_stream(const StreamParams& p0, int bits, int epi, const LaunchCtx& lc) {
    if (!stream_supported(bits, p0.n, p0.k, p0.batch, epi)) return QG_ERR_UNSUPPORTED;
    StreamParams p = p0;
    const int nb = p.k >> 5;
    int l = 0;
    while ((1 << l) < nb) ++l;
    p.log2nb = l;
    const bool two = nb == 512;
    if (epi == EPI_ARGMAX) {
        if (two) return bits == 4 ? launch_stream_t<4, 1, EPI_ARGMAX, true>(p, lc) : launch_stream_t<6, 1, EPI_ARGMAX, true>(p, lc);
        return bits == 4 ? launch_stream_t<4, 1, EPI_ARGMAX, false>(p, lc) : launch_stream_t<6, 1, EPI_ARGMAX, false>(p, lc);
    }
    const int bc = p.batch == 1 ? 1 : p.batch == 2 ? 2 : 4;
    if (two) {
        if (bc == 1) return bits == 4 ? launch_stream_t<4, 1, EPI_STORE, true>(p, lc) : launch_stream_t<6, 1, EPI_STORE, true>(p, lc);
        return bits == 4 ? launch_stream_t<4, 2, EPI_STORE, true>(p, lc) : launch_stream_t<6, 2, EPI_STORE, true>(p, lc);
    }
    switch (bc) {
        case 1:
            return bits == 4 ? launch_stream_t<4, 1, EPI_STORE, false>(p, lc) : launch_stream_t<6, 1, EPI_STORE, false>(p, lc);
        case 2:
            return bits == 4 ? launch_stream_t<4, 2, EPI_STORE, false>(p, lc) : launch_stream_t<6, 2, EPI_STORE, false>(p, lc);
        default:
            return bits == 4 ? launch_stream_t<4, 4, EPI_STORE, false>(p, lc) : launch_stream_t<6, 4, EPI_STORE, false>(p, lc);
    }
}

}  // namespace qg
