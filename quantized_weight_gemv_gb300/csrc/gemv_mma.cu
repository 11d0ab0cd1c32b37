// Small-batch Q4 MMVQ on tensor cores (batch 8..16).
//
// With B activation columns the Q4 GEMV becomes a thin dense contraction (oxinfer
// README, "Speculative decoding": at Q4 the multi-token int8 kernels are
// instruction-bound).  Per block of 32 weights the integer dots D[r][c] =
// sum code * xq are computed with mma.sync m16n8k16 (f16 in, f32 accumulate), fresh
// for every block so that the per-block scales are applied exactly as in the
// single-column kernels:  y[c][r] += s[c] * (d[r] * D[r][c] + m[r] * S[c]).
// Operand mapping (16 weight rows x 8 columns x 16 k per mma):
//  * the k order inside a block is permuted so that a thread's own 32-bit code word
//    is its A fragment: thread (g = lane/4, t = lane%4) reads bytes 4t..4t+3 of the
//    16-byte block of rows g and g+8.  Their low nibbles are elements 4t..4t+3 (first
//    mma): bytes 0 and 2 fill k-slots 2t, 2t+1 and bytes 1 and 3 (the word shifted
//    right by 8) k-slots 2t+8, 2t+9.  The high nibbles, elements 16+4t..16+4t+3, fill
//    the second mma in the same order, masked in place (16 x code).  A nibble v becomes
//    binary16 as the bits 0x6400 | v, which read as 1024 + v.
//  * the B fragments (activations) are written in the same permuted order straight
//    from the quantisation: each float4 of x quantises to exactly one 8-byte fragment;
//    the high half holds x/16, so the second mma adds 64 x + code x per element.
//  * the offsets come out exactly through the accumulator's initial value: the first
//    mma starts from -(1024 X_lo + 64 X_hi), X_lo and X_hi the sums of the block's
//    int8 activations over elements 0-15 and 16-31, so that after both mmas the
//    accumulator holds the block dot D = sum code * xq itself.
// Exactness: 1024 + v (v <= 240) and int8 activations (and their sixteenths) are exact
// in f16, every product is an integer below 2^17 and every partial sum, the initial
// value included, an integer below 2^23 in magnitude, so all of them are exact in f32.
//  * the activation image is made once per call into a workspace (prep kernel) and
//    pulled into shared memory with one bulk copy; 16 warps per CTA share it.
//  * a warp's task is one half of the k range of one group of 16 rows: 1-4 tiles of
//    16 rows x 8 blocks, put in flight at once through a private cp.async ring (all of
//    them for 8 columns, 3 at a time for 9-16)
//    (rows padded to 144 bytes so that the fragment reads are bank-conflict free);
//    warps w and w^1 take the two halves of a row group and add their partial sums
//    through shared memory under a named barrier of the pair (half 0 + half 1, in
//    that order).
#include <cuda_fp16.h>

#include "qg_internal.h"

namespace qg {
namespace mma {

constexpr int KC = 8;     // blocks per tile (256 elements of k)
constexpr int NW = 16;    // warps per CTA
// tiles in flight per warp: as many as shared memory holds at k = 2048 (a warp's task is
// one to four tiles, issued at once so that their DRAM latency is paid about once)
template <int NT>
__host__ __device__ constexpr int depth_of() { return NT == 1 ? 4 : 3; }

// d = a * b + c
__device__ __forceinline__ void mma_16816_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                              const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// two nibbles (bits 0-3 and 16-19 under `mask`, or 4-7 and 20-23) as 1024 + v in f16x2
__device__ __forceinline__ uint32_t nib_h2(uint32_t w, uint32_t mask) { return (w & mask) | 0x64006400u; }

// A fragments of one block from the code words of rows g (w0) and g+8 (w1)
__device__ __forceinline__ void a_frags(uint32_t w0, uint32_t w1, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
    const uint32_t v0 = w0 >> 8, v1 = w1 >> 8;
    lo[0] = nib_h2(w0, 0x000F000Fu);
    lo[1] = nib_h2(w1, 0x000F000Fu);
    lo[2] = nib_h2(v0, 0x000F000Fu);
    lo[3] = nib_h2(v1, 0x000F000Fu);
    hi[0] = nib_h2(w0, 0x00F000F0u);
    hi[1] = nib_h2(w1, 0x00F000F0u);
    hi[2] = nib_h2(v0, 0x00F000F0u);
    hi[3] = nib_h2(v1, 0x00F000F0u);
}

// binary16 number j (0..7) of eight packed in a uint4, as fp32
__device__ __forceinline__ float half8_at(const uint4& v, int j) {
    const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
    const __half2 h = *reinterpret_cast<const __half2*>(&w);
    return (j & 1) ? __high2float(h) : __low2float(h);
}

// two int8 activations as f16, optionally divided by 16 (exact: |q|/16 has at most
// 7 significant bits)
__device__ __forceinline__ uint32_t pack_h2(int a, int b, bool div16) {
    const float f = div16 ? 0.0625f : 1.0f;
    const __half2 h = __halves2half2(__float2half_rn((float)a * f), __float2half_rn((float)b * f));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// A weight tile in shared memory: codes [16 rows][144 B] (8 blocks + 16 B of padding),
// scale [16][8] and min [16][8] binary16.
constexpr int TILE_ROW = 144;
constexpr int TILE_CODES = 16 * TILE_ROW;
constexpr int TILE_BYTES = TILE_CODES + 2 * 16 * 16;

// Shared layout: frag[nb][NT][32][2] uint2 (a lane's low- and high-half B fragments
// side by side) | sS[nb][8*NT] (s, S) f32 pairs |
// C0[nb][8*NT] f32, the first mma's initial value (the activation image, also the
// workspace layout) | part[NW][16][8*NT] f32 | tiles[NW][depth_of<NT>()]
template <int NT>
struct Smem {
    __host__ __device__ static size_t frag_bytes(int nb) { return (size_t)nb * 2 * NT * 32 * 8; }
    __host__ __device__ static size_t sS_off(int nb) { return frag_bytes(nb); }
    __host__ __device__ static size_t C0_off(int nb) { return sS_off(nb) + (size_t)nb * 8 * NT * 8; }
    __host__ __device__ static size_t part_off(int nb) { return C0_off(nb) + (size_t)nb * 8 * NT * 4; }
    __host__ __device__ static size_t tiles_off(int nb) { return part_off(nb) + (size_t)NW * 16 * 8 * NT * 4; }
    __host__ __device__ static size_t bytes(int nb) { return tiles_off(nb) + (size_t)NW * depth_of<NT>() * TILE_BYTES; }
};

// Quantise the B activation columns straight into B fragments (image layout as
// Smem<NT> without the partial sums).  float4 number idx of column c (elements
// 4m..4m+3 of block b, m = idx & 7) becomes the fragment of lane 4*(c%8) + (m%4),
// tile c/8, k half m/4, as the pairs (q0, q2) and (q1, q3); the high half (m >= 4)
// holds x/16, so that its product with the 16x high-nibble codes accumulates onto the
// low half exactly.  Per block and column: s, S and -(1024 X_lo + 64 X_hi).  Items
// [item0, item0 + nthreads * rounds) of the 8*NT*k/4 float4s are done by threads
// t = 0..nthreads-1 (whole warps).
template <int NT>
__device__ __forceinline__ void quantize_to_frags(const float* __restrict__ X, int k, int batch, unsigned char* img,
                                                  int t, int nthreads, int item0, int item_end) {
    const int nb = k >> 5;
    uint2* frag = reinterpret_cast<uint2*>(img);
    float2* sS = reinterpret_cast<float2*>(img + Smem<NT>::sS_off(nb));
    float* C0 = reinterpret_cast<float*>(img + Smem<NT>::C0_off(nb));
    const int nf4 = k >> 2;
    const int total = min(8 * NT * nf4, item_end);  // columns beyond the batch quantise zeros
    const int nf4_log2 = __ffs(nf4) - 1;             // k is a power of two here (512..2048)
    constexpr int CHUNK = 8;
    for (int r0 = item0; r0 < total; r0 += nthreads * CHUNK) {
        float4 rv[CHUNK];
#pragma unroll
        for (int i = 0; i < CHUNK; ++i) {
            const int idx_all = r0 + i * nthreads + t;
            const int c = idx_all >> nf4_log2;
            rv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx_all < total && c < batch)
                rv[i] = __ldg(reinterpret_cast<const float4*>(X + (size_t)c * k) + (idx_all - c * nf4));
        }
#pragma unroll
        for (int i = 0; i < CHUNK; ++i) {
            if (r0 + i * nthreads >= total) break;  // the same for every thread: nothing left in this round
            const int idx_all = r0 + i * nthreads + t;
            const int c = idx_all >> nf4_log2;
            const int idx = idx_all - c * nf4;
            const float4 r = rv[i];
            float a = fmaxf(fmaxf(fabsf(r.x), fabsf(r.y)), fmaxf(fabsf(r.z), fabsf(r.w)));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            const float s = __fdiv_rn(a, 127.0f);
            int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
            if (s != 0.0f) {
                const float inv = __frcp_rn(s);
                q0 = quant_code(r.x, s, inv);
                q1 = quant_code(r.y, s, inv);
                q2 = quant_code(r.z, s, inv);
                q3 = quant_code(r.w, s, inv);
            }
            int H = q0 + q1 + q2 + q3;  // over the 4 float4s of this half of the block
            H += __shfl_xor_sync(0xffffffffu, H, 1);
            H += __shfl_xor_sync(0xffffffffu, H, 2);
            const int Ho = __shfl_xor_sync(0xffffffffu, H, 4);  // the other half
            if (idx_all < total) {
                const int b = idx >> 3, m = idx & 7;
                const int lane = 4 * (c & 7) + (m & 3);
                const bool hi = m >= 4;
                frag[((b * NT + (c >> 3)) * 32 + lane) * 2 + (m >> 2)] =
                    make_uint2(pack_h2(q0, q2, hi), pack_h2(q1, q3, hi));
                if (m == 0) {  // H = X_lo, Ho = X_hi
                    sS[b * 8 * NT + c] = make_float2(s, (float)(H + Ho));
                    C0[b * 8 * NT + c] = -(float)(1024 * H + 64 * Ho);
                }
            }
        }
    }
}

// The activation image, once per call, into the workspace (kernel 1 of 2).
template <int NT>
__global__ void __launch_bounds__(256) mma_prep_kernel(const float* __restrict__ X, int k, int batch,
                                                       unsigned char* __restrict__ img) {
    pdl_wait();
    if (threadIdx.x == 0) pdl_launch_dependents();
    const int item0 = blockIdx.x * 256;  // one float4 per thread: the image is on the GEMV's critical path
    quantize_to_frags<NT>(X, k, batch, img, threadIdx.x, 256, item0, item0 + 256);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// named barrier of the two warps holding one row group's k halves
__device__ __forceinline__ void pair_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Copies one tile (rows r0..r0+15 clamped to n, blocks blk0..blk0+7) into `tile` with
// the warp's lanes: 128 code chunks of 16 B, 16 scale rows and 16 min rows of 16 B.
__device__ __forceinline__ void issue_tile(const PlainParams& p, unsigned char* tile, int r0, int blk0, int lane) {
    const int nb = p.k >> 5;
    const size_t row_bytes = (size_t)(p.k >> 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i;
        const int row = c >> 3, col = c & 7;
        const int rr = min(r0 + row, p.n - 1);
        cp_async16(tile + row * TILE_ROW + col * 16, p.lo + (size_t)rr * row_bytes + (size_t)(blk0 + col) * 16);
    }
    const int row = lane & 15;
    const int rr = min(r0 + row, p.n - 1);
    const uint16_t* plane = lane < 16 ? p.scale : p.min;
    cp_async16(tile + TILE_CODES + (lane >> 4) * 256 + row * 16, plane + (size_t)rr * nb + blk0);
}

// The GEMV (kernel 2 of 2, or alone without a workspace).  With PREP the activation
// image comes from the workspace in one bulk copy; without, every CTA quantises.
template <int NT, bool PREP>
__global__ void __launch_bounds__(NW * 32, 1) mma_batched_kernel(PlainParams p, const unsigned char* img,
                                                                 unsigned int* err) {
    extern __shared__ __align__(16) unsigned char sm[];
    __shared__ __align__(8) uint64_t img_bar;
    const int nb = p.k >> 5;
    constexpr int DEPTH = depth_of<NT>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int n_groups = (p.n + 15) >> 4;
    unsigned char* tiles = sm + Smem<NT>::tiles_off(nb) + (size_t)warp * DEPTH * TILE_BYTES;

    // tasks: (row group, k half); warp w and w^1 hold the two halves of one row group
    const int half_nb = nb >> 1;
    const int TPT = half_nb / KC;                 // tiles per task: 1, 2 or 4
    const int LT = TPT == 1 ? 0 : TPT == 2 ? 1 : 2;  // log2(TPT)
    // this CTA's row groups: an equal share [rg0, rg1) of all, so that every SM takes
    // part; its tasks are the (row group, k half) pairs, warp w taking tasks w, w + NW, ...
    // (NW even: the two halves of a row group fall to warps w and w ^ 1)
    const int rg0 = (int)((long long)n_groups * blockIdx.x / gridDim.x);
    const int rg1 = (int)((long long)n_groups * (blockIdx.x + 1) / gridDim.x);
    const int n_tasks = 2 * (rg1 - rg0);
    const int wstride = NW;
    const int task0 = warp;
    const int my_tasks = task0 < n_tasks ? (n_tasks - task0 + wstride - 1) / wstride : 0;
    const int n_tiles = my_tasks * TPT;
    auto tile_rg = [&](int q) { return rg0 + ((task0 + (q >> LT) * wstride) >> 1); };
    auto tile_blk = [&](int q) { return (warp & 1) * half_nb + (q & (TPT - 1)) * KC; };

    // weights do not depend on earlier work: start the first tiles before waiting for it
#pragma unroll
    for (int d = 0; d < DEPTH; ++d) {
        if (d < n_tiles) issue_tile(p, tiles + d * TILE_BYTES, tile_rg(d) * 16, tile_blk(d), lane);
        cp_async_commit();
    }

    pdl_wait();
    if (threadIdx.x == 0) pdl_launch_dependents();
    if constexpr (PREP) {
        const uint32_t bytes = (uint32_t)Smem<NT>::part_off(nb);
        if (threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&img_bar)) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&img_bar)),
                         "r"(bytes)
                         : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(sm)),
                "l"(img), "r"(bytes), "r"(smem_u32(&img_bar))
                : "memory");
        }
        // thread 0 waits for the image (bounded); the block barrier below then orders the
        // landed bytes for every other thread
        uint32_t ok = 1;
        if (threadIdx.x == 0) {
            const unsigned long long t0 = globaltimer_ns();
            for (;;) {
                asm volatile(
                    "{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], 0;\n\t"
                    "selp.u32 %0, 1, 0, q;\n\t}"
                    : "=r"(ok)
                    : "r"(smem_u32(&img_bar))
                    : "memory");
                if (ok || globaltimer_ns() - t0 > WAIT_LIMIT_NS) break;
            }
        }
        // give up together if the copy never landed (bounded wait), leaving the error word set
        if (__syncthreads_or(ok == 0)) {
            if (threadIdx.x == 0) atomicOr(err, ERR_WAIT_FULL);
            cp_async_wait<0>();
            return;
        }
    } else {
        quantize_to_frags<NT>(p.x, p.k, p.batch, sm, threadIdx.x, NW * 32, 0, 1 << 30);
    }
    __syncthreads();

    const uint2* frag = reinterpret_cast<const uint2*>(sm);
    const float2* sS = reinterpret_cast<const float2*>(sm + Smem<NT>::sS_off(nb));
    const float* C0 = reinterpret_cast<const float*>(sm + Smem<NT>::C0_off(nb));
    float* part = reinterpret_cast<float*>(sm + Smem<NT>::part_off(nb));

    float* mine = part + (size_t)warp * 16 * 8 * NT;
    const float* other = part + (size_t)(warp ^ 1) * 16 * 8 * NT;
    const int pair_bar = 1 + (warp >> 1);
    for (int task = 0; task < my_tasks; ++task) {
        const int rg = rg0 + ((task0 + task * wstride) >> 1);
        float acc[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
        for (int jt = 0; jt < TPT; ++jt) {
            const int q = task * TPT + jt;
            const unsigned char* tile = tiles + (q % DEPTH) * TILE_BYTES;
            cp_async_wait<DEPTH - 1>();
            __syncwarp();
            // scale and min of rows g and g+8 for the tile's 8 blocks (16 bytes a row)
            const uint4 dg = *reinterpret_cast<const uint4*>(tile + TILE_CODES + g * 16);
            const uint4 dg8 = *reinterpret_cast<const uint4*>(tile + TILE_CODES + (g + 8) * 16);
            const uint4 mg = *reinterpret_cast<const uint4*>(tile + TILE_CODES + 256 + g * 16);
            const uint4 mg8 = *reinterpret_cast<const uint4*>(tile + TILE_CODES + 256 + (g + 8) * 16);
            const int blk0 = tile_blk(q);
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                const int b = blk0 + j;
                const uint32_t w0 = *reinterpret_cast<const uint32_t*>(tile + g * TILE_ROW + j * 16 + 4 * t);
                const uint32_t w1 = *reinterpret_cast<const uint32_t*>(tile + (g + 8) * TILE_ROW + j * 16 + 4 * t);
                uint32_t alo[4], ahi[4];
                a_frags(w0, w1, alo, ahi);
                const float d0 = half8_at(dg, j), d1 = half8_at(dg8, j);
                const float m0 = half8_at(mg, j), m1 = half8_at(mg8, j);
#pragma unroll
                for (int tt = 0; tt < NT; ++tt) {
                    const uint4 bf = *reinterpret_cast<const uint4*>(frag + ((b * NT + tt) * 32 + lane) * 2);
                    const int col = b * 8 * NT + tt * 8 + 2 * t;
                    const float4 ss = *reinterpret_cast<const float4*>(sS + col);  // (s, S) of cols 2t, 2t+1
                    const float2 c0 = *reinterpret_cast<const float2*>(C0 + col);
                    const float cinit[4] = {c0.x, c0.y, c0.x, c0.y};
                    float dl[4], D[4];
                    mma_16816_acc(dl, alo, bf.x, bf.y, cinit);
                    mma_16816_acc(D, ahi, bf.z, bf.w, dl);  // exact integer block dots
                    // (row g, col 2t), (row g, col 2t+1), (row g+8, col 2t), (row g+8, col 2t+1)
                    acc[tt][0] = fmaf(ss.x, fmaf(d0, D[0], m0 * ss.y), acc[tt][0]);
                    acc[tt][1] = fmaf(ss.z, fmaf(d0, D[1], m0 * ss.w), acc[tt][1]);
                    acc[tt][2] = fmaf(ss.x, fmaf(d1, D[2], m1 * ss.y), acc[tt][2]);
                    acc[tt][3] = fmaf(ss.z, fmaf(d1, D[3], m1 * ss.w), acc[tt][3]);
                }
            }
            __syncwarp();
            // refill this slot with tile q + DEPTH (an empty group keeps the count)
            if (q + DEPTH < n_tiles)
                issue_tile(p, tiles + (q % DEPTH) * TILE_BYTES, tile_rg(q + DEPTH) * 16, tile_blk(q + DEPTH), lane);
            cp_async_commit();
        }
        // the two k halves of the row group meet: half 1 leaves its sums, half 0 adds them
#pragma unroll
        for (int tt = 0; tt < NT; ++tt) {
            mine[g * 8 * NT + tt * 8 + 2 * t] = acc[tt][0];
            mine[g * 8 * NT + tt * 8 + 2 * t + 1] = acc[tt][1];
            mine[(g + 8) * 8 * NT + tt * 8 + 2 * t] = acc[tt][2];
            mine[(g + 8) * 8 * NT + tt * 8 + 2 * t + 1] = acc[tt][3];
        }
        pair_sync(pair_bar);
        if ((warp & 1) == 0) {
            for (int o = lane; o < 16 * 8 * NT; o += 32) {
                const int r = o / (8 * NT), c = o - r * 8 * NT;
                const int row = rg * 16 + r;
                if (c < p.batch && row < p.n) p.y[(size_t)c * p.n + row] = mine[o] + other[o];
            }
        }
        pair_sync(pair_bar);  // both partial arrays are free for the next task
    }
    cp_async_wait<0>();
}

}  // namespace mma

bool mma_supported(int bits, int k, int batch) {
    const int nb = k >> 5;
    return bits == 4 && batch >= 8 && batch <= 16 && (nb == 16 || nb == 32 || nb == 64);
}

size_t mma_workspace_bytes(int k, int batch) {
    const int nb = k >> 5;
    return batch <= 8 ? mma::Smem<1>::part_off(nb) : mma::Smem<2>::part_off(nb);
}

template <int NT>
static int launch_mma_t(const PlainParams& p, unsigned char* ws, const LaunchCtx& lc) {
    const int nb = p.k >> 5;
    const int n_groups = (p.n + 15) >> 4;
    const size_t smem = mma::Smem<NT>::bytes(nb);
    if (smem > (size_t)lc.max_smem_optin - 1024) return QG_ERR_UNSUPPORTED;
    int grid = n_groups;  // at most one row group per CTA ...
    if (grid > lc.sm_count) grid = lc.sm_count;  // ... and one CTA per SM, every SM taking part
    if (grid < 1) grid = 1;
    if (!ws) {
        auto kern = mma::mma_batched_kernel<NT, false>;
        if (int rc = ensure_smem_attr((const void*)kern, smem, lc)) return rc;
        return launch_kernel(kern, dim3(grid), dim3(mma::NW * 32), smem, lc, p, (const unsigned char*)nullptr, lc.err);
    }
    // 1. the activation image, once; 2. the GEMV, chained by programmatic dependent launch
    const int items = 8 * NT * (p.k >> 2);
    const int pgrid = (items + 255) / 256;
    int rc = launch_kernel(mma::mma_prep_kernel<NT>, dim3(pgrid), dim3(256), 0, lc, p.x, p.k, p.batch, ws);
    if (rc != QG_OK) return rc;
    auto kern = mma::mma_batched_kernel<NT, true>;
    if (int e = ensure_smem_attr((const void*)kern, smem, lc)) return e;
    LaunchCtx lc2 = lc;
    lc2.flags |= QG_FLAG_PDL;
    return launch_kernel(kern, dim3(grid), dim3(mma::NW * 32), smem, lc2, p, (const unsigned char*)ws, lc.err);
}

int launch_mma(const PlainParams& p, unsigned char* ws, const LaunchCtx& lc) {
    return p.batch <= 8 ? launch_mma_t<1>(p, ws, lc) : launch_mma_t<2>(p, ws, lc);
}

}  // namespace qg
