// Internal declarations shared by the kernel files and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qg_common.cuh"

namespace qg {

// Epilogue of the single-matrix kernels: plain store; soft-cap + argmax; soft-cap +
// constrained selection (log-sum-exp and best allowed id, stream kernel only).
enum : int { EPI_STORE = 0, EPI_ARGMAX = 1, EPI_SELECT = 2 };

// per-column shared-memory stride of a quantised activation (16-byte aligned)
__host__ __device__ constexpr int xq_stride(int nb) { return (xq_bytes(nb) + 15) & ~15; }

struct PlainParams {
    const uint8_t* lo;
    const uint8_t* hi;
    const uint16_t* scale;
    const uint16_t* min;
    int n, k, batch;
    const float* x;  // [batch][k]
    float* y;        // EPI_STORE: [batch][n]; EPI_ARGMAX: logits [n] or null
    float softcap;
    int32_t* argmax;
    VocabWorkspace* ws;
};

struct StreamParams {
    const uint8_t* lo;
    const uint8_t* hi;
    const uint16_t* scale;
    const uint16_t* min;
    int n, k, batch;
    int stages;  // ring depth
    const float* x;
    float* y;
    float softcap;
    int32_t* argmax;
    VocabWorkspace* ws;
    unsigned int* err;  // device error word
    // EPI_SELECT: allowed ids (null: all), the selected id and its log-probability
    const int32_t* allowed;
    int n_allowed;
    int32_t* token;
    float* logprob;
    SelectWorkspace* sws;
};

struct CqParams {
    const uint8_t* idx;
    const uint16_t* codebook;
    const uint16_t* row_scale;
    int n, k, group, row_start, row_count;
    float inv_sqrt_group;
    const float* x;
    float* y;
};

// Per-call launch context resolved by the C-ABI layer.
struct LaunchCtx {
    cudaStream_t stream;
    unsigned flags;
    int device;
    int sm_count;
    int max_smem_optin;
    unsigned int* err;  // device address of the error word
    int cluster = 1;    // thread-block cluster size of the launch (1: none)
};

int ensure_smem_attr(const void* kernel, size_t smem, const LaunchCtx& lc);
// resident clusters of `cluster` CTAs at once (cudaOccupancyMaxActiveClusters, cached); 0 on failure
int max_active_clusters(const void* kernel, int cluster, int block, size_t smem, const LaunchCtx& lc);

template <typename... KArgs, typename... Args>
int launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, const LaunchCtx& lc, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (lc.flags & QG_FLAG_PDL) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (lc.cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)lc.cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (na) {
        cfg.attrs = attr;
        cfg.numAttrs = na;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return QG_ERR_CUDA;
    }
    return QG_OK;
}

int launch_plain(const PlainParams& p, int bits, int epi, const LaunchCtx& lc);
// returns QG_ERR_UNSUPPORTED when the shape has no bulk-copy variant
int launch_stream(const StreamParams& p, int bits, int epi, const LaunchCtx& lc);
bool stream_supported(int bits, int n, int k, int batch, int epi);
// split-K streaming for short-N / long-K single GEMVs (gemv_splitk.cu)
bool splitk_wanted(int n, int k, int batch, int epi);
int launch_splitk(const StreamParams& p, int bits, const LaunchCtx& lc);
int launch_cq(const CqParams& p, const LaunchCtx& lc);
// tensor-core small-batch MMVQ (Q4, batch 8..16)
bool mma_supported(int bits, int k, int batch);
size_t mma_workspace_bytes(int k, int batch);
// ws: the activation image (mma_workspace_bytes), or null to quantise in every CTA
int launch_mma(const PlainParams& p, unsigned char* ws, const LaunchCtx& lc);
size_t grouped_workspace_bytes(const qg_gemv_desc* descs, int count);
// descriptor checks shared by qgemv_grouped and qgemv_grouped_noalloc (capi.cu)
int check_grouped(int bits, const qg_gemv_desc* descs, int count, int* active);
// Whether launch_grouped(..., fuse = true) takes the one-launch form for this group:
// its distinct activations (by x and k) are short enough to be quantised in every CTA.
bool grouped_fuses(const qg_gemv_desc* descs, int count);
// An activation image that a grouped launch produces for the next launch from the
// output of its descriptor `desc` (index into its descs array, n % 32 == 0): written
// to img in the workspace image layout for k = n.
constexpr int GROUPED_MAX_OUT = 4;
struct GroupedOut {
    int desc;
    unsigned char* img;
};
// fuse: allow the one-launch form (activations quantised in every CTA) when they are
// short.  outs/nout: images to produce for the next launch.  images_ready: the
// workspace images were produced by the preceding launch (no quantisation launch;
// the GEMV kernel is chained to that launch by the caller's QG_FLAG_PDL).
int launch_grouped(int bits, const qg_gemv_desc* descs, int count, unsigned char* ws, const LaunchCtx& lc,
                   bool fuse = false, const GroupedOut* outs = nullptr, int nout = 0, bool images_ready = false);
size_t chain_workspace_bytes(const qg_gemv_desc* descs, int count, const int* phase_sizes, int nphase);
// ws: the caller's chain workspace (control words first); arguments already validated
int launch_chain(int bits, const qg_gemv_desc* descs, int count, const int* phase_sizes, int nphase,
                 unsigned char* ws, const LaunchCtx& lc);
int launch_select(const float* logits, int n, const int32_t* allowed, int n_allowed, int32_t* token, float* logprob,
                  SelectWorkspace* ws, const LaunchCtx& lc);
int launch_read_floor(const void* src, size_t bytes, uint32_t* out, const LaunchCtx& lc);
int launch_quantize_act(const float* x, int k, int batch, int8_t* xq, float* xs, int32_t* xsum, const LaunchCtx& lc);
int launch_blockdots(int bits, const uint8_t* lo, const uint8_t* hi, int n, int k, const int8_t* xq, int32_t* dots,
                     const LaunchCtx& lc);

}  // namespace qg
