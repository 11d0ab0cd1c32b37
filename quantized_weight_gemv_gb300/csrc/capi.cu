// C ABI of the library: argument validation, variant choice, launch.
#include <mutex>

#include "qg_internal.h"

namespace qg {

// Device error word (see qg_device_error); kernels get its address as a parameter.
__device__ unsigned int g_error_word = 0u;

namespace {

constexpr int MAX_DEVICES = 64;

struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int max_smem_optin = 0;
    unsigned int* err = nullptr;
};
DeviceInfo g_dev[MAX_DEVICES];
std::mutex g_mu;

// (kernel, device) pairs whose opt-in shared-memory limit was already raised
struct AttrEntry {
    const void* kernel;
    int device;
    size_t smem;
};
AttrEntry g_attr[512];
int g_attr_n = 0;

int resolve(void* stream, unsigned flags, LaunchCtx& lc) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        (void)cudaGetLastError();
        return QG_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& di = g_dev[dev];
    if (!di.ready) {
        if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaGetSymbolAddress(reinterpret_cast<void**>(&di.err), g_error_word) != cudaSuccess) {
            (void)cudaGetLastError();
            return QG_ERR_CUDA;
        }
        di.ready = true;
    }
    lc.stream = reinterpret_cast<cudaStream_t>(stream);
    lc.flags = flags;
    lc.device = dev;
    lc.sm_count = di.sm_count;
    lc.max_smem_optin = di.max_smem_optin;
    lc.err = di.err;
    return QG_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int ensure_smem_attr(const void* kernel, size_t smem, const LaunchCtx& lc) {
    if (smem <= 48 * 1024) return QG_OK;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_attr_n; ++i)
        if (g_attr[i].kernel == kernel && g_attr[i].device == lc.device) return g_attr[i].smem >= smem ? QG_OK : QG_ERR_UNSUPPORTED;
    // raise to the most the kernel can take beside its static shared memory, once, so
    // that later calls with other sizes need no new call
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
        (void)cudaGetLastError();
        return QG_ERR_CUDA;
    }
    const int maxdyn = lc.max_smem_optin - (int)fa.sharedSizeBytes;
    if (maxdyn < (int)smem) return QG_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, maxdyn) != cudaSuccess) {
        (void)cudaGetLastError();
        return QG_ERR_CUDA;
    }
    if (g_attr_n < 512) g_attr[g_attr_n++] = AttrEntry{kernel, lc.device, (size_t)maxdyn};
    return QG_OK;
}

// How many thread-block clusters of `cluster` CTAs (block threads, smem bytes of dynamic
// shared memory each) can be resident on the device at once; cached per (kernel,
// device, cluster, smem).  0 on failure.
int max_active_clusters(const void* kernel, int cluster, int block, size_t smem, const LaunchCtx& lc) {
    struct Entry {
        const void* kernel;
        int device, cluster, block;
        size_t smem;
        int count;
    };
    static Entry cache[64];
    static int n = 0;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].kernel == kernel && cache[i].device == lc.device && cache[i].cluster == cluster &&
            cache[i].block == block && cache[i].smem == smem)
            return cache[i].count;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cluster * lc.sm_count));
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = (unsigned)cluster;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int count = 0;
    if (cudaOccupancyMaxActiveClusters(&count, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (n < 64) cache[n++] = Entry{kernel, lc.device, cluster, block, smem, count};
    return count;
}

static int check_weights(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min,
                         int n, int k) {
    if (bits != 2 && bits != 4 && bits != 6) return QG_ERR_UNSUPPORTED;
    if (n < 0 || k <= 0 || (k & 31) != 0 || k > QG_MAX_K) return QG_ERR_INVALID_ARG;
    if (n == 0) return QG_OK;
    // Q2 has no hi and no min plane (zero point 2); Q4 no hi plane
    if (!lo || !scale || (bits != 2 && !min) || (bits == 2 && min) || (bits == 6 && !hi) || (bits != 6 && hi))
        return QG_ERR_INVALID_ARG;
    if (!aligned16(lo) || (bits == 6 && !aligned16(hi)) || !aligned16(scale) || (bits != 2 && !aligned16(min)))
        return QG_ERR_ALIGNMENT;
    return QG_OK;
}

static int gemv_common(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min,
                       int n, int k, int batch, const float* x, float* y, void* ws, size_t ws_bytes, unsigned flags,
                       void* stream) {
    int rc = check_weights(bits, lo, hi, scale, min, n, k);
    if (rc != QG_OK) return rc;
    if (batch < 1 || batch > QG_MAX_BATCH || (long long)batch * k > 131072) return QG_ERR_INVALID_ARG;
    if (n == 0) return QG_OK;
    if (!x || !y) return QG_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return QG_ERR_ALIGNMENT;
    const bool use_mma = !(flags & QG_FLAG_PLAIN) && mma_supported(bits, k, batch);
    if (ws) {
        if (!aligned16(ws)) return QG_ERR_ALIGNMENT;
        if (use_mma && ws_bytes < mma_workspace_bytes(k, batch)) return QG_ERR_WORKSPACE;
    }
    LaunchCtx lc;
    rc = resolve(stream, flags, lc);
    if (rc != QG_OK) return rc;
    PlainParams pp = {lo, hi, scale, min, n, k, batch, x, y, 0.0f, nullptr, nullptr};
    if (use_mma) {
        rc = launch_mma(pp, reinterpret_cast<unsigned char*>(ws), lc);
        if (rc != QG_ERR_UNSUPPORTED) return rc;
    }
    if (!(flags & QG_FLAG_PLAIN) && stream_supported(bits, n, k, batch, EPI_STORE)) {
        StreamParams sp = {lo, hi, scale, min, n, k, batch, 0, x, y, 0.0f, nullptr, nullptr, nullptr};
        rc = launch_stream(sp, bits, EPI_STORE, lc);
        if (rc != QG_ERR_UNSUPPORTED) return rc;
    }
    return launch_plain(pp, bits, EPI_STORE, lc);
}

// The descriptor list of a grouped call: bits 4 or 6, 0 <= count <= QG_MAX_GROUP, every
// descriptor with n >= 0 and k a power of two in [1024, 16384], and the weights, x and y
// of every non-empty one present and aligned.  *active receives the non-empty count.
int check_grouped(int bits, const qg_gemv_desc* descs, int count, int* active) {
    *active = 0;
    if (bits != 4 && bits != 6) return QG_ERR_UNSUPPORTED;
    if (count < 0 || count > QG_MAX_GROUP) return QG_ERR_INVALID_ARG;
    if (count == 0) return QG_OK;
    if (!descs) return QG_ERR_INVALID_ARG;
    for (int i = 0; i < count; ++i) {
        const qg_gemv_desc& d = descs[i];
        if (d.n < 0) return QG_ERR_INVALID_ARG;
        if (d.k < 1024 || d.k > 16384 || (d.k & (d.k - 1)) != 0) return QG_ERR_UNSUPPORTED;
        if (d.n == 0) continue;
        int rc = check_weights(bits, d.lo, d.hi, d.scale, d.min, d.n, d.k);
        if (rc != QG_OK) return rc;
        if (!d.x || !d.y) return QG_ERR_INVALID_ARG;
        if (!aligned16(d.x) || !aligned16(d.y)) return QG_ERR_ALIGNMENT;
        ++*active;
    }
    return QG_OK;
}

}  // namespace qg

using namespace qg;

extern "C" {

const char* qg_status_string(int status) {
    switch (status) {
        case QG_OK:
            return "ok";
        case QG_ERR_INVALID_ARG:
            return "invalid argument";
        case QG_ERR_ALIGNMENT:
            return "buffer not 16-byte aligned";
        case QG_ERR_UNSUPPORTED:
            return "unsupported format or size";
        case QG_ERR_WORKSPACE:
            return "workspace missing or too small";
        case QG_ERR_CUDA:
            return "CUDA launch failed";
    }
    return "unknown status";
}

int qg_version(void) { return 100; }

int qg_device_error(uint32_t* code) {
    if (!code) return QG_ERR_INVALID_ARG;
    unsigned int v = 0, zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return QG_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return QG_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return QG_ERR_CUDA;
    *code = v;
    return QG_OK;
}

int qgemv_q4(const uint8_t* codes, const uint16_t* scale, const uint16_t* min, int n, int k, const float* x,
             float* y, unsigned flags, void* stream) {
    return gemv_common(4, codes, nullptr, scale, min, n, k, 1, x, y, nullptr, 0, flags, stream);
}

int qgemv_q2(const uint8_t* codes, const uint16_t* scale, int n, int k, const float* x, float* y, unsigned flags,
             void* stream) {
    return gemv_common(2, codes, nullptr, scale, nullptr, n, k, 1, x, y, nullptr, 0, flags, stream);
}

int qgemv_q6(const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min, int n, int k,
             const float* x, float* y, unsigned flags, void* stream) {
    if (!hi && n > 0) return QG_ERR_INVALID_ARG;
    return gemv_common(6, lo, hi, scale, min, n, k, 1, x, y, nullptr, 0, flags, stream);
}

size_t qg_batched_workspace_bytes(int bits, int k, int batch) {
    if (k <= 0 || (k & 31) != 0 || k > QG_MAX_K || batch < 1 || batch > QG_MAX_BATCH) return 0;
    return mma_supported(bits, k, batch) ? mma_workspace_bytes(k, batch) : 0;
}

int qgemv_batched(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min, int n,
                  int k, int batch, const float* X, float* Y, void* ws, size_t ws_bytes, unsigned flags,
                  void* stream) {
    return gemv_common(bits, lo, hi, scale, min, n, k, batch, X, Y, ws, ws_bytes, flags, stream);
}

int cq_fwht_matvec(const uint8_t* idx, const uint16_t* codebook, const uint16_t* row_scale, int n, int k, int group,
                   int row_start, int row_count, const float* x, float* y, unsigned flags, void* stream) {
    if (group != 128 && group != 256 && group != 512 && group != 1024) return QG_ERR_UNSUPPORTED;
    if (n < 0 || k <= 0 || k % group != 0 || k > QG_MAX_CQ_K) return QG_ERR_INVALID_ARG;
    if (row_start < 0 || row_count < 0 || (long long)row_start + row_count > n) return QG_ERR_INVALID_ARG;
    if (row_count == 0) return QG_OK;
    if (!idx || !codebook || !row_scale || !x || !y) return QG_ERR_INVALID_ARG;
    if (!aligned16(idx) || !aligned16(x) || !aligned16(y)) return QG_ERR_ALIGNMENT;
    LaunchCtx lc;
    int rc = resolve(stream, flags, lc);
    if (rc != QG_OK) return rc;
    CqParams p = {idx, codebook, row_scale, n, k, group, row_start, row_count,
                  (float)(1.0 / sqrt((double)group)), x, y};
    return launch_cq(p, lc);
}

size_t qg_vocab_workspace_bytes(void) { return sizeof(VocabWorkspace); }

int vocab_softcap_argmax(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min,
                         int n_vocab, int k, const float* x, float softcap, float* logits, int32_t* argmax, void* ws,
                         size_t ws_bytes, unsigned flags, void* stream) {
    int rc = check_weights(bits, lo, hi, scale, min, n_vocab, k);
    if (rc != QG_OK) return rc;
    if (n_vocab < 1) return QG_ERR_INVALID_ARG;
    if (!x || !argmax) return QG_ERR_INVALID_ARG;
    if (!(softcap == softcap)) return QG_ERR_INVALID_ARG;  // NaN cap
    if (!aligned16(x) || (logits && !aligned16(logits))) return QG_ERR_ALIGNMENT;
    if (!ws || ws_bytes < sizeof(VocabWorkspace)) return QG_ERR_WORKSPACE;
    if (!aligned16(ws)) return QG_ERR_ALIGNMENT;
    LaunchCtx lc;
    rc = resolve(stream, flags, lc);
    if (rc != QG_OK) return rc;
    VocabWorkspace* w = reinterpret_cast<VocabWorkspace*>(ws);
    if (!(flags & QG_FLAG_PLAIN) && stream_supported(bits, n_vocab, k, 1, EPI_ARGMAX)) {
        StreamParams sp = {lo, hi, scale, min, n_vocab, k, 1, 0, x, logits, softcap, argmax, w, nullptr};
        rc = launch_stream(sp, bits, EPI_ARGMAX, lc);
        if (rc != QG_ERR_UNSUPPORTED) return rc;
    }
    PlainParams pp = {lo, hi, scale, min, n_vocab, k, 1, x, logits, softcap, argmax, w};
    return launch_plain(pp, bits, EPI_ARGMAX, lc);
}

size_t qg_select_workspace_bytes(void) { return sizeof(SelectWorkspace); }

int qg_logits_select(const float* logits, int n, const int32_t* allowed, int n_allowed, int32_t* token,
                     float* logprob, void* ws, size_t ws_bytes, unsigned flags, void* stream) {
    if (n < 1 || !logits || !token || !logprob) return QG_ERR_INVALID_ARG;
    if (allowed && n_allowed < 0) return QG_ERR_INVALID_ARG;
    if (!ws || ws_bytes < sizeof(SelectWorkspace)) return QG_ERR_WORKSPACE;
    if (!aligned16(ws)) return QG_ERR_ALIGNMENT;
    LaunchCtx lc;
    int rc = resolve(stream, flags, lc);
    if (rc != QG_OK) return rc;
    return launch_select(logits, n, allowed, allowed ? n_allowed : 0, token, logprob,
                         reinterpret_cast<SelectWorkspace*>(ws), lc);
}

size_t qg_vocab_select_workspace_bytes(void) { return sizeof(VocabWorkspace) + sizeof(SelectWorkspace); }

int vocab_softcap_select(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min,
                         int n_vocab, int k, const float* x, float softcap, const int32_t* allowed, int n_allowed,
                         float* logits, int32_t* token, float* logprob, void* ws, size_t ws_bytes, unsigned flags,
                         void* stream) {
    if (!logits || !token || !logprob) return QG_ERR_INVALID_ARG;
    if (allowed && n_allowed < 0) return QG_ERR_INVALID_ARG;
    if (!ws || ws_bytes < qg_vocab_select_workspace_bytes()) return QG_ERR_WORKSPACE;
    if (!aligned16(ws)) return QG_ERR_ALIGNMENT;
    unsigned char* w = reinterpret_cast<unsigned char*>(ws);
    SelectWorkspace* sw = reinterpret_cast<SelectWorkspace*>(w + sizeof(VocabWorkspace));
    // one launch: the streaming kernel's selection epilogue (every CTA scans the allowed
    // list once, hence the bound on its length)
    if (!(flags & QG_FLAG_PLAIN) && (!allowed || n_allowed <= QG_SELECT_FUSED_MAX_ALLOWED) &&
        stream_supported(bits, n_vocab, k, 1, EPI_SELECT)) {
        int rc = check_weights(bits, lo, hi, scale, min, n_vocab, k);
        if (rc != QG_OK) return rc;
        if (n_vocab < 1 || !x) return QG_ERR_INVALID_ARG;
        if (!(softcap == softcap)) return QG_ERR_INVALID_ARG;  // NaN cap
        if (!aligned16(x) || !aligned16(logits)) return QG_ERR_ALIGNMENT;
        LaunchCtx lc;
        rc = resolve(stream, flags, lc);
        if (rc != QG_OK) return rc;
        StreamParams sp = {lo,      hi,       scale,   min,     n_vocab, k,      1,        0,
                           x,       logits,   softcap, nullptr, nullptr, nullptr, allowed, allowed ? n_allowed : 0,
                           token,   logprob,  sw};
        rc = launch_stream(sp, bits, EPI_SELECT, lc);
        if (rc != QG_ERR_UNSUPPORTED) return rc;
    }
    // 1. the soft-capped logits (its unconstrained argmax goes to the workspace's scratch word)
    int rc = vocab_softcap_argmax(bits, lo, hi, scale, min, n_vocab, k, x, softcap, logits, &sw->scratch_index, w,
                                  sizeof(VocabWorkspace), flags, stream);
    if (rc != QG_OK) return rc;
    // 2. the selection, chained by programmatic dependent launch
    return qg_logits_select(logits, n_vocab, allowed, n_allowed, token, logprob, sw, sizeof(SelectWorkspace),
                            flags | QG_FLAG_PDL, stream);
}

size_t qg_grouped_workspace_bytes(const qg_gemv_desc* descs, int count) {
    if (!descs || count <= 0 || count > QG_MAX_GROUP) return 0;
    return grouped_workspace_bytes(descs, count);
}

// [a, a + na) and [b, b + nb) share a byte
static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

// Shape of a chain: phase sizes, every descriptor as qgemv_grouped wants it, and the
// per-phase rules (no output overlapping an output or input of its phase; distinct
// inputs of a phase within QG_CHAIN_MAX_PHASE_K values).
static int check_chain(int bits, const qg_gemv_desc* descs, int count, const int* phase_sizes, int n_phases,
                       int* active) {
    if (bits != 4 && bits != 6) return QG_ERR_UNSUPPORTED;
    if (count < 0 || count > QG_MAX_GROUP || n_phases < 0 || n_phases > count) return QG_ERR_INVALID_ARG;
    *active = 0;
    if (count == 0) return n_phases == 0 ? QG_OK : QG_ERR_INVALID_ARG;
    if (!descs || !phase_sizes || n_phases < 1) return QG_ERR_INVALID_ARG;
    long long sum = 0;
    for (int f = 0; f < n_phases; ++f) {
        if (phase_sizes[f] < 1) return QG_ERR_INVALID_ARG;
        sum += phase_sizes[f];
    }
    if (sum != count) return QG_ERR_INVALID_ARG;
    int off = 0;
    for (int f = 0; f < n_phases; ++f) {
        const qg_gemv_desc* ph = descs + off;
        const int m = phase_sizes[f];
        long long in_k = 0;
        for (int i = 0; i < m; ++i) {
            const qg_gemv_desc& d = ph[i];
            if (d.n < 0) return QG_ERR_INVALID_ARG;
            if (d.k < 1024 || d.k > 16384 || (d.k & (d.k - 1)) != 0) return QG_ERR_UNSUPPORTED;
            if (d.n == 0) continue;
            int rc = check_weights(bits, d.lo, d.hi, d.scale, d.min, d.n, d.k);
            if (rc != QG_OK) return rc;
            if (!d.x || !d.y) return QG_ERR_INVALID_ARG;
            if (!aligned16(d.x) || !aligned16(d.y)) return QG_ERR_ALIGNMENT;
            bool seen = false;
            for (int j = 0; j < i && !seen; ++j) seen = ph[j].n > 0 && ph[j].x == d.x && ph[j].k == d.k;
            if (!seen) in_k += d.k;
            ++*active;
        }
        if (in_k > QG_CHAIN_MAX_PHASE_K) return QG_ERR_UNSUPPORTED;
        for (int i = 0; i < m; ++i) {
            if (ph[i].n == 0) continue;
            const size_t yb = (size_t)ph[i].n * 4;
            for (int j = 0; j < m; ++j) {
                if (ph[j].n == 0) continue;
                if (overlaps(ph[i].y, yb, ph[j].x, (size_t)ph[j].k * 4)) return QG_ERR_INVALID_ARG;
                if (j != i && overlaps(ph[i].y, yb, ph[j].y, (size_t)ph[j].n * 4)) return QG_ERR_INVALID_ARG;
            }
        }
        off += m;
    }
    return QG_OK;
}

size_t qg_chain_workspace_bytes(const qg_gemv_desc* descs, int count, const int* phase_sizes, int n_phases) {
    // 0 for a malformed phase list; descriptors with k out of range add nothing
    if (!descs || !phase_sizes || count <= 0 || count > QG_MAX_GROUP || n_phases < 1 || n_phases > count) return 0;
    long long sum = 0;
    for (int f = 0; f < n_phases; ++f) {
        if (phase_sizes[f] < 1) return 0;
        sum += phase_sizes[f];
    }
    if (sum != count) return 0;
    for (int i = 0; i < count; ++i)
        if (descs[i].k < 1024 || descs[i].k > 16384) return QG_CHAIN_CTL_BYTES;  // the call will refuse it
    return chain_workspace_bytes(descs, count, phase_sizes, n_phases);
}

int qgemv_chain(int bits, const qg_gemv_desc* descs, int count, const int* phase_sizes, int n_phases, void* ws,
                size_t ws_bytes, unsigned flags, void* stream) {
    int active = 0;
    int rc = check_chain(bits, descs, count, phase_sizes, n_phases, &active);
    if (rc != QG_OK || active == 0) return rc;
    if (!ws || ws_bytes < chain_workspace_bytes(descs, count, phase_sizes, n_phases)) return QG_ERR_WORKSPACE;
    if (!aligned16(ws)) return QG_ERR_ALIGNMENT;
    LaunchCtx lc;
    rc = resolve(stream, flags, lc);
    if (rc != QG_OK) return rc;
    return launch_chain(bits, descs, count, phase_sizes, n_phases, reinterpret_cast<unsigned char*>(ws), lc);
}

int qgemv_grouped(int bits, const qg_gemv_desc* descs, int count, void* ws, size_t ws_bytes, unsigned flags,
                  void* stream) {
    int active = 0;
    int rc = check_grouped(bits, descs, count, &active);
    if (rc != QG_OK || active == 0) return rc;
    if (!ws || ws_bytes < grouped_workspace_bytes(descs, count)) return QG_ERR_WORKSPACE;
    if (!aligned16(ws)) return QG_ERR_ALIGNMENT;
    LaunchCtx lc;
    rc = resolve(stream, flags, lc);
    if (rc != QG_OK) return rc;
    return launch_grouped(bits, descs, count, reinterpret_cast<unsigned char*>(ws), lc);
}

int qg_quantize_act(const float* x, int k, int batch, int8_t* xq, float* xs, int32_t* xsum, void* stream) {
    if (k <= 0 || (k & 31) != 0 || k > QG_MAX_K || batch < 1 || batch > QG_MAX_BATCH) return QG_ERR_INVALID_ARG;
    if (!x || !xq || !xs || !xsum) return QG_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq)) return QG_ERR_ALIGNMENT;
    LaunchCtx lc;
    int rc = resolve(stream, 0, lc);
    if (rc != QG_OK) return rc;
    return launch_quantize_act(x, k, batch, xq, xs, xsum, lc);
}

int qg_read_floor(const void* src, size_t bytes, uint32_t* out, unsigned flags, void* stream) {
    if (!src || !out || bytes == 0 || (bytes & 15) != 0) return QG_ERR_INVALID_ARG;
    if (!aligned16(src)) return QG_ERR_ALIGNMENT;
    LaunchCtx lc;
    int rc = resolve(stream, flags, lc);
    if (rc != QG_OK) return rc;
    return launch_read_floor(src, bytes, out, lc);
}

int qg_blockdots(int bits, const uint8_t* lo, const uint8_t* hi, int n, int k, const int8_t* xq, int32_t* dots,
                 void* stream) {
    if (bits != 2 && bits != 4 && bits != 6) return QG_ERR_UNSUPPORTED;
    if (n < 0 || k <= 0 || (k & 31) != 0 || k > QG_MAX_K) return QG_ERR_INVALID_ARG;
    if (n == 0) return QG_OK;
    if (!lo || !xq || !dots || (bits == 6 && !hi) || (bits != 6 && hi)) return QG_ERR_INVALID_ARG;
    if (!aligned16(lo) || (bits == 6 && !aligned16(hi)) || !aligned16(xq)) return QG_ERR_ALIGNMENT;
    LaunchCtx lc;
    int rc = resolve(stream, 0, lc);
    if (rc != QG_OK) return rc;
    return launch_blockdots(bits, lo, hi, n, k, xq, dots, lc);
}

}  // extern "C"
