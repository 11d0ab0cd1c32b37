/*
 * qgemv.h - C ABI of the quantized-weight GEMV library for NVIDIA GB300 (sm_103a).
 *
 * The library computes the decode-time matrix-vector product against
 * block-quantised weights: y = W_deq x with the activation x quantised to int8
 * per block of 32 and the weights stored as 4-bit or 6-bit codes with an fp16
 * scale and min per block of 32 (w = scale * code + min), or as 2-bit codes with
 * an fp16 scale and zero point 2 (w = scale * (code - 2)).  Its neighbours are a
 * small-batch variant, a Walsh-Hadamard + codebook (CQ) matvec, a vocabulary
 * projection finished with logit soft-capping and argmax, constrained token
 * selection, a grouped multi-matrix dispatch and a dependent GEMV chain.
 *
 * Conventions for every call:
 *  - Pointers named as device buffers are CUDA device pointers owned by the
 *    caller; the library keeps no reference to them after the call returns.
 *  - Calls are asynchronous: arguments are validated on the host, the work is
 *    enqueued on `stream` (a cudaStream_t passed as void*; NULL is the legacy
 *    default stream) and the call returns without synchronising.  The stream and
 *    every buffer belong to the current device (cudaGetDevice), whose properties
 *    and device-side words the call uses.
 *  - A negative return value is an error; nothing was enqueued and no output
 *    was touched.  QG_ERR_CUDA reports a launch failure seen right after the
 *    launch; faults raised while a kernel runs surface at the caller's next
 *    synchronisation, like any CUDA error.
 *  - The library allocates no device memory.  Calls are thread-safe.
 *
 * Weight layout (blocks of 32 consecutive weights along K; rows row-major):
 *  Q4  codes  uint8 [n][k/2]: byte 16*b + j of a row holds code 32*b + j in
 *             bits 0-3 and code 32*b + j + 16 in bits 4-7.
 *  Q6  lo     uint8 [n][k/2]: the low 4 bits of each code, in the Q4 order;
 *      hi     uint8 [n][k/4]: 8 bytes per block, byte 8*b + t holding the top
 *             2 bits of codes 32*b + t, +8, +16, +24 in bits 0-1, 2-3, 4-5, 6-7.
 *  scale, min binary16 (as uint16 bits) [n][k/32]; weight = scale*code + min.
 *  Q2  codes  uint8 [n][k/4]: 8 bytes per block, byte 8*b + t holding the 2-bit codes
 *             32*b + t, +8, +16, +24 in bits 0-1, 2-3, 4-5, 6-7; scale binary16
 *             [n][k/32]; no min plane: weight = scale*(code - 2) (the int2 weights with
 *             zero point 2 of the Gemma WebGPU Engine, "Roadmap").  Where a call takes
 *             bits = 2, `lo` is the code plane and `hi` and `min` are NULL.
 *  CQ  idx    uint8 [n][k/2]: index 2j in bits 0-3 of byte j, 2j+1 in bits 4-7;
 *      codebook binary16 [16]; row_scale binary16 [n].
 * Packed planes, x and y must start on 16-byte boundaries.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum qg_status {
    QG_OK = 0,
    QG_ERR_INVALID_ARG = -1, /* null pointer, size out of range, k not a multiple of 32, ... */
    QG_ERR_ALIGNMENT = -2,   /* a buffer that must start on a 16-byte boundary does not */
    QG_ERR_UNSUPPORTED = -3, /* bits not supported by the call, group size not supported, shape too large */
    QG_ERR_WORKSPACE = -4,   /* workspace missing or smaller than the reported size */
    QG_ERR_CUDA = -5         /* the CUDA launch itself failed */
};

/* Launch flags (bitwise OR; 0 = defaults). */
#define QG_FLAG_PDL 0x1u    /* programmatic dependent launch: the kernel may start, and      \
                               begin streaming WEIGHTS, before the preceding work on the     \
                               stream has finished; it waits for that work before reading x, \
                               writing any output or touching the workspace.  The caller     \
                               guarantees that no preceding work writes the weights.         */
#define QG_FLAG_PLAIN 0x2u  /* force the plain-load kernel (128-bit loads, no bulk-copy ring) */
#define QG_FLAG_CHAIN_PERSISTENT 0x4u /* qgemv_chain: one persistent cooperative launch for all  \
                                         phases instead of per-phase launches                     */

/* Largest supported sizes. */
#define QG_MAX_K 65536       /* qgemv_q4/q6 and vocab: k <= QG_MAX_K */
#define QG_MAX_BATCH 16      /* qgemv_batched: 1 <= batch <= 16 */
#define QG_MAX_CQ_K 16384    /* cq_fwht_matvec: k <= QG_MAX_CQ_K */

/* Human-readable text of a status code (static storage). */
const char* qg_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int qg_version(void);

/*
 * Device-side error word.  Kernels that wait on an mbarrier or on the other CTAs
 * give up after a bounded time and record a nonzero code here instead of hanging:
 * 1 a weight tile never landed, 2 a ring slot was never freed (qgemv_chain's
 * producer), 4 a copy in flight never landed while stopping, 8 a grid-wide barrier
 * of qgemv_chain ran out, 16 a CTA of qgemv_chain's persistent kernel stopped at a
 * phase boundary because the chain's abort word was set (by a CTA whose wait ran
 * out, or before the call).  Reads and clears the word of the current device;
 * synchronises the device.
 * Returns QG_OK or QG_ERR_CUDA; *code receives the word (0 = no error).
 */
int qg_device_error(uint32_t* code);

/*
 * qgemv_q4: y[r] = sum_i (scale*code(r,i) + min) * x_deq(i),  r < n.
 * x_deq is x quantised per block of 32: s_b = max|x| / 127 (fp32),
 * xq = clamp(rint(x / s_b), -127, 127), x_deq = s_b * xq.  The integer block
 * dots sum(code * xq) are exact; the block combine and row sum are fp32.
 * Dequant-fused GEMV over int8 dp4a block dots (genie-ai-runtime v1.1 -> v1.3.1,
 * "The decode arc": dp4a int8 MMVQ; oxinfer README, "How it works": per-matmul
 * activation quantisation and int8 block dots).
 *   codes, scale, min : device, Q4 layout above, n x k
 *   n >= 0, k > 0, k % 32 == 0, k <= QG_MAX_K
 *   x : device fp32 [k];  y : device fp32 [n] (written)
 * n == 0 enqueues nothing and returns QG_OK.
 */
int qgemv_q4(const uint8_t* codes, const uint16_t* scale, const uint16_t* min, int n, int k, const float* x,
             float* y, unsigned flags, void* stream);

/* qgemv_q6: as qgemv_q4 with 6-bit codes (lo, hi planes). */
/* qgemv_q2: as qgemv_q4 with 2-bit codes (Q2 layout), w = scale*(code - 2). */
int qgemv_q2(const uint8_t* codes, const uint16_t* scale, int n, int k, const float* x, float* y, unsigned flags,
             void* stream);
int qgemv_q6(const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min, int n, int k,
             const float* x, float* y, unsigned flags, void* stream);

/*
 * qgemv_batched: Y[c][r] = GEMV of column c, for c < batch: every activation
 * column X[c] (fp32 [k], contiguous rows of X [batch][k]) is quantised on its
 * own and all columns share one pass over the weights (the multi-token int8
 * kernels of the oxinfer README, "Speculative decoding" and "How it works").
 *   bits : 2 (hi and min NULL), 4 (hi NULL) or 6
 *   1 <= batch <= QG_MAX_BATCH;  batch * k <= 131072
 *   X : device fp32 [batch][k];  Y : device fp32 [batch][n] (written)
 * For batch >= 8 with 4-bit weights and k in {512, 1024, 2048} the integer
 * block dots run on tensor cores (mma.sync, f16 operands, exact).  That path quantises
 * the activations once into `ws` (at least qg_batched_workspace_bytes(bits, k, batch)
 * bytes of device memory, 16-byte aligned, no initial content; 0 bytes are needed for
 * the other shapes) and chains the GEMV launch to it by programmatic dependent
 * launch; with ws == NULL every CTA quantises the activations itself (slower).
 * Calls that share a workspace must not overlap on the GPU.
 */
size_t qg_batched_workspace_bytes(int bits, int k, int batch);
int qgemv_batched(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min, int n,
                  int k, int batch, const float* X, float* Y, void* ws, size_t ws_bytes, unsigned flags,
                  void* stream);

/*
 * cq_fwht_matvec: selected-row codebook matvec in the Hadamard domain
 * (needle.js "Inference backends": "Pure TypeScript" and "TypeGPU" for the
 * normalised fast Walsh-Hadamard transform of each activation group followed by
 * packed codebook-index decode inside the dot; "Custom backend" for the
 * optional row range).
 *   u = (1/sqrt(group)) * H_group x, independently for each group of `group`
 *       consecutive values (H in natural / Sylvester order);
 *   y[j] = row_scale[r] * sum_i codebook[idx(r, i)] * u[i],  r = row_start + j.
 *   idx : device [n][k/2];  codebook : device binary16 [16];  row_scale : device binary16 [n]
 *   group in {128, 256, 512, 1024};  k % group == 0;  k <= QG_MAX_CQ_K
 *   0 <= row_start, 0 <= row_count, row_start + row_count <= n
 *   x : device fp32 [k];  y : device fp32 [row_count] (written)
 */
int cq_fwht_matvec(const uint8_t* idx, const uint16_t* codebook, const uint16_t* row_scale, int n, int k, int group,
                   int row_start, int row_count, const float* x, float* y, unsigned flags, void* stream);

/*
 * Workspace bytes that vocab_softcap_argmax needs (a small, fixed amount).
 * The workspace is device memory owned by the caller; it must be zero-filled
 * once after allocation, and every completed call leaves it zeroed again.
 * Calls that share one workspace must not overlap in time on the GPU.
 */
size_t qg_vocab_workspace_bytes(void);

/*
 * vocab_softcap_argmax: z = the GEMV of qgemv_q4/q6 over n_vocab rows, then
 * logits l = softcap * tanh(z / softcap) (final-logit soft-capping of
 * genie-ai-runtime, "What Gemma 4 E2B actually is"; softcap <= 0 leaves z
 * as is), and the index of the largest logit, the lowest index among equal
 * maxima and NaN never winning (the deterministic argmax of the Gemma WebGPU
 * Engine, "Roadmap").
 *   bits : 2, 4 or 6 (the pages' LM head is int2);  logits : device fp32 [n_vocab] or NULL;
 *   argmax : device int32 [1] (written);  ws : see qg_vocab_workspace_bytes.
 *   1 <= n_vocab
 */
int vocab_softcap_argmax(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min,
                         int n_vocab, int k, const float* x, float softcap, float* logits, int32_t* argmax, void* ws,
                         size_t ws_bytes, unsigned flags, void* stream);

/*
 * Constrained selection over the vocabulary (needle.js "Inference backends",
 * "Resident layers": the host uploads the grammar-allowed token IDs and reads back
 * only the selected ID and its full-vocabulary log probability; the allowed-token
 * argmax and log-softmax of its "selection" pass).
 * qg_logits_select: over logits l[n] (device fp32),
 *   token   = the allowed ID of the largest logit, the lowest ID among equal maxima,
 *             NaN never selected; -1 if no allowed ID qualifies;
 *   logprob = l[token] - log(sum_i exp(l[i])) over ALL n logits (NaN skipped; a
 *             +inf logit makes the log-sum-exp +inf); NaN when token is -1.
 *   allowed : device int32 [n_allowed] token IDs in any order (ascending as the page
 *             has it; duplicates and IDs outside [0, n) are ignored), or NULL for all.
 *   token : device int32 [1];  logprob : device fp32 [1] (written).
 *   ws : device workspace of qg_select_workspace_bytes() bytes, zero-filled once after
 *        allocation; every completed call leaves it zeroed.  Calls sharing a workspace
 *        must not overlap on the GPU.
 * vocab_softcap_select: vocab_softcap_argmax's soft-capped logits (written to `logits`,
 * required here) and qg_logits_select's token and logprob over them; ws holds
 * qg_vocab_select_workspace_bytes().  When allowed is NULL or holds at most
 * QG_SELECT_FUSED_MAX_ALLOWED IDs and k has the streaming kernel (not QG_FLAG_PLAIN),
 * one launch does both: each CTA folds the rows it has just produced into the
 * selection and the last CTA to finish merges; otherwise two launches, the second
 * chained to the first by programmatic dependent launch.  The token is the same either
 * way; the log-probability differs only by summation order.
 */
#define QG_SELECT_FUSED_MAX_ALLOWED 8192
size_t qg_select_workspace_bytes(void);
int qg_logits_select(const float* logits, int n, const int32_t* allowed, int n_allowed, int32_t* token,
                     float* logprob, void* ws, size_t ws_bytes, unsigned flags, void* stream);
size_t qg_vocab_select_workspace_bytes(void);
int vocab_softcap_select(int bits, const uint8_t* lo, const uint8_t* hi, const uint16_t* scale, const uint16_t* min,
                         int n_vocab, int k, const float* x, float softcap, const int32_t* allowed, int n_allowed,
                         float* logits, int32_t* token, float* logprob, void* ws, size_t ws_bytes, unsigned flags,
                         void* stream);

/*
 * Grouped GEMV: `count` independent GEMVs of one weight format in two launches
 * (needle.js "Inference backends", "Hybrid GPU execution": independent projections
 * batched into one dispatch over a combined weight arena; genie-ai-runtime,
 * "v1.2.0": a QKV GEMV sharing one q8_1 activation).  Each descriptor computes
 * y = GEMV(weights, x) exactly as qgemv_q4/qgemv_q6 define it.
 *   descs : HOST array of `count` descriptors, read during the call only (they are
 *           copied into the kernel parameters); the pointers inside are device
 *           pointers; hi is NULL for bits == 4.
 *   0 <= count <= QG_MAX_GROUP; for every descriptor n >= 0 and k a power of two
 *           with 1024 <= k <= 16384.  Descriptors may share x; outputs must not overlap.
 *   ws    : device workspace of at least qg_grouped_workspace_bytes(descs, count)
 *           bytes (the quantised activations), 16-byte aligned, no initial content.
 * The second launch is always chained to the first by programmatic dependent
 * launch; QG_FLAG_PDL applies to the first.
 */
typedef struct qg_gemv_desc {
    const uint8_t* lo;     /* Q4 codes, or the Q6 low planes */
    const uint8_t* hi;     /* Q6 high planes; NULL for Q4 */
    const uint16_t* scale; /* binary16 [n][k/32] */
    const uint16_t* min;   /* binary16 [n][k/32] */
    const float* x;        /* [k] */
    float* y;              /* [n] */
    int n;
    int k;
} qg_gemv_desc;

#define QG_MAX_GROUP 256

size_t qg_grouped_workspace_bytes(const qg_gemv_desc* descs, int count);
int qgemv_grouped(int bits, const qg_gemv_desc* descs, int count, void* ws, size_t ws_bytes, unsigned flags,
                  void* stream);

/*
 * qgemv_grouped_noalloc: qgemv_grouped without a caller workspace.  This entry point
 * has no counterpart in the pages the library follows; it exists for callers that
 * cannot allocate device memory - code running where the CUDA allocator must not be
 * called (a host callback, a decode loop that forbids allocation), plug-ins whose
 * host application owns all device memory, or C callers without an allocator.
 * The quantised activations go to a fixed QG_NOALLOC_WS_BYTES device array inside
 * the library, which every GPU that loads the library holds until the process exits.
 *   Same arguments and results as qgemv_grouped, minus ws/ws_bytes.  A group whose
 *   activations need more than QG_NOALLOC_WS_BYTES (see qg_grouped_workspace_bytes)
 *   is rejected with QG_ERR_WORKSPACE and nothing is launched.
 *   The first call on a device looks up the array's device address (once per device,
 *   with that device current); make that first call before any stream capture.
 *   All calls share the array: calls whose work may overlap on the GPU race on it
 *   and must be ordered by the caller.  It keeps the last call's contents; nothing
 *   in it needs to start at zero.  The call allocates nothing.
 */
#define QG_NOALLOC_WS_BYTES (2u << 20)
int qgemv_grouped_noalloc(int bits, const qg_gemv_desc* descs, int count, unsigned flags, void* stream);

/*
 * qgemv_chain: dependent GEMVs in decode order.  The `count` descriptors form
 * `n_phases` phases, phase f being the next phase_sizes[f] of them.  A GEMV may read
 * (x) any vector written by an earlier phase or present before the call; the GEMVs
 * of one phase are independent of each other.  Each descriptor computes
 * y = GEMV(weights, x) exactly as qgemv_q4/qgemv_q6 define it, on x as the earlier
 * phases left it.  (Gemma WebGPU Engine, "Roadmap": a layer's ordered dispatches,
 * each projection reading the buffer the previous one wrote; genie-ai-runtime, "The
 * decode arc": the activation is quantised per matmul.)
 *   bits  : 4 (hi NULL) or 6
 *   descs : HOST array of `count` descriptors, read during the call only; n >= 0 and
 *           k a power of two with 1024 <= k <= 16384, as for qgemv_grouped
 *   phase_sizes : HOST int [n_phases], every entry >= 1, summing to count
 *   1 <= n_phases <= count <= QG_MAX_GROUP
 *   Within one phase no output may overlap another output or any input of that
 *   phase, and the distinct inputs (by x and k) total at most QG_CHAIN_MAX_PHASE_K
 *   values.  Across phases buffers may be reused freely.
 *   ws : device workspace of at least qg_chain_workspace_bytes(...) bytes, 16-byte
 *        aligned; its first QG_CHAIN_CTL_BYTES bytes are zero-filled once after
 *        allocation and every call that completes leaves them zero.  Calls sharing a
 *        workspace must not overlap on the GPU.
 * Default: each phase runs as qgemv_grouped's launches, phase f+1 chained to phase f
 * by programmatic dependent launch (QG_FLAG_PDL applies to the first phase); a phase
 * whose distinct inputs are short (6144 values in all) is one launch whose CTAs
 * quantise the inputs themselves, and a phase whose long inputs are all whole outputs
 * of the phase before (x == that y, k == its n) is one launch too: each CTA of the
 * phase before, its rows of such an output aligned to whole blocks of 32, quantises
 * them into the workspace once they are stored.  With QG_FLAG_CHAIN_PERSISTENT: one cooperative
 * launch, one CTA per SM, whose producer warp streams every phase's weights through
 * a bulk-copy ring that runs ahead across phase boundaries, with a grid-wide barrier
 * between phases.  That launch starts after the preceding work on the stream has
 * finished (QG_FLAG_PDL does not apply to it).  A barrier wait gives up after 1 s: the
 * kernel then records a code in the device error word and stops; the outputs are
 * undefined.
 */
#define QG_CHAIN_CTL_BYTES 256
#define QG_CHAIN_MAX_PHASE_K 32768
size_t qg_chain_workspace_bytes(const qg_gemv_desc* descs, int count, const int* phase_sizes, int n_phases);
int qgemv_chain(int bits, const qg_gemv_desc* descs, int count, const int* phase_sizes, int n_phases, void* ws,
                size_t ws_bytes, unsigned flags, void* stream);

/*
 * Exposed steps, for exactness checks of the integer parts.
 * qg_quantize_act: per-block int8 quantisation of `batch` rows of x [batch][k]:
 *   xq int8 [batch][k], xs fp32 [batch][k/32] (s_b), xsum int32 [batch][k/32] (sum of xq).
 * qg_blockdots: D[r][b] = sum_{i<32} code(r, 32b+i) * xq(32b+i), int32 [n][k/32].
 * Same size rules as qgemv_q4; all pointers device.
 */
int qg_quantize_act(const float* x, int k, int batch, int8_t* xq, float* xs, int32_t* xsum, void* stream);
int qg_blockdots(int bits, const uint8_t* lo, const uint8_t* hi, int n, int k, const int8_t* xq, int32_t* dots,
                 void* stream);

/*
 * qg_read_floor: a measurement hook, not part of the method.  Reads every byte of
 * src[0, bytes) once (16-byte streaming loads) and XORs the 32-bit words into *out.
 * The time of this call is the floor of any kernel that streams the same bytes in the
 * same launch setting, which is what the GEMVs' weight streams are compared with
 * (the decode bound of the oxinfer README, "Performance": every weight byte is read
 * once per token).  The reads may start before the preceding work finishes under
 * QG_FLAG_PDL; *out is updated after it.
 *   src : device, 16-byte aligned;  bytes > 0, bytes % 16 == 0;  out : device uint32 [1]
 */
int qg_read_floor(const void* src, size_t bytes, uint32_t* out, unsigned flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
