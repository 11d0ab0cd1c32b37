// Constrained token selection over a logit vector.
//
// needle.js "Inference backends", "Resident layers": tool calling uploads an
// ascending list of grammar-allowed token IDs and reads back only the selected ID
// and its full-vocabulary log probability.  Here one pass over the logits does both
// halves: every CTA folds its share of the logits into an online log-sum-exp
// (running max m and sum of exp(l - m)) and its share of the allowed IDs into a
// (value, lowest ID) best; the last CTA to finish merges all partials, writes the
// selected ID and l[id] - logsumexp(l), and re-arms the counter.  No CTA waits on
// another.
#include "qg_internal.h"

namespace qg {

__global__ void __launch_bounds__(256) select_kernel(const float* __restrict__ logits, int n,
                                                     const int32_t* __restrict__ allowed, int n_allowed,
                                                     int32_t* token, float* logprob, SelectWorkspace* ws) {
    __shared__ SelectPartial sred[8];
    __shared__ int last;
    pdl_wait();  // the logits come from the preceding kernel
    if (threadIdx.x == 0) pdl_launch_dependents();

    // log-sum-exp over this CTA's rows (NaN skipped)
    const long long r0 = (long long)blockIdx.x * n / gridDim.x, r1 = (long long)(blockIdx.x + 1) * n / gridDim.x;
    float m = -INFINITY, s = 0.0f;
    // four logits per step: their max first, then four independent exponentials
    for (long long i0 = r0 + threadIdx.x; i0 < r1; i0 += 4 * (long long)blockDim.x) {
        float v[4];
        float cm = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const long long i = i0 + (long long)q * blockDim.x;
            v[q] = i < r1 ? logits[i] : __int_as_float(0x7fc00000);
            if (v[q] == v[q]) cm = fmaxf(cm, v[q]);
        }
        if (cm == -INFINITY) continue;  // only NaN and -inf: no term
        if (cm == INFINITY) {
            lse_merge(m, s, INFINITY, 1.0f);
            continue;
        }
        float cs = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (v[q] == v[q]) cs += expf(v[q] - cm);
        lse_merge(m, s, cm, cs);
    }
    // best allowed (value, lowest id) over this CTA's share of the allowed list
    float bv = __int_as_float(0x7fc00000);
    int bi = 0x7fffffff;
    const long long cnt = allowed ? n_allowed : n;
    const long long a0 = (long long)blockIdx.x * cnt / gridDim.x, a1 = (long long)(blockIdx.x + 1) * cnt / gridDim.x;
    for (long long j = a0 + threadIdx.x; j < a1; j += blockDim.x) {
        const long long id = allowed ? (long long)allowed[j] : j;
        if (id < 0 || id >= n) continue;
        const float v = logits[id];
        if (better(v, (int)id, bv, bi)) {
            bv = v;
            bi = (int)id;
        }
    }
    select_finish(m, s, bv, bi, ws, token, logprob, sred, &last);
}

int launch_select(const float* logits, int n, const int32_t* allowed, int n_allowed, int32_t* token, float* logprob,
                  SelectWorkspace* ws, const LaunchCtx& lc) {
    long long grid = ((long long)n + 1023) / 1024;
    if (grid > 2LL * lc.sm_count) grid = 2LL * lc.sm_count;
    if (grid > SELECT_MAX_CTAS) grid = SELECT_MAX_CTAS;
    if (grid < 1) grid = 1;
    return launch_kernel(select_kernel, dim3((unsigned)grid), dim3(256), 0, lc, logits, n, allowed, n_allowed, token,
                         logprob, ws);
}

}  // namespace qg
