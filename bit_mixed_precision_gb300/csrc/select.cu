// select_tokens: heavy hitters + recent window (MiniKV review page,
// "Assumptions & free parameters": heavy hitters by cumulative attention,
// chosen once at the end of prefill, plus a recent window; Figure 2
// caption: neither part alone).  One CTA of 1024 threads per unit: a 4-pass
// 8-bit radix select finds the k-th largest score among positions j < T-w,
// then one pass in index order (block scans) keeps every larger score and
// the lowest-position ties, writing positions ascending.
//
// kvq_score_reduce: GQA aggregation of per-query-head column scores
// (MiKV: sum over the group, H2O cumulative attention; DiffKV verdict JSON
// key_machinery: mean attention received, max over the GQA group).
#include "kvq_internal.h"
#include "topk_device.cuh"

namespace kvq {

KVQ_DEFINE_STATUS(select)

namespace {

__global__ void __launch_bounds__(kTopkBlock) select_kernel(const float* __restrict__ score, int T,
                                                           const int32_t* __restrict__ k_hh,
                                                           int kmax, int w,
                                                           int32_t* __restrict__ idx_out,
                                                           int32_t* __restrict__ n_out) {
    __shared__ TopkShared sh;
    const size_t unit = blockIdx.x;
    const float* s = score + unit * (size_t)T;
    int32_t* out = idx_out + unit * (size_t)(kmax + w);
    const int nc = T - w;
    int k = k_hh[unit];
    if (k < 0 || k > kmax) {
        if (threadIdx.x == 0) atomicOr(&g_status_select, kDevCheck);
        k = k < 0 ? 0 : kmax;
    }
    if (k > nc) k = nc;
    if (k > 0) {
        uint32_t kstar, take_eq;
        block_radix_select([&](int i) { return orderable(s[i]); }, nc, k, sh, &kstar, &take_eq);
        uint32_t eq_base = 0, out_base = 0;
        for (int c0 = 0; c0 < nc; c0 += blockDim.x) {
            const int j = c0 + threadIdx.x;
            uint32_t kv = j < nc ? orderable(s[j]) : 0u;
            const uint32_t gt = (j < nc && kv > kstar) ? 1u : 0u;
            const uint32_t eq = (j < nc && kv == kstar) ? 1u : 0u;
            uint32_t eq_tot;
            const uint32_t eq_rank = block_excl_scan(eq, sh, &eq_tot);
            const uint32_t sel = gt | (eq & (eq_base + eq_rank < take_eq ? 1u : 0u));
            uint32_t sel_tot;
            const uint32_t pos = block_excl_scan(sel, sh, &sel_tot);
            if (sel) out[out_base + pos] = j;
            eq_base += eq_tot;
            out_base += sel_tot;
        }
    }
    for (int i = threadIdx.x; i < w; i += blockDim.x) out[k + i] = nc + i;
    if (threadIdx.x == 0) n_out[unit] = k + w;
}

__global__ void score_reduce_kernel(const float* __restrict__ cs, int B, int Hq, int Hkv, int T,
                                    int mode, float* __restrict__ out) {
    const int g = Hq / Hkv;
    const size_t total = (size_t)B * Hkv * T;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int j = (int)(idx % T);
        const size_t u = idx / T;
        const int b = (int)(u / Hkv), h = (int)(u % Hkv);
        const float* base = cs + (((size_t)b * Hq + (size_t)h * g) * T) + j;
        float acc;
        if (mode == 0) {
            acc = 0.0f;
            for (int i = 0; i < g; ++i) acc = __fadd_rn(acc, base[(size_t)i * T]);
        } else {
            const float cnt = (float)(T - j);
            acc = __fdiv_rn(base[0], cnt);
            for (int i = 1; i < g; ++i) acc = fmaxf(acc, __fdiv_rn(base[(size_t)i * T], cnt));
        }
        out[idx] = acc;
    }
}

}  // namespace

cudaError_t launch_select(const float* score, int units, int T, const int32_t* k_hh, int kmax,
                          int w, int32_t* idx_out, int32_t* n_out, cudaStream_t s) {
    if (units == 0) return cudaSuccess;
    select_kernel<<<units, kTopkBlock, 0, s>>>(score, T, k_hh, kmax, w, idx_out, n_out);
    return cudaGetLastError();
}

cudaError_t launch_score_reduce(const float* cs, int B, int Hq, int Hkv, int T, int mode,
                                float* out, cudaStream_t s) {
    size_t total = (size_t)B * Hkv * T;
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;
    score_reduce_kernel<<<(unsigned)blocks, 256, 0, s>>>(cs, B, Hq, Hkv, T, mode, out);
    return cudaGetLastError();
}

}  // namespace kvq
