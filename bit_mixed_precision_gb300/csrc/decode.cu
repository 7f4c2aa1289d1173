// decode_attn_qkv: one decode step of attention over the compressed cache,
// dequantising packed codes inside the kernel (MiKV rebuttal, the INTn x
// FP16 GEMV paragraph: on-the-fly dequantisation; MiniKV verdict JSON
// forward_implications: fused dequantisation kernels during decoding).
//
// One launch per step.  Grid = (token chunks of every tier and of the
// residual ring, units).  Each CTA computes, for the g query heads that
// share its KV head, the base-2 logits of its chunk, the chunk max / sum
// and the unnormalised P.V partial, and writes them to the workspace.  The
// last CTA of a unit (atomic counter) merges the partials, writes o and
// lse, adds this step's attention to the policy scores (DiffKV: per ring
// slot and query head; MiKV: per token, summed over the group) and
// advances the residual length; the last CTA of the grid advances seq_len.
// The tiers are read where they lie (MiKV rebuttal: attention is
// permutation invariant, so each precision group sits in its own region).
#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "pack_device.cuh"

namespace kvq {

KVQ_DEFINE_STATUS(decode)

namespace {

constexpr int kChunk = 256;     // tokens per CTA
constexpr int kThreads = 256;
constexpr int kMaxG = 8;        // query heads per KV head
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct TierArgs {
    int k_bits, v_bits, k_axis, cap;
    const uint32_t* k_codes;
    const uint16_t* k_scale;
    const uint16_t* k_zero;
    const uint32_t* v_codes;
    const uint16_t* v_scale;
    const uint16_t* v_zero;
    const int32_t* token_id;
    const int32_t* count;
    int chunks;                 // ceil(cap / kChunk)
    int slot_base;              // offset of this tier in the logits row
};

struct DecodeArgs {
    const void* q;
    const void* k_new;
    const void* v_new;
    void* o;
    float* lse_out;
    int B, Hq, Hkv, D, G, g, n_tiers, policy, bf16;
    TierArgs tier[KVQ_MAX_TIERS];
    void* res_k;
    void* res_v;
    int32_t* res_token_id;
    const int32_t* res_start;
    int32_t* res_len;
    int res_cap, res_chunks, res_slot_base;
    int32_t* seq_len;
    float* win_acc;
    float* cum_score;
    int score_cap;
    float scale_log2;
    int total_chunks;           // per unit
    int slots;                  // logits row length per (unit, head)
    float* part;                // [unit][g][total_chunks][D + 2]
    float* logits;              // [unit][g][slots] or null
    uint32_t* counters;         // [units + 1]
};

__device__ __forceinline__ float ldf(const void* p, size_t i, bool bf16) {
    return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i])
                : __half2float(reinterpret_cast<const __half*>(p)[i]);
}

__device__ __forceinline__ void stf(void* p, size_t i, float v, bool bf16) {
    if (bf16)
        reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
}

// Dequantised key element (token slot j, channel c) of a tier.
template <int KB, int KAX>
__device__ __forceinline__ float key_at(const TierArgs& t, size_t unit, int j, int c, int D, int G) {
    if (KAX == KVQ_AXIS_CHANNEL) {
        constexpr int per = 32 / KB;
        const uint32_t w = t.k_codes[(unit * (size_t)(t.cap / per) + j / per) * D + c];
        const uint32_t q = (w >> (KB * (j % per))) & ((1u << KB) - 1u);
        const size_t si = (unit * (size_t)(t.cap / G) + j / G) * D + c;
        return fmaf((float)q, h2f_bits(t.k_scale[si]), h2f_bits(t.k_zero[si]));
    } else {
        const uint32_t* row = t.k_codes + (unit * t.cap + j) * (size_t)(D * KB / 32);
        const uint32_t q = code_at(row, c, KB);
        const size_t si = (unit * t.cap + j) * (size_t)(D / G) + c / G;
        return fmaf((float)q, h2f_bits(t.k_scale[si]), h2f_bits(t.k_zero[si]));
    }
}

template <int VB>
__device__ __forceinline__ float value_at(const TierArgs& t, size_t unit, int j, int c, int D, int G) {
    const uint32_t* row = t.v_codes + (unit * t.cap + j) * (size_t)(D * VB / 32);
    const uint32_t q = code_at(row, c, VB);
    const size_t si = (unit * t.cap + j) * (size_t)(D / G) + c / G;
    return fmaf((float)q, h2f_bits(t.v_scale[si]), h2f_bits(t.v_zero[si]));
}

struct Smem {
    float q[kMaxG][128];
    float lg[kMaxG][kChunk];
    float red[kMaxG][kThreads / 32];
    float m[kMaxG];
    float opart[4][kMaxG][128];
    int last;
};

// Logits and P.V of one chunk of n tokens.  KeyFn(i, c) / ValFn(i, c) give
// the dequantised (or full-precision) element of chunk token i.
template <typename KeyFn, typename ValFn>
__device__ void chunk_attend(const DecodeArgs& a, Smem& sm, int n, KeyFn key, ValFn val,
                             float* part_out /* [g][total_chunks][D+2] at this chunk */,
                             float* lg_out /* [g][slots] at this chunk's first slot, or null */) {
    const int D = a.D, g = a.g;
    // phase 1: logits (base-2 units), one token per thread
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        float acc[kMaxG];
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) acc[h] = 0.0f;
        for (int c = 0; c < D; ++c) {
            const float x = key(i, c);
#pragma unroll
            for (int h = 0; h < kMaxG; ++h)
                if (h < g) acc[h] = fmaf(sm.q[h][c], x, acc[h]);
        }
#pragma unroll
        for (int h = 0; h < kMaxG; ++h)
            if (h < g) sm.lg[h][i] = acc[h];
    }
    __syncthreads();
    // phase 2: chunk max per head
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = 0; h < g; ++h) {
        float mx = -__int_as_float(0x7f800000);
        for (int i = threadIdx.x; i < n; i += blockDim.x) mx = fmaxf(mx, sm.lg[h][i]);
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) sm.red[h][warp] = mx;
    }
    __syncthreads();
    if (threadIdx.x < g) {
        float mx = -__int_as_float(0x7f800000);
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, sm.red[threadIdx.x][w]);
        sm.m[threadIdx.x] = mx;
    }
    __syncthreads();
    // logits out (for score accumulation), then p in place
    for (int h = 0; h < g; ++h)
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const float s = sm.lg[h][i];
            if (lg_out) lg_out[(size_t)h * a.slots + i] = s;
            sm.lg[h][i] = ex2_approx(s - sm.m[h]);
        }
    __syncthreads();
    // phase 3: P.V, channel c per thread, tokens split over blockDim / D groups
    const int nsplit = blockDim.x / D;
    const int c = threadIdx.x % D, sp = threadIdx.x / D;
    if (sp < nsplit && sp < 4) {
        float ov[kMaxG];
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) ov[h] = 0.0f;
        for (int i = sp; i < n; i += nsplit) {
            const float x = val(i, c);
#pragma unroll
            for (int h = 0; h < kMaxG; ++h)
                if (h < g) ov[h] = fmaf(sm.lg[h][i], x, ov[h]);
        }
#pragma unroll
        for (int h = 0; h < kMaxG; ++h)
            if (h < g) sm.opart[sp][h][c] = ov[h];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < g * D; idx += blockDim.x) {
        const int h = idx / D, cc = idx % D;
        float s = 0.0f;
        for (int k = 0; k < nsplit && k < 4; ++k) s += sm.opart[k][h][cc];
        part_out[(size_t)h * a.total_chunks * (D + 2) + 2 + cc] = s;
    }
    // row sums
    for (int h = 0; h < g; ++h) {
        float l = 0.0f;
        for (int i = threadIdx.x; i < n; i += blockDim.x) l += sm.lg[h][i];
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) sm.red[h][warp] = l;
    }
    __syncthreads();
    if (threadIdx.x < g) {
        float l = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) l += sm.red[threadIdx.x][w];
        float* po = part_out + (size_t)threadIdx.x * a.total_chunks * (D + 2);
        po[0] = sm.m[threadIdx.x];
        po[1] = l;
    }
}

template <int KB, int KAX, int VB>
__device__ void tier_chunk(const DecodeArgs& a, Smem& sm, const TierArgs& t, size_t unit, int chunk,
                           float* part_out, float* lg_out) {
    const int cnt = min(t.count[unit], t.cap);
    const int j0 = chunk * kChunk;
    const int n = min(kChunk, cnt - j0);
    const int D = a.D, G = a.G;
    auto key = [&](int i, int c) { return key_at<KB, KAX>(t, unit, j0 + i, c, D, G); };
    auto val = [&](int i, int c) { return value_at<VB>(t, unit, j0 + i, c, D, G); };
    chunk_attend(a, sm, n, key, val, part_out, lg_out ? lg_out + j0 : nullptr);
}

__device__ void dispatch_tier(const DecodeArgs& a, Smem& sm, const TierArgs& t, size_t unit,
                              int chunk, float* part_out, float* lg_out) {
    const int kb = t.k_bits, vb = t.v_bits, ax = t.k_axis;
    if (ax == KVQ_AXIS_CHANNEL && kb == 2 && vb == 2)
        tier_chunk<2, KVQ_AXIS_CHANNEL, 2>(a, sm, t, unit, chunk, part_out, lg_out);
    else if (ax == KVQ_AXIS_CHANNEL && kb == 4 && vb == 4)
        tier_chunk<4, KVQ_AXIS_CHANNEL, 4>(a, sm, t, unit, chunk, part_out, lg_out);
    else if (ax == KVQ_AXIS_TOKEN && kb == 8 && vb == 4)
        tier_chunk<8, KVQ_AXIS_TOKEN, 4>(a, sm, t, unit, chunk, part_out, lg_out);
    else if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 2)
        tier_chunk<4, KVQ_AXIS_TOKEN, 2>(a, sm, t, unit, chunk, part_out, lg_out);
    else if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 4)
        tier_chunk<4, KVQ_AXIS_TOKEN, 4>(a, sm, t, unit, chunk, part_out, lg_out);
    else if (ax == KVQ_AXIS_TOKEN && kb == 2 && vb == 2)
        tier_chunk<2, KVQ_AXIS_TOKEN, 2>(a, sm, t, unit, chunk, part_out, lg_out);
    else if (ax == KVQ_AXIS_TOKEN && kb == 2 && vb == 4)
        tier_chunk<2, KVQ_AXIS_TOKEN, 4>(a, sm, t, unit, chunk, part_out, lg_out);
    else if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 8)
        tier_chunk<4, KVQ_AXIS_TOKEN, 8>(a, sm, t, unit, chunk, part_out, lg_out);
    else if (ax == KVQ_AXIS_TOKEN && kb == 8 && vb == 8)
        tier_chunk<8, KVQ_AXIS_TOKEN, 8>(a, sm, t, unit, chunk, part_out, lg_out);
    else if (ax == KVQ_AXIS_CHANNEL && kb == 8 && vb == 8)
        tier_chunk<8, KVQ_AXIS_CHANNEL, 8>(a, sm, t, unit, chunk, part_out, lg_out);
}

__device__ void empty_partial(const DecodeArgs& a, float* part_out) {
    if (threadIdx.x < a.g) {
        float* po = part_out + (size_t)threadIdx.x * a.total_chunks * (a.D + 2);
        po[0] = -__int_as_float(0x7f800000);
        po[1] = 0.0f;
    }
}

__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const size_t unit = blockIdx.y;
    const int units = gridDim.y;
    const int b = (int)(unit / a.Hkv), hkv = (int)(unit % a.Hkv);
    const int D = a.D, g = a.g;
    const bool bf = a.bf16 != 0;

    // query rows of the group, pre-scaled to base-2 logits
    for (int idx = threadIdx.x; idx < g * D; idx += blockDim.x) {
        const int h = idx / D, c = idx % D;
        const size_t qi = ((size_t)b * a.Hq + (size_t)hkv * g + h) * D + c;
        sm.q[h][c] = ldf(a.q, qi, bf) * a.scale_log2;
    }
    __syncthreads();

    float* part_out = a.part + (unit * g * a.total_chunks + blockIdx.x) * (size_t)(D + 2);
    float* lg_unit = a.logits ? a.logits + unit * g * (size_t)a.slots : nullptr;
    int chunk = blockIdx.x, tier = -1;
    for (int t = 0; t < a.n_tiers; ++t) {
        if (chunk < a.tier[t].chunks) { tier = t; break; }
        chunk -= a.tier[t].chunks;
    }
    if (tier >= 0) {
        const TierArgs& t = a.tier[tier];
        if (t.count[unit] > t.cap && threadIdx.x == 0) atomicOr(&g_status_decode, kDevCheck);
        if (chunk * kChunk < min(t.count[unit], t.cap))
            dispatch_tier(a, sm, t, unit, chunk, part_out,
                          (a.policy == KVQ_POLICY_MIKV && lg_unit) ? lg_unit + t.slot_base : nullptr);
        else
            empty_partial(a, part_out);
    } else {
        const int cap = a.res_cap;
        const int len = min(max(a.res_len[unit], 0), cap - 1), start = a.res_start[unit];
        if (a.res_len[unit] != len && threadIdx.x == 0) atomicOr(&g_status_decode, kDevCheck);
        const int j0 = chunk * kChunk;
        const int n = min(kChunk, len + 1 - j0);
        const size_t rbase = unit * (size_t)cap;
        if (n > 0) {
            auto key = [&](int i, int c) -> float {
                const int li = j0 + i;
                return li < len ? ldf(a.res_k, (rbase + (start + li) % cap) * D + c, bf)
                                : ldf(a.k_new, unit * D + c, bf);
            };
            auto val = [&](int i, int c) -> float {
                const int li = j0 + i;
                return li < len ? ldf(a.res_v, (rbase + (start + li) % cap) * D + c, bf)
                                : ldf(a.v_new, unit * D + c, bf);
            };
            chunk_attend(a, sm, n, key, val, part_out,
                         (lg_unit && a.policy != KVQ_POLICY_MINIKV) ? lg_unit + a.res_slot_base + j0
                                                                    : nullptr);
        } else {
            empty_partial(a, part_out);
        }
        if (chunk == 0) {
            // the new token joins the ring; no CTA reads this slot in this step
            const size_t slot = rbase + (start + len) % cap;
            for (int c = threadIdx.x; c < D; c += blockDim.x) {
                stf(a.res_k, slot * D + c, ldf(a.k_new, unit * D + c, bf), bf);
                stf(a.res_v, slot * D + c, ldf(a.v_new, unit * D + c, bf), bf);
            }
            if (threadIdx.x == 0) a.res_token_id[slot] = a.seq_len[b];
        }
    }

    // ---- completion: the last CTA of the unit merges the partials
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(&a.counters[unit], 1u);
        sm.last = (prev == (uint32_t)a.total_chunks - 1u) ? 1 : 0;
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();

    const float* pu = a.part + unit * g * a.total_chunks * (size_t)(D + 2);
    if (threadIdx.x < g) {
        const float* ph = pu + (size_t)threadIdx.x * a.total_chunks * (D + 2);
        float M = -__int_as_float(0x7f800000);
        for (int x = 0; x < a.total_chunks; ++x)
            if (__ldcg(ph + (size_t)x * (D + 2) + 1) > 0.0f) M = fmaxf(M, __ldcg(ph + (size_t)x * (D + 2)));
        float L = 0.0f;
        for (int x = 0; x < a.total_chunks; ++x) {
            const float l = __ldcg(ph + (size_t)x * (D + 2) + 1);
            if (l > 0.0f) L += l * ex2_approx(__ldcg(ph + (size_t)x * (D + 2)) - M);
        }
        sm.red[threadIdx.x][0] = M;
        sm.red[threadIdx.x][1] = L;
        sm.m[threadIdx.x] = M + __log2f(L);          // base-2 lse
        if (a.lse_out) a.lse_out[(size_t)b * a.Hq + hkv * g + threadIdx.x] = (M + __log2f(L)) * kLn2;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < g * D; idx += blockDim.x) {
        const int h = idx / D, c = idx % D;
        const float* ph = pu + (size_t)h * a.total_chunks * (D + 2);
        const float M = sm.red[h][0], L = sm.red[h][1];
        float acc = 0.0f;
        for (int x = 0; x < a.total_chunks; ++x) {
            const float l = __ldcg(ph + (size_t)x * (D + 2) + 1);
            if (l > 0.0f) acc += __ldcg(ph + (size_t)x * (D + 2) + 2 + c) * ex2_approx(__ldcg(ph + (size_t)x * (D + 2)) - M);
        }
        stf(a.o, ((size_t)b * a.Hq + hkv * g + h) * D + c, acc / L, bf);
    }

    const int cap = a.res_cap;
    const int len = min(max(a.res_len[unit], 0), cap - 1), start = a.res_start[unit];
    if (a.policy == KVQ_POLICY_MIKV && lg_unit) {
        float* cs = a.cum_score + unit * (size_t)a.score_cap;
        for (int t = 0; t < a.n_tiers; ++t) {
            const TierArgs& ti = a.tier[t];
            const int cnt = min(ti.count[unit], ti.cap);
            for (int j = threadIdx.x; j < cnt; j += blockDim.x) {
                float p = 0.0f;
                for (int h = 0; h < g; ++h)
                    p += ex2_approx(__ldcg(lg_unit + (size_t)h * a.slots + ti.slot_base + j) - sm.m[h]);
                const int id = ti.token_id[unit * (size_t)ti.cap + j];
                if (id >= 0 && id < a.score_cap) cs[id] = __fadd_rn(cs[id], p);
                else atomicOr(&g_status_decode, kDevCheck);
            }
        }
        for (int li = threadIdx.x; li <= len; li += blockDim.x) {
            float p = 0.0f;
            for (int h = 0; h < g; ++h)
                p += ex2_approx(__ldcg(lg_unit + (size_t)h * a.slots + a.res_slot_base + li) - sm.m[h]);
            const int id = li < len ? a.res_token_id[unit * (size_t)cap + (start + li) % cap] : a.seq_len[b];
            if (id < 0 || id >= a.score_cap) atomicOr(&g_status_decode, kDevCheck);
            else cs[id] = li < len ? __fadd_rn(cs[id], p) : p;
        }
    } else if (a.policy == KVQ_POLICY_DIFFKV && lg_unit) {
        for (int idx = threadIdx.x; idx < (len + 1) * g; idx += blockDim.x) {
            const int li = idx / g, h = idx % g;
            const float p = ex2_approx(__ldcg(lg_unit + (size_t)h * a.slots + a.res_slot_base + li) - sm.m[h]);
            float* wa = a.win_acc + ((size_t)b * a.Hq + hkv * g + h) * cap + (start + li) % cap;
            *wa = li < len ? __fadd_rn(*wa, p) : p;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        a.res_len[unit] = len + 1;
        a.counters[unit] = 0u;
        __threadfence();
        const uint32_t prev = atomicAdd(&a.counters[units], 1u);
        if (prev == (uint32_t)units - 1u) {
            __threadfence();
            for (int bb = 0; bb < a.B; ++bb) a.seq_len[bb] += 1;
            a.counters[units] = 0u;
        }
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
    int total_chunks, slots;
    size_t part, logits, counters, total;
};

WsLayout ws_layout(const kvq_cache& c) {
    WsLayout w{};
    const int units = c.B * c.Hkv, g = c.Hq / c.Hkv;
    int chunks = 0, slots = 0;
    for (int t = 0; t < c.n_tiers; ++t) {
        chunks += (c.tier[t].cap + kChunk - 1) / kChunk;
        slots += c.tier[t].cap;
    }
    chunks += (c.res_cap + kChunk - 1) / kChunk;
    slots += c.res_cap;
    w.total_chunks = chunks;
    w.slots = slots;
    w.part = 0;
    size_t off = align256((size_t)units * g * chunks * (c.D + 2) * sizeof(float));
    w.logits = off;
    if (c.policy != KVQ_POLICY_MINIKV) off += align256((size_t)units * g * slots * sizeof(float));
    w.counters = off;
    off += align256((size_t)(units + 1) * sizeof(uint32_t));
    w.total = off;
    return w;
}

}  // namespace

size_t decode_workspace_bytes(const kvq_cache& c) { return ws_layout(c).total; }

cudaError_t launch_decode(const void* q, const void* k_new, const void* v_new, const kvq_cache& c,
                          float sm_scale, void* o, float* lse_out, void* ws, cudaStream_t s) {
    const WsLayout w = ws_layout(c);
    const int units = c.B * c.Hkv;
    DecodeArgs a{};
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.o = o;
    a.lse_out = lse_out;
    a.B = c.B;
    a.Hq = c.Hq;
    a.Hkv = c.Hkv;
    a.D = c.D;
    a.G = c.G;
    a.g = c.Hq / c.Hkv;
    a.n_tiers = c.n_tiers;
    a.policy = c.policy;
    a.bf16 = c.dtype == KVQ_BF16 ? 1 : 0;
    int slot = 0;
    for (int t = 0; t < c.n_tiers; ++t) {
        const kvq_tier& ct = c.tier[t];
        TierArgs& ta = a.tier[t];
        ta.k_bits = ct.k_bits;
        ta.v_bits = ct.v_bits;
        ta.k_axis = ct.k_axis;
        ta.cap = ct.cap;
        ta.k_codes = ct.k_codes;
        ta.k_scale = ct.k_scale;
        ta.k_zero = ct.k_zero;
        ta.v_codes = ct.v_codes;
        ta.v_scale = ct.v_scale;
        ta.v_zero = ct.v_zero;
        ta.token_id = ct.token_id;
        ta.count = ct.count;
        ta.chunks = (ct.cap + kChunk - 1) / kChunk;
        ta.slot_base = slot;
        slot += ct.cap;
    }
    a.res_k = c.res_k;
    a.res_v = c.res_v;
    a.res_token_id = c.res_token_id;
    a.res_start = c.res_start;
    a.res_len = c.res_len;
    a.res_cap = c.res_cap;
    a.res_chunks = (c.res_cap + kChunk - 1) / kChunk;
    a.res_slot_base = slot;
    a.seq_len = c.seq_len;
    a.win_acc = c.win_acc;
    a.cum_score = c.cum_score;
    a.score_cap = c.score_cap;
    a.scale_log2 = sm_scale * kLog2e;
    a.total_chunks = w.total_chunks;
    a.slots = w.slots;
    uint8_t* base = static_cast<uint8_t*>(ws);
    a.part = reinterpret_cast<float*>(base + w.part);
    a.logits = c.policy != KVQ_POLICY_MINIKV ? reinterpret_cast<float*>(base + w.logits) : nullptr;
    a.counters = reinterpret_cast<uint32_t*>(base + w.counters);
    cudaError_t e = cudaMemsetAsync(a.counters, 0, (size_t)(units + 1) * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    dim3 grid(w.total_chunks, units);
    decode_kernel<<<grid, kThreads, sizeof(Smem), s>>>(a);
    return cudaGetLastError();
}

}  // namespace kvq
