// requant_demote: the cache life cycles.
//
// MiniKV (review page, "Assumptions & free parameters"; verdict JSON
// key_machinery): selection persists from the end of prefill; selected
// tokens are packed once (per-channel INT2 keys, per-token INT2 values),
// the newest stay at full precision in the residual and move to the packed
// tier G at a time.
// DiffKV (verdict JSON key_machinery, Algorithm 1 comments): significance =
// mean attention received, max over the GQA group; K8V4 above alpha_h/N,
// K4V2 above alpha_l/N, pruned below, decided once as a token leaves the
// recent window.
// MiKV (rebuttal: re-quantisation paragraph, Q1, regrouping paragraph): the
// top share by cumulative attention is INT4, the rest INT2, nothing is
// evicted, INT4 tokens that leave the top share are re-quantised to INT2.
//
// One CTA per unit for every per-unit decision; radix select with ties to
// the lower position; tier slots are filled in a fixed order so results
// are deterministic.
#include <algorithm>

#include "kvq_internal.h"
#include "pack_device.cuh"
#include "topk_device.cuh"

namespace kvq {

KVQ_DEFINE_STATUS(policy)

namespace {

__device__ __forceinline__ float unorderable(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

__device__ __forceinline__ float ld_act(const void* p, size_t i, bool bf) {
    return bf ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i])
              : __half2float(reinterpret_cast<const __half*>(p)[i]);
}

__device__ __forceinline__ void copy_act(void* dst, size_t di, const void* src, size_t si, bool bf) {
    reinterpret_cast<uint16_t*>(dst)[di] = reinterpret_cast<const uint16_t*>(src)[si];
    (void)bf;
}

struct TierDev {
    int k_bits, v_bits, k_axis, cap;
    uint32_t* k_codes;
    uint16_t* k_scale;
    uint16_t* k_zero;
    uint32_t* v_codes;
    uint16_t* v_scale;
    uint16_t* v_zero;
    int32_t* token_id;
    int32_t* count;
    // paged tiers (page_table != nullptr): slot s of unit u lives in page
    // page_table[u * max_pages + s / P] at row s mod P (P = KVQ_PAGE_TOKENS)
    int32_t* page_table;
    int32_t* page_owner;
    int32_t* free_ring;
    uint32_t* ring_ctr;
    int max_pages, n_pages;
};

// Flat row of slot `slot` of unit `unit` in the tier's arrays (the page's row when paged).
__device__ __forceinline__ size_t slot_row(const TierDev& t, size_t unit, int slot) {
    if (t.page_table) {
        const int pg = t.page_table[unit * (size_t)t.max_pages + (slot / KVQ_PAGE_TOKENS)];
        return (size_t)pg * KVQ_PAGE_TOKENS + (size_t)(slot % KVQ_PAGE_TOKENS);
    }
    return unit * (size_t)t.cap + slot;
}

struct PolicyArgs {
    int B, Hq, Hkv, D, G, g, bf16, n_tiers, nr, hi_den;
    TierDev tier[KVQ_MAX_TIERS];
    void* res_k;
    void* res_v;
    int32_t* res_token_id;
    int32_t* res_start;
    int32_t* res_len;
    int res_cap;
    int32_t* seq_len;           // [units] position of the next token
    float* win_acc;
    float* alpha;
    float* cum_score;
    int score_cap;
    // build inputs
    const void* k_src;
    const void* v_src;
    int T;
    const int32_t* sel_idx;
    int n_sel;
    const float* colscore;
    const int32_t* n_high;
    const int32_t* n_low;
};

// Quantise one token row (token grouping, any bit width) into a tier slot.
template <typename Load>
__device__ void quant_row(Load load, int D, int G, int bits, uint32_t* codes, uint16_t* s,
                          uint16_t* z) {
    for (int grp = 0; grp < D / G; ++grp)
        quant_token_group([&](int i) { return load(grp * G + i); }, G, bits,
                          codes + grp * (G * bits / 32), s + grp, z + grp);
}

__device__ __forceinline__ uint32_t* krow(const TierDev& t, size_t unit, int slot, int D) {
    return t.k_codes + slot_row(t, unit, slot) * (size_t)(D * t.k_bits / 32);
}
__device__ __forceinline__ uint32_t* vrow(const TierDev& t, size_t unit, int slot, int D) {
    return t.v_codes + slot_row(t, unit, slot) * (size_t)(D * t.v_bits / 32);
}
__device__ __forceinline__ size_t srow(const TierDev& t, size_t unit, int slot, int D, int G) {
    return slot_row(t, unit, slot) * (size_t)(D / G);
}

// Quantise raw token `pos` of a [units][T][D] source (or ring slot) into a
// token-grouped tier slot.
__device__ void put_raw_token(const PolicyArgs& a, const TierDev& t, size_t unit, int slot,
                              const void* ksrc, const void* vsrc, size_t row_elem, int token_id) {
    const int D = a.D, G = a.G;
    const bool bf = a.bf16 != 0;
    quant_row([&](int c) { return ld_act(ksrc, row_elem + c, bf); }, D, G, t.k_bits,
              krow(t, unit, slot, D), t.k_scale + srow(t, unit, slot, D, G),
              t.k_zero + srow(t, unit, slot, D, G));
    quant_row([&](int c) { return ld_act(vsrc, row_elem + c, bf); }, D, G, t.v_bits,
              vrow(t, unit, slot, D), t.v_scale + srow(t, unit, slot, D, G),
              t.v_zero + srow(t, unit, slot, D, G));
    t.token_id[slot_row(t, unit, slot)] = token_id;
}

// One warp: the same token into a tier slot, group-parallel for G = 32
// (lanes 0 .. D/32 - 1 take the key groups, the next D/32 lanes the value
// groups, each group loaded once); other group sizes run serially on lane 0.
__device__ void put_token_warp(const PolicyArgs& a, const TierDev& t, size_t unit, int slot,
                               const void* ksrc, const void* vsrc, size_t row_elem, int token_id) {
    const int lane = threadIdx.x & 31;
    const int D = a.D, G = a.G, ng = D / G;
    if (G != 32 || 2 * ng > 32) {
        if (lane == 0) put_raw_token(a, t, unit, slot, ksrc, vsrc, row_elem, token_id);
        return;
    }
    const bool bf = a.bf16 != 0;
    if (lane < 2 * ng) {
        const bool isv = lane >= ng;
        const int grp = isv ? lane - ng : lane;
        const void* src = isv ? vsrc : ksrc;
        const int bits = isv ? t.v_bits : t.k_bits;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = ld_act(src, row_elem + (size_t)grp * 32 + i, bf);
        const QParams q = params32(v, bits);
        uint32_t* codes = (isv ? vrow(t, unit, slot, D) : krow(t, unit, slot, D)) + grp * bits;
        switch (bits) {
            case 2: pack32<2>(v, q, codes, 1); break;
            case 4: pack32<4>(v, q, codes, 1); break;
            default: pack32<8>(v, q, codes, 1); break;
        }
        const size_t so = srow(t, unit, slot, D, G) + grp;
        (isv ? t.v_scale : t.k_scale)[so] = q.s_bits;
        (isv ? t.v_zero : t.k_zero)[so] = q.z_bits;
    }
    if (lane == 0) t.token_id[slot_row(t, unit, slot)] = token_id;
}

// ----------------------------------------------------------------- MiniKV

// Token ids, residual and counters after the two packing launches.
// Grid (units, row blocks): each warp copies whole residual rows with
// 16-byte vectors; block 0 of a unit also writes the packed tokens' ids and
// the counters.
constexpr int kTailRows = 8;          // residual rows per CTA (one per warp)
__global__ void __launch_bounds__(kTailRows * 32) minikv_build_tail(PolicyArgs a, int npk, int r0) {
    const size_t unit = blockIdx.x;
    const int32_t* sel = a.sel_idx + unit * (size_t)a.n_sel;
    const TierDev& t = a.tier[0];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.y * kTailRows + warp;             // residual row of this warp
    if (i < r0) {
        const int pos = sel[npk + i];
        if (pos < 0 || pos >= a.T) {
            if (lane == 0) atomicOr(&g_status_policy, kDevCheck);
        } else {
            const int vec = a.D * 2 / 16;                    // 16-byte pieces per row
            const uint4* ks = reinterpret_cast<const uint4*>(
                reinterpret_cast<const uint16_t*>(a.k_src) + (unit * a.T + pos) * (size_t)a.D);
            const uint4* vs = reinterpret_cast<const uint4*>(
                reinterpret_cast<const uint16_t*>(a.v_src) + (unit * a.T + pos) * (size_t)a.D);
            uint4* kd = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.res_k) +
                                                 (unit * a.res_cap + i) * (size_t)a.D);
            uint4* vd = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.res_v) +
                                                 (unit * a.res_cap + i) * (size_t)a.D);
            for (int e = lane; e < 2 * vec; e += 32) {
                if (e < vec) kd[e] = ks[e];
                else vd[e - vec] = vs[e - vec];
            }
            if (lane == 0) a.res_token_id[unit * a.res_cap + i] = pos;
        }
    }
    if (blockIdx.y == 0) {
        for (int k = threadIdx.x; k < npk; k += blockDim.x) t.token_id[unit * t.cap + k] = sel[k];
        if (threadIdx.x == 0) {
            t.count[unit] = npk;
            a.res_start[unit] = 0;
            a.res_len[unit] = r0;
            a.seq_len[unit] = a.T;
        }
    }
}

// The whole prefill-end build of one unit in one CTA, straight from its
// column scores: heavy hitters (radix select over positions < T - w, ties to
// the lower position) plus the recent window into shared memory, ascending;
// then the per-channel key groups and the per-token value groups of the
// packed part, the residual rows, token ids and counters.  Same arithmetic
// and layout as select_tokens followed by requant_demote(step 0).
template <typename T, int KB, int VB>
__global__ void __launch_bounds__(kTopkBlock) minikv_fused_build(PolicyArgs a, const float* __restrict__ score,
                                                                 const int32_t* __restrict__ k_hh, int kmax, int w,
                                                                 int32_t* __restrict__ idx_out) {
    __shared__ TopkShared sh;
    extern __shared__ int32_t sel[];                 // [kmax + w] selected positions, ascending
    const size_t unit = blockIdx.x;
    const int Tn = a.T, D = a.D, nc = Tn - w;
    const float* sc = score + unit * (size_t)Tn;
    int k = k_hh[unit];
    if (k < 0 || k > kmax) {
        if (threadIdx.x == 0) atomicOr(&g_status_policy, kDevCheck);
        k = k < 0 ? 0 : kmax;
    }
    if (k > nc) k = nc;
    if (k > 0) {
        uint32_t kstar, take_eq;
        block_radix_select([&](int i) { return orderable(sc[i]); }, nc, k, sh, &kstar, &take_eq);
        uint32_t eq_base = 0, out_base = 0;
        for (int c0 = 0; c0 < nc; c0 += blockDim.x) {
            const int j = c0 + threadIdx.x;
            const uint32_t kv = j < nc ? orderable(sc[j]) : 0u;
            const uint32_t gt = (j < nc && kv > kstar) ? 1u : 0u;
            const uint32_t eq = (j < nc && kv == kstar) ? 1u : 0u;
            uint32_t eq_tot;
            const uint32_t eq_rank = block_excl_scan(eq, sh, &eq_tot);
            const uint32_t take = gt | (eq & (eq_base + eq_rank < take_eq ? 1u : 0u));
            uint32_t sel_tot;
            const uint32_t pos = block_excl_scan(take, sh, &sel_tot);
            if (take) sel[out_base + pos] = j;
            eq_base += eq_tot;
            out_base += sel_tot;
        }
    }
    for (int i = threadIdx.x; i < w; i += blockDim.x) sel[k + i] = nc + i;
    __syncthreads();
    const int n = k + w, nr = a.nr;
    const int r0 = n <= nr ? n : nr + (n - nr) % 32, npk = n - r0;
    const TierDev& t = a.tier[0];
    if (idx_out)
        for (int i = threadIdx.x; i < n; i += blockDim.x) idx_out[unit * (size_t)(kmax + w) + i] = sel[i];
    const T* ks = reinterpret_cast<const T*>(a.k_src) + unit * (size_t)Tn * D;
    const T* vs = reinterpret_cast<const T*>(a.v_src) + unit * (size_t)Tn * D;
    // keys: channel c of packed group grp (32 selected tokens), one task per thread
    const int kgroups = npk / 32;
    for (int task = threadIdx.x; task < kgroups * D; task += blockDim.x) {
        const int grp = task / D, c = task - grp * D;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = Elem<T>::to_f(ks[(size_t)sel[grp * 32 + i] * D + c]);
        const QParams q = params32(v, KB);
        pack32<KB>(v, q, t.k_codes + (unit * (size_t)(t.cap * KB / 32) + (size_t)grp * KB) * D + c, D);
        const size_t so = (unit * (size_t)(t.cap / 32) + grp) * D + c;
        t.k_scale[so] = q.s_bits;
        t.k_zero[so] = q.z_bits;
    }
    // values: 32-channel group g of packed token i (four 16-byte loads)
    const int vg = D / 32;
    for (int task = threadIdx.x; task < npk * vg; task += blockDim.x) {
        const int i = task / vg, g = task - i * vg;
        const uint4* src = reinterpret_cast<const uint4*>(vs + (size_t)sel[i] * D + (size_t)g * 32);
        float v[32];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const uint4 wv = src[q4];
            const T* e = reinterpret_cast<const T*>(&wv);
#pragma unroll
            for (int u = 0; u < 8; ++u) v[8 * q4 + u] = Elem<T>::to_f(e[u]);
        }
        const QParams q = params32(v, VB);
        const size_t orow = unit * (size_t)t.cap + i;
        pack32<VB>(v, q, t.v_codes + orow * (D * VB / 32) + (size_t)g * VB, 1);
        t.v_scale[orow * vg + g] = q.s_bits;
        t.v_zero[orow * vg + g] = q.z_bits;
    }
    // residual rows (16-byte pieces), token ids, counters
    const int vec = D * 2 / 16;
    for (int task = threadIdx.x; task < r0 * 2 * vec; task += blockDim.x) {
        const int i = task / (2 * vec), e = task - i * (2 * vec);
        const int pos = sel[npk + i];
        const bool isv = e >= vec;
        const uint4* src = reinterpret_cast<const uint4*>((isv ? vs : ks) + (size_t)pos * D) + (isv ? e - vec : e);
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(isv ? a.res_v : a.res_k) +
                                              (unit * a.res_cap + i) * (size_t)D) + (isv ? e - vec : e);
        *dst = *src;
    }
    for (int i = threadIdx.x; i < r0; i += blockDim.x) a.res_token_id[unit * a.res_cap + i] = sel[npk + i];
    for (int i = threadIdx.x; i < npk; i += blockDim.x) t.token_id[unit * t.cap + i] = sel[i];
    if (threadIdx.x == 0) {
        t.count[unit] = npk;
        a.res_start[unit] = 0;
        a.res_len[unit] = r0;
        a.seq_len[unit] = Tn;
    }
}

// ----------------------------------------------------------------- DiffKV

__global__ void __launch_bounds__(kTopkBlock) diffkv_build(PolicyArgs a) {
    __shared__ TopkShared sh;
    const size_t unit = blockIdx.x;
    const int b = (int)(unit / a.Hkv), hkv = (int)(unit % a.Hkv);
    const int T = a.T, W = a.nr, g = a.g, D = a.D;
    const int nc = T - W;
    const float* cs = a.colscore + ((size_t)b * a.Hq + (size_t)hkv * g) * T;
    auto sig = [&](int j) -> float {
        const float cnt = (float)(T - j);
        float m = __fdiv_rn(cs[j], cnt);
        for (int h = 1; h < g; ++h) m = fmaxf(m, __fdiv_rn(cs[(size_t)h * T + j], cnt));
        return m;
    };
    auto key = [&](int j) { return orderable(sig(j)); };
    int nh = a.n_high[unit], nl = a.n_low[unit];
    nh = max(0, min(nh, nc));
    nl = max(0, min(nl, nc - nh));
    uint32_t k1 = 0xffffffffu, t1 = 0, k2 = 0xffffffffu, t2 = 0;
    if (nh > 0) block_radix_select(key, nc, nh, sh, &k1, &t1);
    if (nh + nl > 0) block_radix_select(key, nc, nh + nl, sh, &k2, &t2);
    const float Tf = (float)T;
    const float alpha_h = nh > 0 ? __fmul_rn(Tf, unorderable(k1)) : __int_as_float(0x7f800000);
    const float alpha_l = nl > 0 ? __fmul_rn(Tf, unorderable(k2)) : alpha_h;
    const TierDev& th = a.tier[0];
    const TierDev& tl = a.tier[1];
    // slots each tier can hold for this unit: its capacity, or for a paged tier the pages
    // the build gave it (fewer when the pool ran out)
    __shared__ int lim_s[2];
    if (threadIdx.x < 2) {
        const TierDev& t = a.tier[threadIdx.x];
        int lim = t.cap;
        if (t.page_table) {
            int k = 0;
            while (k < t.max_pages && t.page_table[unit * (size_t)t.max_pages + k] >= 0) ++k;
            lim = min(lim, k * KVQ_PAGE_TOKENS);
        }
        lim_s[threadIdx.x] = lim;
    }
    __syncthreads();
    const uint32_t lim_h = (uint32_t)lim_s[0], lim_l = (uint32_t)lim_s[1];
    uint32_t eq1_base = 0, eq2_base = 0, hi_base = 0, lo_base = 0;
    for (int c0 = 0; c0 < nc; c0 += blockDim.x) {
        const int j = c0 + threadIdx.x;
        const uint32_t kv = j < nc ? key(j) : 0u;
        const uint32_t e1 = (j < nc && nh > 0 && kv == k1) ? 1u : 0u;
        const uint32_t e2 = (j < nc && nh + nl > 0 && kv == k2) ? 1u : 0u;
        uint32_t tot1, tot2;
        const uint32_t r1 = block_excl_scan(e1, sh, &tot1);
        const uint32_t r2 = block_excl_scan(e2, sh, &tot2);
        const bool in1 = j < nc && nh > 0 && (kv > k1 || (e1 && eq1_base + r1 < t1));
        const bool in2 = j < nc && nh + nl > 0 && (kv > k2 || (e2 && eq2_base + r2 < t2));
        const uint32_t is_hi = in1 ? 1u : 0u, is_lo = (in2 && !in1) ? 1u : 0u;
        uint32_t tot_hi, tot_lo;
        const uint32_t ph = block_excl_scan(is_hi, sh, &tot_hi);
        const uint32_t pl = block_excl_scan(is_lo, sh, &tot_lo);
        const size_t row = (unit * T + j) * (size_t)D;
        if (is_hi && hi_base + ph < lim_h)
            put_raw_token(a, th, unit, hi_base + ph, a.k_src, a.v_src, row, j);
        if (is_lo && lo_base + pl < lim_l)
            put_raw_token(a, tl, unit, lo_base + pl, a.k_src, a.v_src, row, j);
        if ((is_hi && hi_base + ph >= lim_h) || (is_lo && lo_base + pl >= lim_l))
            atomicOr(&g_status_policy, kDevCheck);
        eq1_base += tot1;
        eq2_base += tot2;
        hi_base += tot_hi;
        lo_base += tot_lo;
    }
    // recent window -> ring, with the attention each head already gave it
    const bool bf = a.bf16 != 0;
    for (int idx = threadIdx.x; idx < W * D; idx += blockDim.x) {
        const int i = idx / D, c = idx % D;
        const size_t src = (unit * T + nc + i) * (size_t)D + c;
        const size_t dst = (unit * a.res_cap + i) * (size_t)D + c;
        copy_act(a.res_k, dst, a.k_src, src, bf);
        copy_act(a.res_v, dst, a.v_src, src, bf);
    }
    for (int idx = threadIdx.x; idx < W * g; idx += blockDim.x) {
        const int i = idx / g, h = idx % g;
        a.win_acc[((size_t)b * a.Hq + (size_t)hkv * g + h) * a.res_cap + i] = cs[(size_t)h * T + nc + i];
    }
    for (int i = threadIdx.x; i < W; i += blockDim.x) a.res_token_id[unit * a.res_cap + i] = nc + i;
    if (threadIdx.x == 0) {
        th.count[unit] = min((int)hi_base, (int)lim_h);
        tl.count[unit] = min((int)lo_base, (int)lim_l);
        a.res_start[unit] = 0;
        a.res_len[unit] = W;
        a.alpha[unit * 2] = alpha_h;
        a.alpha[unit * 2 + 1] = alpha_l;
        a.seq_len[unit] = T;
    }
}

// The oldest window token leaves: K8V4, K4V2 or pruned.
__global__ void diffkv_exit(PolicyArgs a) {
    const size_t unit = blockIdx.x;
    const int len = a.res_len[unit];
    if (len <= a.nr) return;
    const int b = (int)(unit / a.Hkv), hkv = (int)(unit % a.Hkv);
    const int start = a.res_start[unit], cap = a.res_cap, g = a.g;
    const int tc = a.res_token_id[unit * cap + start];
    const int N = a.seq_len[unit];
    const float cnt = (float)(N - tc);
    float score = -__int_as_float(0x7f800000);
    for (int h = 0; h < g; ++h)
        score = fmaxf(score, __fdiv_rn(a.win_acc[((size_t)b * a.Hq + (size_t)hkv * g + h) * cap + start], cnt));
    const float th_h = __fdiv_rn(a.alpha[unit * 2], (float)N);
    const float th_l = __fdiv_rn(a.alpha[unit * 2 + 1], (float)N);
    const int cls = score >= th_h ? 0 : (score >= th_l ? 1 : 2);
    bool stored = false;
    if (cls < 2) {
        const TierDev& t = a.tier[cls];
        const int slot = t.count[unit];
        bool room = slot < t.cap;
        if (room && t.page_table && slot % KVQ_PAGE_TOKENS == 0) {
            // the token opens a logical page: one page from the ring head
            int pg = -1;
            if (threadIdx.x == 0) {
                const uint32_t h = atomicAdd(&t.ring_ctr[0], 1u);
                const uint32_t tail = *(volatile uint32_t*)&t.ring_ctr[1];
                if (h < tail) {
                    pg = t.free_ring[h % (uint32_t)t.n_pages];
                    const int li = slot / KVQ_PAGE_TOKENS;
                    t.page_table[unit * (size_t)t.max_pages + li] = pg;
                    t.page_owner[pg] = (int)unit * t.max_pages + li;
                }
            }
            pg = __shfl_sync(0xffffffffu, pg, 0);
            __syncwarp();                                  // the table entry before the row writes
            room = pg >= 0;
        }
        if (!room) {
            if (threadIdx.x == 0) atomicOr(&g_status_policy, kDevCheck);
        } else {
            put_token_warp(a, t, unit, slot, a.res_k, a.res_v, (unit * cap + start) * (size_t)a.D, tc);
            stored = true;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (stored) a.tier[cls].count[unit] += 1;
        a.res_start[unit] = (start + 1) % cap;
        a.res_len[unit] = len - 1;
    }
}

// ---- DiffKV page pools ([DiffKV-J] unified pages, circular free page list,
// bidirectional page table, parallel compaction): one CTA per pool operation.

// Every page held by the units u with rel(u) goes back to the ring tail: units in
// order, pages in logical order (each unit's run starts at the exclusive prefix
// sum of the held counts).  Pages of a unit are a prefix of its table row.
template <typename Rel>
__device__ void pages_push(const TierDev& t, int units, Rel rel, TopkShared& sh, uint32_t* tail) {
    const uint32_t n = (uint32_t)t.n_pages;
    uint32_t base = 0;
    for (int u0 = 0; u0 < units; u0 += blockDim.x) {
        const int u = u0 + threadIdx.x;
        uint32_t held = 0;
        if (u < units && rel(u))
            for (int i = 0; i < t.max_pages && t.page_table[(size_t)u * t.max_pages + i] >= 0; ++i) ++held;
        uint32_t tot;
        const uint32_t off = block_excl_scan(held, sh, &tot);
        for (uint32_t i = 0; i < held; ++i) {
            int32_t* e = &t.page_table[(size_t)u * t.max_pages + i];
            const int pg = *e;
            t.free_ring[(*tail + base + off + i) % n] = pg;
            t.page_owner[pg] = -1;
            *e = -1;
        }
        base += tot;
    }
    __syncthreads();
    if (threadIdx.x == 0) *tail += base;
    __syncthreads();
}

// Prefill-end allocation of the paged tiers: every unit's old pages back to the
// ring, then ceil(n / P) pages per unit for its n tokens of the tier (the same n
// diffkv_build stores), one run per unit from the ring head in unit order.
__global__ void __launch_bounds__(kTopkBlock) pages_build_alloc(PolicyArgs a) {
    __shared__ TopkShared sh;
    __shared__ uint32_t ctr[2];
    const int units = a.B * a.Hkv, nc = a.T - a.nr;
    for (int ti = 0; ti < a.n_tiers; ++ti) {
        const TierDev& t = a.tier[ti];
        if (!t.page_table) continue;
        if (threadIdx.x == 0) {
            ctr[0] = t.ring_ctr[0];
            ctr[1] = t.ring_ctr[1];
        }
        __syncthreads();
        pages_push(t, units, [](int) { return true; }, sh, &ctr[1]);
        auto demand = [&](int u) -> uint32_t {
            const int nh = max(0, min(a.n_high[u], nc));
            const int n = ti == 0 ? nh : max(0, min(a.n_low[u], nc - nh));
            return (uint32_t)min((n + KVQ_PAGE_TOKENS - 1) / KVQ_PAGE_TOKENS, t.max_pages);
        };
        uint32_t total = 0;
        for (int u0 = 0; u0 < units; u0 += blockDim.x) {
            const int u = u0 + threadIdx.x;
            uint32_t tot;
            (void)block_excl_scan(u < units ? demand(u) : 0u, sh, &tot);
            total += tot;
        }
        const bool fits = total <= ctr[1] - ctr[0];
        if (!fits && threadIdx.x == 0) atomicOr(&g_status_policy, kDevCheck);
        const uint32_t n = (uint32_t)t.n_pages;
        uint32_t base = 0;
        for (int u0 = 0; fits && u0 < units; u0 += blockDim.x) {
            const int u = u0 + threadIdx.x;
            const uint32_t d = u < units ? demand(u) : 0u;
            uint32_t tot;
            const uint32_t off = block_excl_scan(d, sh, &tot);
            for (uint32_t i = 0; i < d; ++i) {
                const int pg = t.free_ring[(ctr[0] + base + off + i) % n];
                t.page_table[(size_t)u * t.max_pages + i] = pg;
                t.page_owner[pg] = u * t.max_pages + (int)i;
            }
            base += tot;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            t.ring_ctr[0] = ctr[0] + (fits ? total : 0u);
            t.ring_ctr[1] = ctr[1];
        }
        __syncthreads();
    }
}

// Every paged tier empty: ring = 0 .. n_pages-1, no owners, no table entries, counts 0.
__global__ void pages_init_kernel(PolicyArgs a) {
    const int units = a.B * a.Hkv;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (int ti = 0; ti < a.n_tiers; ++ti) {
        const TierDev& t = a.tier[ti];
        if (!t.page_table) continue;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)t.n_pages; i += stride) {
            t.free_ring[i] = (int32_t)i;
            t.page_owner[i] = -1;
        }
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)units * t.max_pages; i += stride)
            t.page_table[i] = -1;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)units; i += stride) t.count[i] = 0;
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            t.ring_ctr[0] = 0u;
            t.ring_ctr[1] = (uint32_t)t.n_pages;
        }
    }
}

// A request is done: the units with mask[u] != 0 give their pages back (parallel
// compaction at the ring tail) and are left empty.
__global__ void __launch_bounds__(kTopkBlock) pages_release_kernel(PolicyArgs a, const int32_t* __restrict__ mask) {
    __shared__ TopkShared sh;
    __shared__ uint32_t tail;
    const int units = a.B * a.Hkv;
    for (int ti = 0; ti < a.n_tiers; ++ti) {
        const TierDev& t = a.tier[ti];
        if (t.page_table) {
            if (threadIdx.x == 0) tail = t.ring_ctr[1];
            __syncthreads();
            pages_push(t, units, [&](int u) { return mask[u] != 0; }, sh, &tail);
            if (threadIdx.x == 0) t.ring_ctr[1] = tail;
        }
        for (int u = threadIdx.x; u < units; u += blockDim.x)
            if (mask[u]) t.count[u] = 0;
    }
    for (int u = threadIdx.x; u < units; u += blockDim.x)
        if (mask[u]) {
            a.res_len[u] = 0;
            a.res_start[u] = 0;
            a.seq_len[u] = 0;
        }
}

// ----------------------------------------------------------------- MiKV

__global__ void __launch_bounds__(kTopkBlock) mikv_build(PolicyArgs a) {
    __shared__ TopkShared sh;
    const size_t unit = blockIdx.x;
    const int b = (int)(unit / a.Hkv), hkv = (int)(unit % a.Hkv);
    const int T = a.T, g = a.g, D = a.D, nr = a.nr;
    const int nq = max(T - nr, 0);
    const float* cs = a.colscore + ((size_t)b * a.Hq + (size_t)hkv * g) * T;
    float* cum = a.cum_score + unit * (size_t)a.score_cap;
    for (int j = threadIdx.x; j < T; j += blockDim.x) {
        float acc = 0.0f;
        for (int h = 0; h < g; ++h) acc = __fadd_rn(acc, cs[(size_t)h * T + j]);
        cum[j] = acc;
    }
    __syncthreads();
    const int n4 = nq / a.hi_den;
    auto key = [&](int j) { return orderable(cum[j]); };
    uint32_t k1 = 0xffffffffu, t1 = 0;
    if (n4 > 0) block_radix_select(key, nq, n4, sh, &k1, &t1);
    const TierDev& th = a.tier[0];
    const TierDev& tl = a.tier[1];
    uint32_t eq_base = 0, hi_base = 0, lo_base = 0;
    for (int c0 = 0; c0 < nq; c0 += blockDim.x) {
        const int j = c0 + threadIdx.x;
        const uint32_t kv = j < nq ? key(j) : 0u;
        const uint32_t e1 = (j < nq && n4 > 0 && kv == k1) ? 1u : 0u;
        uint32_t tot1;
        const uint32_t r1 = block_excl_scan(e1, sh, &tot1);
        const bool in1 = j < nq && n4 > 0 && (kv > k1 || (e1 && eq_base + r1 < t1));
        const uint32_t is_hi = in1 ? 1u : 0u, is_lo = (j < nq && !in1) ? 1u : 0u;
        uint32_t tot_hi, tot_lo;
        const uint32_t ph = block_excl_scan(is_hi, sh, &tot_hi);
        const uint32_t pl = block_excl_scan(is_lo, sh, &tot_lo);
        const size_t row = (unit * T + j) * (size_t)D;
        if (is_hi && hi_base + ph < (uint32_t)th.cap)
            put_raw_token(a, th, unit, hi_base + ph, a.k_src, a.v_src, row, j);
        if (is_lo && lo_base + pl < (uint32_t)tl.cap)
            put_raw_token(a, tl, unit, lo_base + pl, a.k_src, a.v_src, row, j);
        if ((is_hi && hi_base + ph >= (uint32_t)th.cap) || (is_lo && lo_base + pl >= (uint32_t)tl.cap))
            atomicOr(&g_status_policy, kDevCheck);
        eq_base += tot1;
        hi_base += tot_hi;
        lo_base += tot_lo;
    }
    const bool bf = a.bf16 != 0;
    const int r0 = T - nq;
    for (int idx = threadIdx.x; idx < r0 * D; idx += blockDim.x) {
        const int i = idx / D, c = idx % D;
        const size_t src = (unit * T + nq + i) * (size_t)D + c;
        const size_t dst = (unit * a.res_cap + i) * (size_t)D + c;
        copy_act(a.res_k, dst, a.k_src, src, bf);
        copy_act(a.res_v, dst, a.v_src, src, bf);
    }
    for (int i = threadIdx.x; i < r0; i += blockDim.x) a.res_token_id[unit * a.res_cap + i] = nq + i;
    if (threadIdx.x == 0) {
        th.count[unit] = min((int)hi_base, th.cap);
        tl.count[unit] = min((int)lo_base, tl.cap);
        a.res_start[unit] = 0;
        a.res_len[unit] = r0;
        a.seq_len[unit] = T;
    }
}

struct MikvShared {
    TopkShared tk;
    uint32_t cnt_eq;
    uint32_t kmin, kmax;                 // the population's smallest and largest ranking keys
};

// One warp: INT4 slot i of tier th dequantised and re-quantised into slot `slot` of tier
// tl, group-parallel for G = 32 (lanes 0 .. D/32 - 1 the key groups, the next D/32 lanes
// the value groups); other group sizes run serially on lane 0.
__device__ void requant_row_warp(const PolicyArgs& a, const TierDev& th, const TierDev& tl, size_t unit, int i,
                                 int slot) {
    const int lane = threadIdx.x & 31;
    const int D = a.D, G = a.G, ng = D / G;
    const uint32_t* k4 = krow(th, unit, i, D);
    const uint32_t* v4 = vrow(th, unit, i, D);
    const size_t s4 = srow(th, unit, i, D, G);
    if (G != 32 || 2 * ng > 32) {
        if (lane == 0) {
            quant_row([&](int c) {
                          return dequant(code_at(k4, c, th.k_bits), h2f_bits(th.k_scale[s4 + c / G]),
                                         h2f_bits(th.k_zero[s4 + c / G]));
                      },
                      D, G, tl.k_bits, krow(tl, unit, slot, D), tl.k_scale + srow(tl, unit, slot, D, G),
                      tl.k_zero + srow(tl, unit, slot, D, G));
            quant_row([&](int c) {
                          return dequant(code_at(v4, c, th.v_bits), h2f_bits(th.v_scale[s4 + c / G]),
                                         h2f_bits(th.v_zero[s4 + c / G]));
                      },
                      D, G, tl.v_bits, vrow(tl, unit, slot, D), tl.v_scale + srow(tl, unit, slot, D, G),
                      tl.v_zero + srow(tl, unit, slot, D, G));
            tl.token_id[unit * tl.cap + slot] = th.token_id[unit * th.cap + i];
        }
        return;
    }
    if (lane < 2 * ng) {
        const bool isv = lane >= ng;
        const int grp = isv ? lane - ng : lane;
        const uint32_t* src = isv ? v4 : k4;
        const int sb = isv ? th.v_bits : th.k_bits, db = isv ? tl.v_bits : tl.k_bits;
        const float sc = h2f_bits((isv ? th.v_scale : th.k_scale)[s4 + grp]);
        const float zp = h2f_bits((isv ? th.v_zero : th.k_zero)[s4 + grp]);
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = dequant(code_at(src, grp * 32 + c, sb), sc, zp);
        const QParams q = params32(v, db);
        uint32_t* codes = (isv ? vrow(tl, unit, slot, D) : krow(tl, unit, slot, D)) + grp * db;
        switch (db) {
            case 2: pack32<2>(v, q, codes, 1); break;
            case 4: pack32<4>(v, q, codes, 1); break;
            default: pack32<8>(v, q, codes, 1); break;
        }
        const size_t so = srow(tl, unit, slot, D, G) + grp;
        (isv ? tl.v_scale : tl.k_scale)[so] = q.s_bits;
        (isv ? tl.v_zero : tl.k_zero)[so] = q.z_bits;
    }
    if (lane == 0) tl.token_id[unit * tl.cap + slot] = th.token_id[unit * th.cap + i];
}

// Oldest residual token leaves; the top floor(N_q / hi_den) by cumulative
// score (ties to the lower position) is recomputed; INT4 tokens outside it
// are re-quantised to INT2 from their dequantised values.
// One CTA (any multiple of 32 threads up to 1024) on one unit; `holes` holds the tier-0
// capacity in ints, then (key_cache) the population's keys.
__device__ __forceinline__ void mikv_step_unit(const PolicyArgs& a, size_t unit, int key_cache, int32_t* holes,
                                               MikvShared& sh) {
    const int len = a.res_len[unit];
    if (len <= a.nr) return;
    const int D = a.D, G = a.G, cap = a.res_cap;
    const bool bf = a.bf16 != 0;
    const int start = a.res_start[unit];
    const int e_id = a.res_token_id[unit * cap + start];
    const TierDev& th = a.tier[0];
    const TierDev& tl = a.tier[1];
    const int c0 = th.count[unit], c1 = tl.count[unit];
    const int nq = c0 + c1 + 1;
    const int n4 = nq / a.hi_den;
    const float* cum = a.cum_score + unit * (size_t)a.score_cap;
    auto id_of = [&](int i) -> int {
        return i < c0 ? th.token_id[unit * th.cap + i]
                      : (i < c0 + c1 ? tl.token_id[unit * tl.cap + (i - c0)] : e_id);
    };
    // the ranking keys of the population, gathered once into shared memory when
    // they fit (every pass of the selection then reads them from there)
    uint32_t* kc = reinterpret_cast<uint32_t*>(holes + th.cap);
    int start_shift = 24;                              // the radix digit the selection starts at
    uint32_t kpfx = 0;
    if (key_cache) {
        if (threadIdx.x == 0) {
            sh.kmin = 0xffffffffu;
            sh.kmax = 0u;
        }
        __syncthreads();
        uint32_t mn = 0xffffffffu, mx = 0u;
        for (int i = threadIdx.x; i < nq; i += blockDim.x) {
            const uint32_t kv = orderable(cum[id_of(i)]);
            kc[i] = kv;
            mn = min(mn, kv);
            mx = max(mx, kv);
        }
        mn = __reduce_min_sync(0xffffffffu, mn);
        mx = __reduce_max_sync(0xffffffffu, mx);
        if ((threadIdx.x & 31) == 0) {
            atomicMin(&sh.kmin, mn);
            atomicMax(&sh.kmax, mx);
        }
        __syncthreads();
        // the keys share their leading bits down to the first one where min and max differ:
        // the selection starts at the 8-bit digit holding that bit
        const uint32_t diff = sh.kmin ^ sh.kmax;
        const int lead = diff ? __clz(diff) : 32;
        start_shift = lead >= 32 ? 0 : 24 - 8 * (lead / 8);
        kpfx = sh.kmin;
    }
    auto key = [&](int i) { return key_cache ? kc[i] : orderable(cum[id_of(i)]); };
    uint32_t k1 = 0xffffffffu, t1 = 0;
    uint32_t id_star = 0xffffffffu;                    // ties: position <= id_star are in
    if (n4 > 0) {
        block_radix_select(key, nq, n4, sh.tk, &k1, &t1, start_shift, kpfx);
        if (threadIdx.x == 0) sh.cnt_eq = 0;
        __syncthreads();
        uint32_t local = 0;
        for (int i = threadIdx.x; i < nq; i += blockDim.x) local += key(i) == k1 ? 1u : 0u;
        atomicAdd(&sh.cnt_eq, local);
        __syncthreads();
        const uint32_t cnt_eq = sh.cnt_eq;
        __syncthreads();
        if (t1 < cnt_eq) {
            // among equal scores keep the t1 lowest positions
            uint32_t k2, t2;
            block_radix_select(
                [&](int i) { return key(i) == k1 ? 0xffffffffu - (uint32_t)id_of(i) : 0u; }, nq,
                (int)t1, sh.tk, &k2, &t2);
            id_star = 0xffffffffu - k2;
        }
    }
    auto in_top = [&](int i) -> bool {
        if (n4 == 0) return false;
        const uint32_t kv = key(i);
        return kv > k1 || (kv == k1 && (uint32_t)id_of(i) <= id_star);
    };
    const bool e_in = in_top(nq - 1);
    // demotions: INT4 slots outside the set, in slot order
    uint32_t dem_base = 0;
    const int c0_new_pred = 0;
    (void)c0_new_pred;
    const int lo_first = c1 + (e_in ? 0 : 1);
    // (each chunk's demoted slots are listed in `holes`, free until the hole filling below,
    // then re-quantised one row per warp)
    const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int s0 = 0; s0 < c0; s0 += blockDim.x) {
        const int i = s0 + threadIdx.x;
        const uint32_t dem = (i < c0 && !in_top(i)) ? 1u : 0u;
        uint32_t tot;
        const uint32_t r = block_excl_scan(dem, sh.tk, &tot);
        if (dem) holes[r] = i;                         // tot <= c0 <= the tier-0 capacity
        __syncthreads();
        for (int e = warp; e < (int)tot; e += nwarps) {
            const int slot = lo_first + (int)dem_base + e;
            if (slot < tl.cap) {
                requant_row_warp(a, th, tl, unit, holes[e], slot);
            } else if ((threadIdx.x & 31) == 0) {
                atomicOr(&g_status_policy, kDevCheck);
            }
        }
        __syncthreads();
        dem_base += tot;
    }
    const int n_dem = (int)dem_base;
    const int c0n = c0 - n_dem;
    __syncthreads();
    // fill the holes below c0n with the kept tokens at or above c0n
    uint32_t hole_base = 0;
    for (int s0 = 0; s0 < c0n; s0 += blockDim.x) {
        const int i = s0 + threadIdx.x;
        const uint32_t hole = (i < c0n && !in_top(i)) ? 1u : 0u;
        uint32_t tot;
        const uint32_t r = block_excl_scan(hole, sh.tk, &tot);
        if (hole) holes[hole_base + r] = i;
        hole_base += tot;
    }
    __syncthreads();
    uint32_t mov_base = 0;
    const int kw = D * th.k_bits / 32, vw = D * th.v_bits / 32, ng = D / G;
    for (int s0 = c0n; s0 < c0; s0 += blockDim.x) {
        const int i = s0 + threadIdx.x;
        const uint32_t mov = (i < c0 && in_top(i)) ? 1u : 0u;
        uint32_t tot;
        const uint32_t r = block_excl_scan(mov, sh.tk, &tot);
        if (mov) {
            const int dst = holes[mov_base + r];
            uint32_t* kd = krow(th, unit, dst, D);
            const uint32_t* ks = krow(th, unit, i, D);
            for (int w = 0; w < kw; ++w) kd[w] = ks[w];
            uint32_t* vd = vrow(th, unit, dst, D);
            const uint32_t* vs = vrow(th, unit, i, D);
            for (int w = 0; w < vw; ++w) vd[w] = vs[w];
            const size_t sd = srow(th, unit, dst, D, G), ss = srow(th, unit, i, D, G);
            for (int w = 0; w < ng; ++w) {
                th.k_scale[sd + w] = th.k_scale[ss + w];
                th.k_zero[sd + w] = th.k_zero[ss + w];
                th.v_scale[sd + w] = th.v_scale[ss + w];
                th.v_zero[sd + w] = th.v_zero[ss + w];
            }
            th.token_id[unit * th.cap + dst] = th.token_id[unit * th.cap + i];
        }
        mov_base += tot;
    }
    __syncthreads();
    // the leaving token, quantised from its full-precision values (warp 0)
    if (threadIdx.x < 32) {
        const size_t row = (unit * cap + start) * (size_t)D;
        if (e_in) {
            if (c0n < th.cap) put_token_warp(a, th, unit, c0n, a.res_k, a.res_v, row, e_id);
            else if (threadIdx.x == 0) atomicOr(&g_status_policy, kDevCheck);
        } else {
            if (c1 < tl.cap) put_token_warp(a, tl, unit, c1, a.res_k, a.res_v, row, e_id);
            else if (threadIdx.x == 0) atomicOr(&g_status_policy, kDevCheck);
        }
    }
    if (threadIdx.x == 0) {
        th.count[unit] = min(c0n + (e_in ? 1 : 0), th.cap);
        tl.count[unit] = min(c1 + n_dem + (e_in ? 0 : 1), tl.cap);
        a.res_start[unit] = (start + 1) % cap;
        a.res_len[unit] = len - 1;
    }
    (void)bf;
}

// The same, without the key cache, as one out-of-line copy for the sampled step's fallbacks.
__device__ __noinline__ void mikv_step_general(const PolicyArgs& a, size_t unit, int32_t* holes, MikvShared& sh) {
    mikv_step_unit(a, unit, 0, holes, sh);
}

__global__ void __launch_bounds__(kTopkBlock) mikv_step(PolicyArgs a, int key_cache) {
    __shared__ MikvShared sh;
    extern __shared__ int32_t holes[];
    mikv_step_unit(a, blockIdx.x, key_cache, holes, sh);
}

// ------------------------------------------------- MiKV step by sample selection
//
// MiKV evicts nothing and tokens leave the residual window in position order, so when the
// leaving token is position e = c0 + c1 the population is exactly positions 0 .. e and its
// ranking keys are the first e + 1 cumulative scores, read in order (no gather by token
// id).  The ranking value of position p is R(p) = key(p) * 2^32 + (2^32 - 1 - p): larger
// ranks higher, equal scores go to the lower position, and no two values are equal.  The
// top floor((e + 1) / hi_den) is {R >= R*}, and R* comes from a sample selection:
//  1. a strided sample of 256 keys, ranked in shared memory, gives seven boundary keys around
//     the sample rank where R* is expected;
//  2. one pass counts the keys at or above each boundary, which places R* between two
//     neighbouring boundaries (or above or below all of them) and gives its rank there;
//  3. a second pass (the scores are in L2 by then) gathers the values between those two
//     (the band), and a radix select inside the band gives R* exactly.
// A band larger than its buffer, or a population that is not positions 0 .. e, takes the
// general step above, with the same result.

constexpr int kMikvThreads = 256;
constexpr int kMikvSample = 256;                     // sampled keys (one thread ranks each)
constexpr int kMikvNB = 7;                           // boundaries
constexpr int kMikvStep = 10;                        // sample ranks between boundaries
constexpr int kMikvBand = 4096;                      // band buffer, 64-bit values
static_assert(kMikvSample == kMikvThreads, "one thread per sampled key");
static_assert(2 * kMikvSample * 4 <= kMikvBand * 8, "sample in the band buffer");

struct MikvSampledShared {
    MikvShared gen;
    uint32_t cnt[kMikvNB];                           // keys at or above each boundary
    uint32_t bnd[kMikvNB];                           // the boundary keys, non-increasing
    uint32_t nb_got;
    int bad;
};

// One count per lane with `on` into h[bin], by all 32 lanes of a warp together: lanes that
// share a bin add once (neighbouring positions' scores are close, so a warp's lanes often
// fall into one bin, which would serialise their atomics).
__device__ __forceinline__ void warp_hist_add(uint32_t* h, uint32_t bin, bool on) {
    const uint32_t m = __ballot_sync(0xffffffffu, on);
    if (!m) return;
    const int lane = threadIdx.x & 31;
    const int first = __ffs(m) - 1;
    const uint32_t b0 = __shfl_sync(0xffffffffu, bin, first);
    if (__all_sync(0xffffffffu, !on || bin == b0)) {
        if (lane == first) atomicAdd(&h[b0], (uint32_t)__popc(m));
    } else {
        const uint32_t peers = __match_any_sync(0xffffffffu, on ? bin : 0xffffffffu);
        if (on && lane == __ffs(peers) - 1) atomicAdd(&h[bin], (uint32_t)__popc(peers));
    }
}

// The r-th largest (1 <= r <= n) of n distinct 64-bit values that all lie in [lo, hi]:
// 8-bit digits from the highest bit where lo and hi differ; once the chosen bin holds a
// single value, that value is the answer.
__device__ unsigned long long band_select(const unsigned long long* v, int n, uint32_t r, unsigned long long lo,
                                          unsigned long long hi, TopkShared& sh) {
    const unsigned long long diff = lo ^ hi;
    const int top = diff ? 63 - __clzll((long long)diff) : 0;
    unsigned long long mask = top >= 63 ? 0ull : ~0ull << (top + 1);
    unsigned long long prefix = lo & mask;
    uint32_t remaining = r;
    for (int s_ = top - 7;; s_ -= 8) {
        const int s = s_ < 0 ? 0 : s_;
        for (int i = threadIdx.x; i < 256; i += blockDim.x) sh.hist[i] = 0;
        __syncthreads();
        for (int i0 = 0; i0 < n; i0 += blockDim.x) {
            const int i = i0 + threadIdx.x;
            const unsigned long long x = i < n ? v[i] : 0ull;
            warp_hist_add(sh.hist, (uint32_t)(x >> s) & 255u, i < n && (x & mask) == prefix);
        }
        __syncthreads();
        if (threadIdx.x < 32) radix_pick_bin(sh, remaining);
        __syncthreads();
        const uint32_t bin = sh.bcast[0];
        prefix |= (unsigned long long)bin << s;
        mask |= 255ull << s;
        remaining = sh.bcast[1];
        const uint32_t in_bin = sh.hist[bin];
        __syncthreads();
        if (s == 0) return prefix;
        if (in_bin == 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const unsigned long long x = v[i];
                if ((x & mask) == prefix) {
                    sh.bcast[2] = (uint32_t)(x >> 32);
                    sh.bcast[3] = (uint32_t)x;
                }
            }
            __syncthreads();
            const unsigned long long out = ((unsigned long long)sh.bcast[2] << 32) | sh.bcast[3];
            __syncthreads();
            return out;
        }
    }
}

// Bytes of the front of the sampled step's dynamic shared memory: the band, which later
// holds the demoted slots (or the general step's holes: the tier-0 capacity in ints).
__host__ __device__ __forceinline__ size_t mikv_front_bytes(int cap0) {
    const size_t b = (size_t)kMikvBand * 8, h = (size_t)cap0 * 4;
    return ((b > h ? b : h) + 15) & ~(size_t)15;
}

__device__ __forceinline__ unsigned long long rank_value(float score, int p) {
    return ((unsigned long long)orderable(score) << 32) | (0xffffffffu - (uint32_t)p);
}

// Launched with kMikvThreads threads; dynamic shared memory: mikv_front_bytes (the sample,
// then the band, then the demoted slots or the general step's holes), then one bit per
// tier-0 slot (kept).
__global__ void __launch_bounds__(kMikvThreads, 4) mikv_step_sampled(PolicyArgs a) {
    __shared__ MikvSampledShared sh;
    extern __shared__ __align__(16) uint8_t mikv_dyn[];
    const size_t unit = blockIdx.x;
    const TierDev& th = a.tier[0];
    const TierDev& tl = a.tier[1];
    unsigned long long* band = reinterpret_cast<unsigned long long*>(mikv_dyn);
    int32_t* dem = reinterpret_cast<int32_t*>(mikv_dyn);      // once the band is done with
    uint32_t* keep = reinterpret_cast<uint32_t*>(mikv_dyn + mikv_front_bytes(th.cap));
    const int len = a.res_len[unit];
    if (len <= a.nr) return;
    const int cap = a.res_cap, start = a.res_start[unit];
    const int e_id = a.res_token_id[unit * cap + start];
    const int c0 = th.count[unit], c1 = tl.count[unit];
    const int nq = c0 + c1 + 1;
    const int n4 = nq / a.hi_den;
    if (n4 < 1 || e_id != c0 + c1 || nq > a.score_cap) {
        mikv_step_general(a, unit, dem, sh.gen);
        return;
    }
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const float* cum = a.cum_score + unit * (size_t)a.score_cap;

    // 1. the sample: the key of position floor(j n / S) with its low 8 bits replaced by j
    //    (distinct values; any values serve as edges), ranked in shared memory
    const int S = min(kMikvSample, nq);
    uint32_t* skey = reinterpret_cast<uint32_t*>(band);  // [kMikvSample], zero past S
    uint32_t* srt = skey + kMikvSample;
    skey[tid] = tid < S ? (orderable(cum[(int)(((long long)tid * nq) / S)]) & 0xffffff00u) | (uint32_t)tid : 0u;
    if (tid < kMikvNB) sh.cnt[tid] = 0u;
    if (tid == 0) {
        sh.nb_got = 0;
        sh.bad = 0;
    }
    __syncthreads();
    {
        // this thread's sample rank: the sampled values above it (the zeros past S never are)
        const uint32_t x = skey[tid];
        const uint4* s4 = reinterpret_cast<const uint4*>(skey);
        uint32_t rk = 0;
#pragma unroll 4
        for (int i = 0; i < kMikvSample / 4; ++i) {
            const uint4 y = s4[i];
            rk += (y.x > x ? 1u : 0u) + (y.y > x ? 1u : 0u) + (y.z > x ? 1u : 0u) + (y.w > x ? 1u : 0u);
        }
        if (tid < S) srt[rk] = x;
    }
    __syncthreads();

    // 2. keys at or above each of kMikvNB boundaries: the sample's keys kMikvStep ranks
    //    apart around where R* is expected, counted in registers (no shared-memory traffic
    //    per key).  Positions past the end read as the pattern 0xffffffff, whose key is 0,
    //    below every boundary.
    const int rho = (int)(((long long)n4 * S + nq / 2) / nq);
    uint32_t bnd[kMikvNB], cnt[kMikvNB];
#pragma unroll
    for (int i = 0; i < kMikvNB; ++i) {
        bnd[i] = max(srt[min(max(rho + (i - kMikvNB / 2) * kMikvStep, 0), S - 1)], 1u);
        cnt[i] = 0u;
    }
    if (tid < kMikvNB) sh.bnd[tid] = bnd[tid];
    const uint32_t* cumw = reinterpret_cast<const uint32_t*>(cum);
    constexpr int kU = 16;
    for (int p0 = 0; p0 < nq; p0 += nt * kU) {
        uint32_t w[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int p = p0 + u * nt + tid;
            w[u] = p < nq ? cumw[p] : 0xffffffffu;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const uint32_t kv = orderable(__uint_as_float(w[u]));
#pragma unroll
            for (int i = 0; i < kMikvNB; ++i) cnt[i] += kv >= bnd[i] ? 1u : 0u;
        }
    }
#pragma unroll
    for (int i = 0; i < kMikvNB; ++i) {
        const uint32_t t = __reduce_add_sync(0xffffffffu, cnt[i]);
        if (lane == 0) atomicAdd(&sh.cnt[i], t);
    }
    __syncthreads();
    // the first boundary with at least n4 keys at or above it bounds R* from below, the one
    // before it (if any) from above; the keys between them are the band
    int ib = kMikvNB;
    for (int i = kMikvNB - 1; i >= 0; --i)
        if (sh.cnt[i] >= (uint32_t)n4) ib = i;
    const uint32_t above = ib > 0 ? sh.cnt[ib - 1] : 0u;
    const uint32_t nb = (ib < kMikvNB ? sh.cnt[ib] : (uint32_t)nq) - above;
    const uint32_t r = (uint32_t)n4 - above;           // R*'s rank in the band (1 = largest)
    const uint32_t lo_key = ib < kMikvNB ? sh.bnd[ib] : 0u;
    const unsigned long long hi_key = ib > 0 ? (unsigned long long)sh.bnd[ib - 1] : (1ull << 32);   // exclusive
    if (nb > (uint32_t)kMikvBand || r < 1u || r > nb || hi_key == 0ull) {
        __syncthreads();
        mikv_step_general(a, unit, dem, sh.gen);
        return;
    }

    // 3. the band, then R* inside it
    for (int p0 = 0; p0 < nq; p0 += nt * kU) {
        float v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int p = p0 + u * nt + tid;
            v[u] = p < nq ? cum[p] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int p = p0 + u * nt + tid;
            const uint32_t kv = orderable(v[u]);
            const bool inb = p < nq && kv >= lo_key && (unsigned long long)kv < hi_key;
            const uint32_t bal = __ballot_sync(0xffffffffu, inb);
            if (bal) {
                uint32_t base = 0;
                if (lane == 0) base = atomicAdd(&sh.nb_got, (uint32_t)__popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (inb) {
                    const uint32_t at = base + (uint32_t)__popc(bal & ((1u << lane) - 1u));
                    if (at < (uint32_t)kMikvBand) band[at] = rank_value(v[u], p);
                }
            }
        }
    }
    __syncthreads();
    if (sh.nb_got != nb) {                               // the scores changed under the step
        __syncthreads();
        mikv_step_general(a, unit, dem, sh.gen);
        return;
    }
    const unsigned long long rstar = band_select(band, (int)nb, r, (unsigned long long)lo_key << 32,
                                                 ((hi_key - 1ull) << 32) | 0xffffffffull, sh.gen.tk);

    // INT4 slots still in the top set (one bit per slot), from their positions' scores
    const int nwords = (c0 + 31) >> 5;
    for (int s0 = 0; s0 < c0; s0 += nt * 8) {
        int pid[8];
        float sv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int sl = s0 + u * nt + tid;
            pid[u] = sl < c0 ? th.token_id[unit * th.cap + sl] : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool ok = pid[u] >= 0 && pid[u] < e_id;
            if (s0 + u * nt + tid < c0 && !ok) sh.bad = 1;
            sv[u] = ok ? cum[pid[u]] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool kept = pid[u] >= 0 && pid[u] < e_id && rank_value(sv[u], pid[u]) >= rstar;
            const uint32_t bal = __ballot_sync(0xffffffffu, kept);
            const int wd = ((s0 + u * nt) >> 5) + warp;
            if (lane == 0 && wd < nwords) keep[wd] = bal;
        }
    }
    __syncthreads();
    if (sh.bad) {                                      // a tier-0 token outside positions 0 .. e - 1
        __syncthreads();
        mikv_step_general(a, unit, dem, sh.gen);
        return;
    }
    const bool e_in = rank_value(cum[e_id], e_id) >= rstar;

    // demoted slots in slot order
    uint32_t dem_base = 0;
    for (int w0 = 0; w0 < nwords; w0 += nt) {
        const int w = w0 + tid;
        uint32_t dm = 0u;
        if (w < nwords) {
            const int nv = min(32, c0 - 32 * w);
            dm = ~keep[w] & (nv >= 32 ? 0xffffffffu : ((1u << nv) - 1u));
        }
        uint32_t tot;
        uint32_t at = dem_base + block_excl_scan((uint32_t)__popc(dm), sh.gen.tk, &tot);
        while (dm) {
            dem[at++] = 32 * w + (__ffs(dm) - 1);
            dm &= dm - 1u;
        }
        dem_base += tot;
    }
    __syncthreads();
    const int n_dem = (int)dem_base;
    const int D = a.D, G = a.G;
    // re-quantised to INT2 after the leaving token's tier-1 slot (when it goes there)
    const int lo_first = c1 + (e_in ? 0 : 1);
    for (int e = warp; e < n_dem; e += nw) {
        const int slot = lo_first + e;
        if (slot < tl.cap) requant_row_warp(a, th, tl, unit, dem[e], slot);
        else if (lane == 0) atomicOr(&g_status_policy, kDevCheck);
    }
    __syncthreads();
    // kept slots at or above c0 - n_dem fill the demoted slots below it (a prefix of `dem`)
    const int c0n = c0 - n_dem;
    const int kw = D * th.k_bits / 32, vw = D * th.v_bits / 32, ng = D / G;
    uint32_t mov_base = 0;
    for (int s0 = c0n; s0 < c0; s0 += nt) {
        const int i = s0 + tid;
        const uint32_t mov = (i < c0 && ((keep[i >> 5] >> (i & 31)) & 1u)) ? 1u : 0u;
        uint32_t tot;
        const uint32_t r = block_excl_scan(mov, sh.gen.tk, &tot);
        if (mov) {
            const int dst = dem[mov_base + r];
            uint32_t* kd = krow(th, unit, dst, D);
            const uint32_t* ks = krow(th, unit, i, D);
            for (int w = 0; w < kw; ++w) kd[w] = ks[w];
            uint32_t* vd = vrow(th, unit, dst, D);
            const uint32_t* vs = vrow(th, unit, i, D);
            for (int w = 0; w < vw; ++w) vd[w] = vs[w];
            const size_t sd = srow(th, unit, dst, D, G), ss = srow(th, unit, i, D, G);
            for (int w = 0; w < ng; ++w) {
                th.k_scale[sd + w] = th.k_scale[ss + w];
                th.k_zero[sd + w] = th.k_zero[ss + w];
                th.v_scale[sd + w] = th.v_scale[ss + w];
                th.v_zero[sd + w] = th.v_zero[ss + w];
            }
            th.token_id[unit * th.cap + dst] = th.token_id[unit * th.cap + i];
        }
        mov_base += tot;
    }
    __syncthreads();
    // the leaving token, quantised from its full-precision values (warp 0)
    if (tid < 32) {
        const size_t row = (unit * cap + start) * (size_t)D;
        if (e_in) {
            if (c0n < th.cap) put_token_warp(a, th, unit, c0n, a.res_k, a.res_v, row, e_id);
            else if (tid == 0) atomicOr(&g_status_policy, kDevCheck);
        } else {
            if (c1 < tl.cap) put_token_warp(a, tl, unit, c1, a.res_k, a.res_v, row, e_id);
            else if (tid == 0) atomicOr(&g_status_policy, kDevCheck);
        }
    }
    if (tid == 0) {
        th.count[unit] = min(c0n + (e_in ? 1 : 0), th.cap);
        tl.count[unit] = min(c1 + n_dem + (e_in ? 0 : 1), tl.cap);
        a.res_start[unit] = (start + 1) % cap;
        a.res_len[unit] = len - 1;
    }
}

PolicyArgs make_args(const kvq_cache& c, const kvq_policy_params* p) {
    PolicyArgs a{};
    a.B = c.B;
    a.Hq = c.Hq;
    a.Hkv = c.Hkv;
    a.D = c.D;
    a.G = c.G;
    a.g = c.Hq / c.Hkv;
    a.bf16 = c.dtype == KVQ_BF16;
    a.n_tiers = c.n_tiers;
    a.nr = c.nr;
    a.hi_den = c.hi_den;
    for (int t = 0; t < c.n_tiers; ++t) {
        const kvq_tier& s = c.tier[t];
        TierDev& d = a.tier[t];
        d.k_bits = s.k_bits;
        d.v_bits = s.v_bits;
        d.k_axis = s.k_axis;
        d.cap = s.cap;
        d.k_codes = s.k_codes;
        d.k_scale = s.k_scale;
        d.k_zero = s.k_zero;
        d.v_codes = s.v_codes;
        d.v_scale = s.v_scale;
        d.v_zero = s.v_zero;
        d.token_id = s.token_id;
        d.count = s.count;
        d.page_table = s.page_table;
        d.page_owner = s.page_owner;
        d.free_ring = s.free_ring;
        d.ring_ctr = s.ring_ctr;
        d.max_pages = s.max_pages;
        d.n_pages = s.n_pages;
    }
    a.res_k = c.res_k;
    a.res_v = c.res_v;
    a.res_token_id = c.res_token_id;
    a.res_start = c.res_start;
    a.res_len = c.res_len;
    a.res_cap = c.res_cap;
    a.seq_len = c.seq_len;
    a.win_acc = c.win_acc;
    a.alpha = c.alpha;
    a.cum_score = c.cum_score;
    a.score_cap = c.score_cap;
    if (p) {
        a.k_src = p->k_src;
        a.v_src = p->v_src;
        a.T = p->T;
        a.sel_idx = p->sel_idx;
        a.n_sel = p->n_sel;
        a.colscore = p->colscore;
        a.n_high = p->n_high;
        a.n_low = p->n_low;
    }
    return a;
}

kvq_status launched(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("requant_demote (%s): %s", what, cudaGetErrorString(e));
        return KVQ_ECUDA;
    }
    return KVQ_OK;
}

}  // namespace

template <typename T>
static cudaError_t launch_fused_t(const PolicyArgs& a, int units, int kb, int vb, const float* score,
                                  const int32_t* k_hh, int kmax, int w, int32_t* idx_out, cudaStream_t s) {
    const size_t smem = (size_t)(kmax + w) * sizeof(int32_t);
    auto go = [&](auto kern) -> cudaError_t {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        kern<<<units, kTopkBlock, smem, s>>>(a, score, k_hh, kmax, w, idx_out);
        return cudaGetLastError();
    };
    if (kb == 2 && vb == 2) return go(minikv_fused_build<T, 2, 2>);
    if (kb == 4 && vb == 4) return go(minikv_fused_build<T, 4, 4>);
    if (kb == 4 && vb == 2) return go(minikv_fused_build<T, 4, 2>);
    return cudaErrorInvalidValue;
}

kvq_status run_minikv_fused_build(const kvq_cache& c, const void* k, const void* v, int T, const float* score,
                                  const int32_t* k_hh, int kmax, int w, int32_t* idx_out, cudaStream_t s) {
    kvq_policy_params p{};
    p.k_src = k;
    p.v_src = v;
    p.T = T;
    PolicyArgs a = make_args(c, &p);
    const int units = c.B * c.Hkv;
    const kvq_tier& t = c.tier[0];
    cudaError_t e = c.dtype == KVQ_BF16
                        ? launch_fused_t<__nv_bfloat16>(a, units, t.k_bits, t.v_bits, score, k_hh, kmax, w, idx_out, s)
                        : launch_fused_t<__half>(a, units, t.k_bits, t.v_bits, score, k_hh, kmax, w, idx_out, s);
    if (e != cudaSuccess) {
        set_error("minikv_prefill_build launch: %s", cudaGetErrorString(e));
        return KVQ_ECUDA;
    }
    return KVQ_OK;
}

kvq_status run_pages_init(const kvq_cache& c, cudaStream_t s) {
    PolicyArgs a = make_args(c, nullptr);
    pages_init_kernel<<<152, 256, 0, s>>>(a);
    return launched("kvq_pages_init");
}

kvq_status run_pages_release(const kvq_cache& c, const int32_t* mask, cudaStream_t s) {
    PolicyArgs a = make_args(c, nullptr);
    pages_release_kernel<<<1, kTopkBlock, 0, s>>>(a, mask);
    return launched("kvq_pages_release");
}

kvq_status run_policy(const kvq_cache& c, int mode, const kvq_policy_params* p, int step,
                      cudaStream_t s) {
    const int units = c.B * c.Hkv;
    PolicyArgs a = make_args(c, p);
    if (mode == KVQ_POLICY_MINIKV) {
        if (step == 0) {
            const int n = p->n_sel, nr = c.nr, G = c.G;
            const int r0 = n <= nr ? n : nr + (n - nr) % G;
            const int npk = n - r0;
            const kvq_tier& t = c.tier[0];
            cudaError_t e = launch_quant_pack_strided(p->k_src, c.dtype, units, p->T, c.D, p->sel_idx, n,
                                                      npk, t.k_bits, G, KVQ_AXIS_CHANNEL, t.cap,
                                                      t.k_codes, t.k_scale, t.k_zero, s);
            if (e == cudaSuccess)
                e = launch_quant_pack_strided(p->v_src, c.dtype, units, p->T, c.D, p->sel_idx, n, npk,
                                              t.v_bits, G, KVQ_AXIS_TOKEN, t.cap, t.v_codes, t.v_scale,
                                              t.v_zero, s);
            if (e != cudaSuccess) {
                set_error("requant_demote (MiniKV pack): %s", cudaGetErrorString(e));
                return KVQ_ECUDA;
            }
            minikv_build_tail<<<dim3(units, (unsigned)std::max(1, (r0 + kTailRows - 1) / kTailRows)),
                                kTailRows * 32, 0, s>>>(a, npk, r0);
            return launched("MiniKV build");
        }
        // the residual flush runs inside decode_attn_qkv (its last step)
        return KVQ_OK;
    }
    if (mode == KVQ_POLICY_DIFFKV) {
        if (step == 0) {
            if (c.tier[0].page_table || c.tier[1].page_table) pages_build_alloc<<<1, kTopkBlock, 0, s>>>(a);
            diffkv_build<<<units, kTopkBlock, 0, s>>>(a);
            return launched("DiffKV build");
        }
        diffkv_exit<<<units, 32, 0, s>>>(a);
        return launched("DiffKV exit");
    }
    if (step == 0) {
        mikv_build<<<units, kTopkBlock, 0, s>>>(a);
        return launched("MiKV build");
    }
    constexpr size_t kMaxDyn = 200 * 1024;
    const size_t cap0 = (size_t)c.tier[0].cap;
    const size_t dyn_s = mikv_front_bytes((int)cap0) + (cap0 + 31) / 32 * sizeof(uint32_t);
    if (dyn_s <= kMaxDyn) {
        if (dyn_s > 48 * 1024) {
            static bool attr_s = false;
            if (!attr_s) {
                cudaFuncSetAttribute(mikv_step_sampled, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDyn);
                attr_s = true;
            }
        }
        mikv_step_sampled<<<units, kMikvThreads, dyn_s, s>>>(a);
        return launched("MiKV step");
    }
    // holes of tier 0, then the population's keys when both fit in shared memory
    const size_t holes = (size_t)c.tier[0].cap * sizeof(int32_t);
    const size_t keys = ((size_t)c.tier[0].cap + c.tier[1].cap + 1) * sizeof(uint32_t);
    const int key_cache = holes + keys <= kMaxDyn ? 1 : 0;
    const size_t dyn = key_cache ? holes + keys : holes;
    if (dyn > 48 * 1024) {
        static bool attr = false;
        if (!attr) {
            cudaFuncSetAttribute(mikv_step, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDyn);
            attr = true;
        }
    }
    mikv_step<<<units, kTopkBlock, dyn, s>>>(a, key_cache);
    return launched("MiKV step");
}

}  // namespace kvq
