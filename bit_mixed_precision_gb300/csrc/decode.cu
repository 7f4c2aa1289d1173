// decode_attn_qkv: one decode step of attention over the compressed cache,
// dequantising packed codes inside the kernel (MiKV rebuttal, the INTn x
// FP16 GEMV paragraph: on-the-fly dequantisation; MiniKV verdict JSON
// forward_implications: fused dequantisation kernels during decoding).
//
// One launch per step.  Grid = (token chunks of every tier and of the
// residual ring, units).  A CTA first requests every byte of its chunk with
// bulk asynchronous copies into shared memory (one mbarrier), then its
// four warps take 32-token groups: keys -> base-2 logits for the g query
// heads of the KV head, online softmax per warp, P.V with the codes turned
// into floats by one rotate and one LOP3 each.  The CTA writes its partial
// (max, sum, unnormalised output); the last CTA of a unit (atomic counter)
// merges the partials, writes o and lse, adds this step's attention to the
// policy scores (DiffKV: per ring slot and query head; MiKV: per token,
// summed over the group) and advances the residual length; the last CTA of
// the grid advances seq_len.  Tiers are read where they lie (MiKV rebuttal:
// attention is permutation invariant, so each precision group sits in its
// own region).
#include <algorithm>
#include <mutex>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "pack_device.cuh"

namespace kvq {

KVQ_DEFINE_STATUS(decode)

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kSub = 128;        // packed tokens per staged sub-chunk: one 32-token group per warp
constexpr int kMaxSubs = 4;      // sub-chunks per CTA at most, streamed through two staging buffers
constexpr int kResChunk = 32;    // residual tokens per CTA (full-precision rows are large)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

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
    int chunks;                 // ceil(cap / chunk_tokens)
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
    uint32_t stage_bytes;       // one staging buffer (two per CTA)
    int chunk_tokens;           // packed tokens per CTA: kSub * (1 .. kMaxSubs)
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

// Code i (KB bits) of a packed word as the float 1 + c * 2^-KB: one rotate
// moves the code to the top of the mantissa, one LOP3 masks it and sets the
// exponent of 1.0.  fma(x, y, acc) adds y + c * y * 2^-KB; the constant y
// is removed once per dot product and the result scaled by 2^KB.
template <int KB>
__device__ __forceinline__ float code_f(uint32_t w, int i) {
    const int rot = ((23 - KB - KB * i) % 32 + 32) % 32;
    const uint32_t x = __funnelshift_l(w, w, rot);
    constexpr uint32_t mask = ((1u << KB) - 1u) << (23 - KB);
    return __uint_as_float((x & mask) | 0x3F800000u);
}

// 32 lanes each hold v[0..31]; afterwards lane t returns the sum over lanes of v[t].
__device__ __forceinline__ float reduce_scatter32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = up ? v[i] : v[i + s];
            const float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

template <int NG, int D>
struct Smem {
    float q[NG][D];                      // query rows, pre-scaled to base-2 logits
    float wm[kWarps][NG];
    float wl[kWarps][NG];
    float wo[kWarps][NG][D];
    float lg[kWarps][NG][32];            // logits of the warp's current group
    unsigned long long bar[2];           // one staging mbarrier per buffer
    int n_total, last;
};

// Online-softmax state of one warp for NG heads; o holds the lane's share.
template <int NG, int NO>
struct WarpAcc {
    float m[NG], l[NG];
    float o[NG][NO];
    float off[NG], zs[NG];               // packed V: sum p*s and sum p*z over this lane's tokens
};

template <int NG, int NO>
__device__ __forceinline__ void acc_init(WarpAcc<NG, NO>& acc) {
#pragma unroll
    for (int h = 0; h < NG; ++h) {
        acc.m[h] = kNegInf;
        acc.l[h] = 0.0f;
        acc.off[h] = 0.0f;
        acc.zs[h] = 0.0f;
#pragma unroll
        for (int i = 0; i < NO; ++i) acc.o[h][i] = 0.0f;
    }
}

// Logits of the group (lane t holds token t, -inf past nt) -> rescale the
// accumulators, return p_h(t) in lg and write the logits out when asked.
template <int NG, int NO>
__device__ __forceinline__ void group_softmax(WarpAcc<NG, NO>& acc, float (&lg)[NG], int nt,
                                              float* lg_out, int slots) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 0; h < NG; ++h) {
        const float s = lane < nt ? lg[h] : kNegInf;
        if (lg_out && lane < nt) lg_out[(size_t)h * slots + lane] = s;
        const float mn = fmaxf(acc.m[h], warp_max(s));
        const float corr = acc.m[h] == kNegInf ? 0.0f : ex2_approx(acc.m[h] - mn);
        const float p = lane < nt ? ex2_approx(s - mn) : 0.0f;
        acc.l[h] = acc.l[h] * corr + warp_sum(p);
#pragma unroll
        for (int i = 0; i < NO; ++i) acc.o[h][i] *= corr;
        acc.off[h] *= corr;
        acc.zs[h] *= corr;
        acc.m[h] = mn;
        lg[h] = p;
    }
}

// ---- shared-memory staging: every byte a CTA needs is requested at once

// One chunk of packed tokens in shared memory, indexed from the chunk start.
struct View {
    const uint32_t* kc;   // CHANNEL keys: [n/per][D]; TOKEN keys: [n][D*KB/32]
    const uint16_t* ks;   // CHANNEL keys: [n/G][D];   TOKEN keys: [n][D/G]
    const uint16_t* kz;
    const uint32_t* vc;   // [n][D*VB/32]
    const uint16_t* vs;   // [n][D/G]
    const uint16_t* vz;
};

__host__ __device__ __forceinline__ uint32_t a16(uint32_t x) { return (x + 15u) & ~15u; }

// Byte sizes of the six arrays of a staged tier chunk of npad tokens.
struct StageSizes {
    uint32_t kc, ks, vc, vs;
    __host__ __device__ uint32_t total() const { return a16(kc) + 2 * a16(ks) + a16(vc) + 2 * a16(vs); }
};

__host__ __device__ inline StageSizes tier_stage_sizes(int k_axis, int kb, int vb, int npad, int D, int G) {
    StageSizes z;
    if (k_axis == KVQ_AXIS_CHANNEL) {
        z.kc = (uint32_t)(npad / (32 / kb)) * D * 4;
        z.ks = (uint32_t)(npad / G) * D * 2;
    } else {
        z.kc = (uint32_t)npad * (D * kb / 8);
        z.ks = (uint32_t)npad * (D / G) * 2;
    }
    z.vc = (uint32_t)npad * (D * vb / 8);
    z.vs = (uint32_t)npad * (D / G) * 2;
    return z;
}

__device__ __forceinline__ View tier_view(const TierArgs& t, int npad, int D, int G, const uint8_t* buf) {
    const StageSizes z = tier_stage_sizes(t.k_axis, t.k_bits, t.v_bits, npad, D, G);
    const uint32_t o_ks = a16(z.kc), o_kz = o_ks + a16(z.ks), o_vc = o_kz + a16(z.ks);
    const uint32_t o_vs = o_vc + a16(z.vc), o_vz = o_vs + a16(z.vs);
    View v;
    v.kc = reinterpret_cast<const uint32_t*>(buf);
    v.ks = reinterpret_cast<const uint16_t*>(buf + o_ks);
    v.kz = reinterpret_cast<const uint16_t*>(buf + o_kz);
    v.vc = reinterpret_cast<const uint32_t*>(buf + o_vc);
    v.vs = reinterpret_cast<const uint16_t*>(buf + o_vs);
    v.vz = reinterpret_cast<const uint16_t*>(buf + o_vz);
    return v;
}

// Called by one thread: the six bulk copies of tokens [j0, j0 + npad) of a tier.
__device__ void stage_tier(const TierArgs& t, size_t unit, int j0, int npad, int D, int G,
                           const uint8_t* buf, uint32_t bar) {
    const StageSizes z = tier_stage_sizes(t.k_axis, t.k_bits, t.v_bits, npad, D, G);
    const void *kc_src, *ks_src, *kz_src;
    if (t.k_axis == KVQ_AXIS_CHANNEL) {
        const int per = 32 / t.k_bits;
        kc_src = t.k_codes + (unit * (size_t)(t.cap / per) + j0 / per) * D;
        const size_t so = (unit * (size_t)(t.cap / G) + j0 / G) * D;
        ks_src = t.k_scale + so;
        kz_src = t.k_zero + so;
    } else {
        kc_src = t.k_codes + (unit * (size_t)t.cap + j0) * (D * t.k_bits / 32);
        const size_t so = (unit * (size_t)t.cap + j0) * (D / G);
        ks_src = t.k_scale + so;
        kz_src = t.k_zero + so;
    }
    const size_t vo = unit * (size_t)t.cap + j0;
    const uint32_t o_ks = a16(z.kc), o_kz = o_ks + a16(z.ks), o_vc = o_kz + a16(z.ks);
    const uint32_t o_vs = o_vc + a16(z.vc), o_vz = o_vs + a16(z.vs);
    const uint32_t d = smem_u32(buf);
    mbar_expect_tx(bar, z.kc + 2 * z.ks + z.vc + 2 * z.vs);
    bulk_load(d, kc_src, z.kc, bar);
    bulk_load(d + o_ks, ks_src, z.ks, bar);
    bulk_load(d + o_kz, kz_src, z.ks, bar);
    bulk_load(d + o_vc, t.v_codes + vo * (D * t.v_bits / 32), z.vc, bar);
    bulk_load(d + o_vs, t.v_scale + vo * (D / G), z.vs, bar);
    bulk_load(d + o_vz, t.v_zero + vo * (D / G), z.vs, bar);
}

// Called by one thread: residual rows [j0, j0 + n) in logical order (oldest
// first, the new token last) as [n][D] 16-bit rows, K at buf, V at
// buf + a16(n * D * 2).
__device__ void stage_residual(const DecodeArgs& a, size_t unit, int len, int start, int j0, int n,
                               int D, const uint8_t* buf, uint32_t bar) {
    const uint32_t row = (uint32_t)D * 2;
    const uint32_t d = smem_u32(buf), dv = d + a16((uint32_t)n * row);
    const int cap = a.res_cap;
    mbar_expect_tx(bar, 2u * (uint32_t)n * row);
    const int n_old = max(0, min(j0 + n, len) - j0);
    const int first = (start + j0) % cap;
    const int seg1 = min(n_old, cap - first), seg2 = n_old - seg1;
    const uint16_t* rk = reinterpret_cast<const uint16_t*>(a.res_k) + unit * (size_t)cap * D;
    const uint16_t* rv = reinterpret_cast<const uint16_t*>(a.res_v) + unit * (size_t)cap * D;
    if (seg1 > 0) {
        bulk_load(d, rk + (size_t)first * D, seg1 * row, bar);
        bulk_load(dv, rv + (size_t)first * D, seg1 * row, bar);
    }
    if (seg2 > 0) {
        bulk_load(d + seg1 * row, rk, seg2 * row, bar);
        bulk_load(dv + seg1 * row, rv, seg2 * row, bar);
    }
    if (len >= j0 && len < j0 + n) {
        const uint32_t r = (uint32_t)(len - j0) * row;
        bulk_load(d + r, reinterpret_cast<const uint16_t*>(a.k_new) + unit * (size_t)D, row, bar);
        bulk_load(dv + r, reinterpret_cast<const uint16_t*>(a.v_new) + unit * (size_t)D, row, bar);
    }
}

// ---- key paths: each leaves this lane's token logit (base 2) for every head

// Keys grouped per channel (packed along tokens): lane owns CPL channels;
// partial dot products of 32 tokens, then a reduce-scatter across lanes.
template <int KB, int CPL, int NG>
__device__ __forceinline__ void logits_channel(const View& v, int tl, const Smem<NG, CPL * 32>& sm,
                                               int G, float (&lg)[NG]) {
    constexpr int D = CPL * 32;
    constexpr int per = 32 / KB;          // tokens per word
    constexpr int rows = 32 / per;        // word rows per 32-token group
    const int lane = threadIdx.x & 31;
    const int c0 = lane * CPL;
    float s[CPL], z[CPL];
#pragma unroll
    for (int ci = 0; ci < CPL; ++ci) {
        s[ci] = h2f_bits(v.ks[(tl / G) * D + c0 + ci]);
        z[ci] = h2f_bits(v.kz[(tl / G) * D + c0 + ci]);
    }
    uint32_t w[rows][CPL];
    const uint32_t* base = v.kc + (size_t)(tl / per) * D + c0;
#pragma unroll
    for (int r = 0; r < rows; ++r) {
        if (CPL == 4) {
            const uint4 v4 = *reinterpret_cast<const uint4*>(base + (size_t)r * D);
            w[r][0] = v4.x; w[r][1] = v4.y; w[r][2] = v4.z; w[r][3] = v4.w;
        } else {
            const uint2 v2 = *reinterpret_cast<const uint2*>(base + (size_t)r * D);
            w[r][0] = v2.x; w[r][CPL - 1] = v2.y;
        }
    }
#pragma unroll 1
    for (int h = 0; h < NG; ++h) {
        float qs[CPL], off = 0.0f, bias = 0.0f;
#pragma unroll
        for (int ci = 0; ci < CPL; ++ci) {
            const float qv = sm.q[h][c0 + ci];
            qs[ci] = qv * s[ci];
            off += qs[ci];
            bias = fmaf(qv, z[ci], bias);
        }
        float part[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) part[k] = 0.0f;
#pragma unroll
        for (int r = 0; r < rows; ++r)
#pragma unroll
            for (int ci = 0; ci < CPL; ++ci)
#pragma unroll
                for (int i = 0; i < per; ++i)
                    part[r * per + i] = fmaf(code_f<KB>(w[r][ci], i), qs[ci], part[r * per + i]);
        const float raw = reduce_scatter32(part);
        lg[h] = (raw - warp_sum(off)) * (float)(1 << KB) + warp_sum(bias);
    }
}

// Keys grouped per token (packed along channels): lane owns one word of a
// token row; dot over the word, scaled by the token's group scale, summed
// over the lanes of the token.
template <int KB, int D, int NG>
__device__ __forceinline__ void logits_token(const View& v, int tl, Smem<NG, D>& sm, int G,
                                             float (&lg)[NG]) {
    constexpr int lpt = D * KB / 32;      // words (lanes) per token
    constexpr int tpp = 32 / lpt;         // tokens per pass
    constexpr int cpw = 32 / KB;          // channels per word
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wi = lane % lpt, to = lane / lpt;
    const int c0 = wi * cpw, grp = c0 / G;
    float qsum[NG];
#pragma unroll
    for (int h = 0; h < NG; ++h) {
        qsum[h] = 0.0f;
#pragma unroll
        for (int i = 0; i < cpw; ++i) qsum[h] += sm.q[h][c0 + i];
    }
#pragma unroll 4
    for (int ps = 0; ps < lpt; ++ps) {
        const int tk = ps * tpp + to;
        const int row = tl + tk;
        const uint32_t w = v.kc[(size_t)row * lpt + wi];
        const float sc = h2f_bits(v.ks[row * (D / G) + grp]);
        const float zc = h2f_bits(v.kz[row * (D / G) + grp]);
        float c[NG];
#pragma unroll
        for (int h = 0; h < NG; ++h) {
            float d = 0.0f;
#pragma unroll
            for (int i = 0; i < cpw; ++i) d = fmaf(code_f<KB>(w, i), sm.q[h][c0 + i], d);
            c[h] = fmaf(sc * (float)(1 << KB), d - qsum[h], zc * qsum[h]);
        }
#pragma unroll
        for (int h = 0; h < NG; ++h) {
#pragma unroll
            for (int o = lpt / 2; o; o >>= 1) c[h] += __shfl_xor_sync(0xffffffffu, c[h], o);
            if (wi == 0) sm.lg[warp][h][tk] = c[h];
        }
    }
    __syncwarp();
#pragma unroll
    for (int h = 0; h < NG; ++h) lg[h] = sm.lg[warp][h][lane];
    __syncwarp();
}

// ---- value paths

// Values grouped per token: lane owns word wi of the tokens to, to + tpp, ...
template <int VB, int D, int NG>
__device__ __forceinline__ void values_token(const View& v, int tl, int nt, const float (&p)[NG],
                                             int G, WarpAcc<NG, 32 / VB>& acc) {
    constexpr int lpt = D * VB / 32, tpp = 32 / lpt, cpw = 32 / VB;
    const int lane = threadIdx.x & 31;
    const int wi = lane % lpt, to = lane / lpt;
    const int grp = (wi * cpw) / G;
#pragma unroll 4
    for (int ps = 0; ps < lpt; ++ps) {
        const int tk = ps * tpp + to;
        float pk[NG];
#pragma unroll
        for (int h = 0; h < NG; ++h) pk[h] = __shfl_sync(0xffffffffu, p[h], tk);
        if (tk < nt) {
            const int row = tl + tk;
            const uint32_t w = v.vc[(size_t)row * lpt + wi];
            const float sc = h2f_bits(v.vs[row * (D / G) + grp]);
            const float zc = h2f_bits(v.vz[row * (D / G) + grp]);
#pragma unroll
            for (int h = 0; h < NG; ++h) {
                const float psc = pk[h] * sc;
                acc.off[h] += psc;
                acc.zs[h] = fmaf(pk[h], zc, acc.zs[h]);
#pragma unroll
                for (int i = 0; i < cpw; ++i) acc.o[h][i] = fmaf(code_f<VB>(w, i), psc, acc.o[h][i]);
            }
        }
    }
}

// Finish a packed-V warp: remove the constants, sum the lanes that share a
// word, publish to smem.
template <int VB, int D, int NG>
__device__ __forceinline__ void finish_token_values(WarpAcc<NG, 32 / VB>& acc, Smem<NG, D>& sm) {
    constexpr int lpt = D * VB / 32, cpw = 32 / VB;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wi = lane % lpt, to = lane / lpt;
#pragma unroll
    for (int h = 0; h < NG; ++h)
#pragma unroll
        for (int i = 0; i < cpw; ++i) {
            float x = (acc.o[h][i] - acc.off[h]) * (float)(1 << VB) + acc.zs[h];
#pragma unroll
            for (int o = lpt; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (to == 0) sm.wo[warp][h][wi * cpw + i] = x;
        }
}

// ---- residual (full precision ring + the new token), staged as [n][D] rows

template <int CPL>
__device__ __forceinline__ void row_vals(const uint16_t* row, bool bf, float (&x)[CPL]) {
    if (CPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(row);
        const uint32_t e[2] = {u.x, u.y};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float2 f = bf ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&e[k]))
                                : __half22float2(*reinterpret_cast<const __half2*>(&e[k]));
            x[2 * k] = f.x;
            x[2 * k + 1] = f.y;
        }
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(row);
        const float2 f = bf ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u))
                            : __half22float2(*reinterpret_cast<const __half2*>(&u));
        x[0] = f.x;
        x[CPL - 1] = f.y;
    }
}

template <int NG, int D>
__device__ void warp_residual(const DecodeArgs& a, Smem<NG, D>& sm, const uint16_t* rk,
                              const uint16_t* rv, int n, float* lg_out) {
    constexpr int CPL = D / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c0 = lane * CPL;
    const bool bf = a.bf16 != 0;
    WarpAcc<NG, CPL> acc;
    acc_init(acc);
    for (int gi = warp; gi * 32 < n; gi += kWarps) {
        const int tl = gi * 32;
        const int nt = min(32, n - tl);
        float lg[NG];
#pragma unroll 1
        for (int h = 0; h < NG; ++h) {
            float part[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                part[k] = 0.0f;
                if (k < nt) {
                    float x[CPL];
                    row_vals<CPL>(rk + (size_t)(tl + k) * D + c0, bf, x);
#pragma unroll
                    for (int ci = 0; ci < CPL; ++ci) part[k] = fmaf(sm.q[h][c0 + ci], x[ci], part[k]);
                }
            }
            lg[h] = reduce_scatter32(part);
        }
        group_softmax(acc, lg, nt, lg_out ? lg_out + tl : nullptr, a.slots);
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            if (k < nt) {
                float x[CPL];
                row_vals<CPL>(rv + (size_t)(tl + k) * D + c0, bf, x);
#pragma unroll
                for (int h = 0; h < NG; ++h) {
                    const float pk = __shfl_sync(0xffffffffu, lg[h], k);
#pragma unroll
                    for (int ci = 0; ci < CPL; ++ci) acc.o[h][ci] = fmaf(pk, x[ci], acc.o[h][ci]);
                }
            }
        }
    }
#pragma unroll
    for (int h = 0; h < NG; ++h) {
        if (lane == 0) {
            sm.wm[warp][h] = acc.m[h];
            sm.wl[warp][h] = acc.l[h];
        }
#pragma unroll
        for (int ci = 0; ci < CPL; ++ci) sm.wo[warp][h][c0 + ci] = acc.o[h][ci];
    }
}

// A chunk of up to chunk_tokens tokens of one tier, streamed in kSub-token
// sub-chunks through the two staging buffers: sub-chunk k + 2 is requested
// as soon as sub-chunk k has been consumed.  Warp w takes the w-th 32-token
// group of every sub-chunk; its online-softmax state spans the sub-chunks.
template <int KB, int KAX, int VB, int D, int NG>
__device__ void warp_tier(const DecodeArgs& a, Smem<NG, D>& sm, const TierArgs& t, size_t unit,
                          int j0, int n_total, uint8_t* stage_base, float* lg_out) {
    constexpr int cpw = 32 / VB;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nsub = (n_total + kSub - 1) / kSub;
    WarpAcc<NG, cpw> acc;
    acc_init(acc);
    bool ok = true;
    for (int sub = 0; sub < nsub; ++sub) {
        const int buf = sub & 1;
        uint8_t* stage = stage_base + (size_t)buf * a.stage_bytes;
        const int n = min(kSub, n_total - sub * kSub);
        ok = ok && __syncthreads_and(mbar_wait(smem_u32(&sm.bar[buf]), (sub >> 1) & 1, nullptr));
        if (ok) {
            const View v = tier_view(t, (n + 31) & ~31, D, a.G, stage);
            const int tl = warp * 32;
            if (tl < n) {
                const int nt = min(32, n - tl);
                float lg[NG];
                if (KAX == KVQ_AXIS_CHANNEL)
                    logits_channel<KB, D / 32, NG>(v, tl, sm, a.G, lg);
                else
                    logits_token<KB, D, NG>(v, tl, sm, a.G, lg);
                group_softmax(acc, lg, nt, lg_out ? lg_out + sub * kSub + tl : nullptr, a.slots);
                values_token<VB, D, NG>(v, tl, nt, lg, a.G, acc);
            }
        }
        __syncthreads();                       // buffer consumed by every warp
        if (threadIdx.x == 0 && sub + 2 < nsub) {
            const int n2 = min(kSub, n_total - (sub + 2) * kSub);
            stage_tier(t, unit, j0 + (sub + 2) * kSub, (n2 + 31) & ~31, D, a.G, stage,
                       smem_u32(&sm.bar[buf]));
        }
    }
    if (!ok && threadIdx.x == 0) atomicOr(&g_status_decode, kDevTimeout);
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < NG; ++h) {
            sm.wm[warp][h] = acc.m[h];
            sm.wl[warp][h] = acc.l[h];
        }
    }
    finish_token_values<VB, D, NG>(acc, sm);
}

template <int NG, int D>
__device__ bool dispatch_tier(const DecodeArgs& a, Smem<NG, D>& sm, const TierArgs& t, size_t unit,
                              int j0, int n, uint8_t* stage, float* lg_out) {
    const int kb = t.k_bits, vb = t.v_bits, ax = t.k_axis;
    if (ax == KVQ_AXIS_CHANNEL && kb == 2 && vb == 2) { warp_tier<2, KVQ_AXIS_CHANNEL, 2, D, NG>(a, sm, t, unit, j0, n, stage, lg_out); return true; }
    if (D == 128) {
        if (ax == KVQ_AXIS_TOKEN && kb == 8 && vb == 4) { warp_tier<8, KVQ_AXIS_TOKEN, 4, D, NG>(a, sm, t, unit, j0, n, stage, lg_out); return true; }
        if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 2) { warp_tier<4, KVQ_AXIS_TOKEN, 2, D, NG>(a, sm, t, unit, j0, n, stage, lg_out); return true; }
        if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 4) { warp_tier<4, KVQ_AXIS_TOKEN, 4, D, NG>(a, sm, t, unit, j0, n, stage, lg_out); return true; }
        if (ax == KVQ_AXIS_TOKEN && kb == 2 && vb == 2) { warp_tier<2, KVQ_AXIS_TOKEN, 2, D, NG>(a, sm, t, unit, j0, n, stage, lg_out); return true; }
    }
    return false;
}

// Grid = (chunks of every tier and of the residual ring, units).
template <int NG, int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem<NG, D>& sm = *reinterpret_cast<Smem<NG, D>*>(smem_raw);
    uint8_t* stage_base = smem_raw + ((sizeof(Smem<NG, D>) + 127) & ~(size_t)127);
    const size_t unit = blockIdx.y;
    const int units = gridDim.y;
    const int TC = a.total_chunks;
    const int b = (int)(unit / a.Hkv), hkv = (int)(unit % a.Hkv);
    const bool bf = a.bf16 != 0;

    int chunk = blockIdx.x, tier = -1;
    for (int t = 0; t < a.n_tiers; ++t) {
        if (chunk < a.tier[t].chunks) { tier = t; break; }
        chunk -= a.tier[t].chunks;
    }
    // thread 0 requests the first bytes before anything else
    if (threadIdx.x == 0) {
        const uint32_t b0 = smem_u32(&sm.bar[0]), b1 = smem_u32(&sm.bar[1]);
        mbar_init(b0, 1);
        mbar_init(b1, 1);
        fence_mbar_init();
        int n = 0;
        if (tier >= 0) {
            const TierArgs& t = a.tier[tier];
            const int raw = t.count[unit];
            if (raw > t.cap || raw < 0) atomicOr(&g_status_decode, kDevCheck);
            const int j0 = chunk * a.chunk_tokens;
            n = min(a.chunk_tokens, min(max(raw, 0), t.cap) - j0);
            if (n > 0) {
                const int n0 = min(kSub, n);
                stage_tier(t, unit, j0, (n0 + 31) & ~31, D, a.G, stage_base, b0);
                if (n > kSub) {
                    const int n1 = min(kSub, n - kSub);
                    stage_tier(t, unit, j0 + kSub, (n1 + 31) & ~31, D, a.G, stage_base + a.stage_bytes, b1);
                }
            }
        } else {
            const int cap = a.res_cap;
            const int raw = a.res_len[unit];
            const int len = min(max(raw, 0), cap - 1), start = a.res_start[unit];
            if (raw != len || start < 0 || start >= cap) atomicOr(&g_status_decode, kDevCheck);
            const int j0 = chunk * kResChunk;
            n = min(kResChunk, len + 1 - j0);
            if (n > 0 && start >= 0 && start < cap) stage_residual(a, unit, len, start, j0, n, D, stage_base, b0);
            else n = 0;
        }
        sm.n_total = max(n, 0);
    }
    for (int idx = threadIdx.x; idx < NG * D; idx += blockDim.x) {
        const int h = idx / D, c = idx % D;
        sm.q[h][c] = ldf(a.q, ((size_t)b * a.Hq + (size_t)hkv * NG + h) * D + c, bf) * a.scale_log2;
    }
    for (int idx = threadIdx.x; idx < kWarps * NG; idx += blockDim.x) {
        sm.wm[idx / NG][idx % NG] = kNegInf;
        sm.wl[idx / NG][idx % NG] = 0.0f;
    }
    for (int idx = threadIdx.x; idx < kWarps * NG * D; idx += blockDim.x) (&sm.wo[0][0][0])[idx] = 0.0f;
    __syncthreads();

    float* lg_unit = a.logits ? a.logits + unit * NG * (size_t)a.slots : nullptr;
    const int n = sm.n_total;
    if (n > 0) {
        if (tier >= 0) {
            const TierArgs& t = a.tier[tier];
            const int j0 = chunk * a.chunk_tokens;
            float* lg = (a.policy == KVQ_POLICY_MIKV && lg_unit) ? lg_unit + t.slot_base + j0 : nullptr;
            if (!dispatch_tier<NG, D>(a, sm, t, unit, j0, n, stage_base, lg) && threadIdx.x == 0)
                atomicOr(&g_status_decode, kDevCheck);
        } else {
            const int j0 = chunk * kResChunk;
            const bool ok = __syncthreads_and(mbar_wait(smem_u32(&sm.bar[0]), 0, nullptr));
            if (!ok) {
                if (threadIdx.x == 0) atomicOr(&g_status_decode, kDevTimeout);
            } else {
                const uint16_t* rk = reinterpret_cast<const uint16_t*>(stage_base);
                const uint16_t* rv = reinterpret_cast<const uint16_t*>(stage_base + a16((uint32_t)n * D * 2));
                float* lg = (lg_unit && a.policy != KVQ_POLICY_MINIKV) ? lg_unit + a.res_slot_base + j0 : nullptr;
                warp_residual<NG, D>(a, sm, rk, rv, n, lg);
            }
        }
    }
    if (tier < 0 && chunk == 0) {
        // the new token joins the ring; no CTA reads this slot in this step
        const int cap = a.res_cap;
        const int len = min(max(a.res_len[unit], 0), cap - 1);
        const int start = min(max(a.res_start[unit], 0), cap - 1);
        const size_t slot = unit * (size_t)cap + (start + len) % cap;
        for (int c = threadIdx.x; c < D; c += blockDim.x) {
            stf(a.res_k, slot * D + c, ldf(a.k_new, unit * D + c, bf), bf);
            stf(a.res_v, slot * D + c, ldf(a.v_new, unit * D + c, bf), bf);
        }
        if (threadIdx.x == 0) a.res_token_id[slot] = a.seq_len[b];
    }
    __syncthreads();

    // ---- chunk partial: merge the four warps
    float* part_out = a.part + (unit * NG * TC + blockIdx.x) * (size_t)(D + 2);
    for (int idx = threadIdx.x; idx < NG * D; idx += blockDim.x) {
        const int h = idx / D, c = idx % D;
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][h]);
        float L = 0.0f, O = 0.0f;
        if (M != kNegInf) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = sm.wm[w][h] == kNegInf ? 0.0f : ex2_approx(sm.wm[w][h] - M);
                L = fmaf(sm.wl[w][h], f, L);
                O = fmaf(sm.wo[w][h][c], f, O);
            }
        }
        float* po = part_out + (size_t)h * TC * (D + 2);
        po[2 + c] = O;
        if (c == 0) {
            po[0] = M;
            po[1] = L;
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(&a.counters[unit], 1u);
        sm.last = (prev == (uint32_t)TC - 1u) ? 1 : 0;
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();

    const float* pu = a.part + unit * NG * TC * (size_t)(D + 2);
    // chunk maxima and sums, all loads in flight together (scratch = the staging buffers)
    float* cm = reinterpret_cast<float*>(stage_base);      // [NG][TC]
    float* cw = cm + NG * TC;                               // [NG][TC]
    for (int idx = threadIdx.x; idx < NG * TC; idx += blockDim.x) {
        const float* ph = pu + (size_t)idx * (D + 2);
        const float l = __ldcg(ph + 1);
        cm[idx] = l > 0.0f ? __ldcg(ph) : kNegInf;
        cw[idx] = l;
    }
    __syncthreads();
    if (threadIdx.x < NG) {
        const int h = threadIdx.x;
        float M = kNegInf;
        for (int y = 0; y < TC; ++y) M = fmaxf(M, cm[h * TC + y]);
        float L = 0.0f;
        for (int y = 0; y < TC; ++y) {
            const float wgt = cm[h * TC + y] == kNegInf ? 0.0f : ex2_approx(cm[h * TC + y] - M);
            L = fmaf(cw[h * TC + y], wgt, L);
            cw[h * TC + y] = wgt;
        }
        sm.wl[0][h] = L;
        sm.wm[0][h] = M + __log2f(L);          // base-2 lse
        if (a.lse_out) a.lse_out[(size_t)b * a.Hq + hkv * NG + h] = (M + __log2f(L)) * kLn2;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < NG * D; idx += blockDim.x) {
        const int h = idx / D, c = idx % D;
        const float* ph = pu + (size_t)h * TC * (D + 2) + 2 + c;
        float acc = 0.0f;
#pragma unroll 8
        for (int y = 0; y < TC; ++y) acc = fmaf(__ldcg(ph + (size_t)y * (D + 2)), cw[h * TC + y], acc);
        stf(a.o, ((size_t)b * a.Hq + hkv * NG + h) * D + c, acc / sm.wl[0][h], bf);
    }
    const int cap = a.res_cap;
    const int len = min(max(a.res_len[unit], 0), cap - 1);
    const int start = min(max(a.res_start[unit], 0), cap - 1);
    const float* lse2 = sm.wm[0];
    if (a.policy == KVQ_POLICY_MIKV && lg_unit) {
        float* cs = a.cum_score + unit * (size_t)a.score_cap;
        for (int t = 0; t < a.n_tiers; ++t) {
            const TierArgs& ti = a.tier[t];
            const int cnt = min(max(ti.count[unit], 0), ti.cap);
            for (int j = threadIdx.x; j < cnt; j += blockDim.x) {
                float p = 0.0f;
#pragma unroll
                for (int h = 0; h < NG; ++h)
                    p += ex2_approx(__ldcg(lg_unit + (size_t)h * a.slots + ti.slot_base + j) - lse2[h]);
                const int id = ti.token_id[unit * (size_t)ti.cap + j];
                if (id >= 0 && id < a.score_cap) cs[id] = __fadd_rn(cs[id], p);
                else atomicOr(&g_status_decode, kDevCheck);
            }
        }
        for (int li = threadIdx.x; li <= len; li += blockDim.x) {
            float p = 0.0f;
#pragma unroll
            for (int h = 0; h < NG; ++h)
                p += ex2_approx(__ldcg(lg_unit + (size_t)h * a.slots + a.res_slot_base + li) - lse2[h]);
            const int id = li < len ? a.res_token_id[unit * (size_t)cap + (start + li) % cap] : a.seq_len[b];
            if (id < 0 || id >= a.score_cap) atomicOr(&g_status_decode, kDevCheck);
            else cs[id] = li < len ? __fadd_rn(cs[id], p) : p;
        }
    } else if (a.policy == KVQ_POLICY_DIFFKV && lg_unit) {
        for (int idx = threadIdx.x; idx < (len + 1) * NG; idx += blockDim.x) {
            const int li = idx / NG, h = idx % NG;
            const float p = ex2_approx(__ldcg(lg_unit + (size_t)h * a.slots + a.res_slot_base + li) - lse2[h]);
            float* wa = a.win_acc + ((size_t)b * a.Hq + hkv * NG + h) * cap + (start + li) % cap;
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

// Packed tokens per CTA: as many sub-chunks (up to kMaxSubs) as keeps about
// six CTAs' worth of sub-chunks per SM; small caches get one sub-chunk per
// CTA so that every SM has work.
int chunk_tokens_for(const kvq_cache& c) {
    long subs = 0;
    for (int t = 0; t < c.n_tiers; ++t) subs += (long)c.B * c.Hkv * ((c.tier[t].cap + kSub - 1) / kSub);
    const long per = (subs + 152L * 6 - 1) / (152L * 6);
    return kSub * (int)std::max(1L, std::min((long)kMaxSubs, per));
}

WsLayout ws_layout(const kvq_cache& c) {
    WsLayout w{};
    const int units = c.B * c.Hkv, g = c.Hq / c.Hkv;
    const int ct = chunk_tokens_for(c);
    int chunks = 0, slots = 0;
    for (int t = 0; t < c.n_tiers; ++t) {
        chunks += (c.tier[t].cap + ct - 1) / ct;
        slots += c.tier[t].cap;
    }
    chunks += (c.res_cap + kResChunk - 1) / kResChunk;
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

template <int NG, int D>
cudaError_t launch_typed(DecodeArgs& a, const kvq_cache& c, int units, cudaStream_t s) {
    uint32_t stage = a16((uint32_t)kResChunk * D * 2) * 2u;
    for (int t = 0; t < c.n_tiers; ++t)
        stage = std::max(stage, tier_stage_sizes(c.tier[t].k_axis, c.tier[t].k_bits, c.tier[t].v_bits,
                                                 kSub, D, c.G).total());
    stage = (stage + 127u) & ~127u;
    a.stage_bytes = stage;
    // the merge reuses both buffers as scratch
    const uint32_t scratch = (uint32_t)(2 * NG * a.total_chunks * sizeof(float));
    const size_t bufs = std::max((size_t)2 * stage, (size_t)scratch);
    const size_t sh = ((sizeof(Smem<NG, D>) + 127) & ~(size_t)127) + bufs;
    static size_t attr = 0;
    if (sh > 48 * 1024 && sh > attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<NG, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sh);
        if (e != cudaSuccess) return e;
        attr = sh;
    }
    dim3 grid(a.total_chunks, units);
    decode_kernel<NG, D><<<grid, kThreads, sh, s>>>(a);
    return cudaGetLastError();
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
    a.chunk_tokens = chunk_tokens_for(c);
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
        ta.chunks = (ct.cap + a.chunk_tokens - 1) / a.chunk_tokens;
        ta.slot_base = slot;
        slot += ct.cap;
    }
    a.res_k = c.res_k;
    a.res_v = c.res_v;
    a.res_token_id = c.res_token_id;
    a.res_start = c.res_start;
    a.res_len = c.res_len;
    a.res_cap = c.res_cap;
    a.res_chunks = (c.res_cap + kResChunk - 1) / kResChunk;
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
    if (a.g == 1 && c.D == 128) return launch_typed<1, 128>(a, c, units, s);
    if (a.g == 1 && c.D == 64) return launch_typed<1, 64>(a, c, units, s);
    if (a.g == 2 && c.D == 128) return launch_typed<2, 128>(a, c, units, s);
    if (a.g == 4 && c.D == 128) return launch_typed<4, 128>(a, c, units, s);
    if (a.g == 5 && c.D == 128) return launch_typed<5, 128>(a, c, units, s);
    if (a.g == 8 && c.D == 128) return launch_typed<8, 128>(a, c, units, s);
    return cudaErrorInvalidConfiguration;
}

// ---- workspace in the library's own device memory, for callers that cannot
// allocate one.  The array lives in every context that loads the library,
// for as long as the library stays loaded.  In host code its name is only a
// host-side stand-in, so its device address is looked up once per device.
static __device__ __align__(256) uint8_t g_decode_scratch[KVQ_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
}  // namespace

// Device address of the static scratch on the current device (looked up on
// the first call made with that device current).
cudaError_t static_decode_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace kvq
